// Decode-phase dequantizing GEMV, 1 <= M <= 16:
//   out[m, n] = sum_k x[m, k] * dequant(W)[n, k]
// (metaltile PR #250 qgemv commits: output[row] = sum_k dequant(weight[row,k])
// * input[k], and the multi-row qmm; rlx-cpu thunk/ops/quant.rs
// dequant_matmul_nvfp4, whose m == 1 loop streams the packed codes once and
// folds each block scale into a per-block partial sum, and lowp_scaled_matmul,
// which factors both operands' block scales out of each block's sum).
//
// The pages' Metal GEMVs give each row one threadgroup and reduce with scalar
// code; they note it reads at a low fraction of bandwidth.  On GB300 the HBM
// delivers about 46 four-bit codes per SM per clock, so the decode has to cost
// well under three issue slots per code.  The design:
//  * a CTA owns 16 weight rows; its 8 warps split K in 64-code units, several
//    units in flight per lane, every lane loading word t of each 16-byte row
//    segment (the four lanes of a quad share each scale block);
//  * element codes go to f16 with the hardware conversions (E2M1, E4M3, E5M2 ->
//    f16x2 are exact; int4 becomes the exact f16 1024 + q), and the weights
//    are the 16-row A operand of mma.sync m16n8k16 (f16 in, float32 out);
//  * the activations are staged once per CTA in shared memory as f16 with a
//    power-of-two scale per (row, 64-code unit) that puts the unit's largest
//    |x| in [2^14, 2^15): exact for every bf16 value within 2^28 of that
//    maximum;
//  * block scales multiply float32 partial sums (one scale block per MMA k
//    slice), except nvfp4 whose E4M3 micro-scale times the E2M1 value is exact
//    in f16 and is applied before the MMA; the activation scale and the nvfp4
//    global scale follow in float32;
//  * per-warp partial tiles are summed through shared memory.
#include <cuda_runtime.h>

#include <atomic>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {
namespace gemv {

constexpr int WARPS = 8;

__device__ __forceinline__ void mma_f16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ldg32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ldg8(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// 8 E2M1 codes -> f16x2 in natural order (c0,c1) (c2,c3) (c4,c5) (c6,c7).
__device__ __forceinline__ void e2m1x8_f16(uint32_t w, uint32_t r[4]) {
  asm("{.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

// 4 E4M3 (or E5M2) codes -> f16x2 (c0,c1) (c2,c3).
template <bool E5>
__device__ __forceinline__ void f8x4_f16(uint32_t w, uint32_t r[2]) {
  if constexpr (E5)
    asm("{.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, h0;\n\tcvt.rn.f16x2.e5m2x2 %1, h1;}"
        : "=r"(r[0]), "=r"(r[1]) : "r"(w));
  else
    asm("{.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;}"
        : "=r"(r[0]), "=r"(r[1]) : "r"(w));
}

// One E4M3 byte -> f16x2 with the value in both halves (exact).
__device__ __forceinline__ uint32_t e4m3_f16x2_splat(uint32_t b) {
  uint32_t r;
  const uint16_t h = uint16_t(b | (b << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// f16 bits of 1024 + q for 8 unsigned 4-bit q, paired (q0,q4) (q1,q5) (q2,q6) (q3,q7).
__device__ __forceinline__ void int4x8_f16_biased(uint32_t w, uint32_t r[4]) {
  r[0] = (w & 0x000F000Fu) | 0x64006400u;
  r[1] = ((w >> 4) & 0x000F000Fu) | 0x64006400u;
  r[2] = ((w >> 8) & 0x000F000Fu) | 0x64006400u;
  r[3] = ((w >> 12) & 0x000F000Fu) | 0x64006400u;
}

template <int F, int R>
struct Cfg {
  static constexpr bool four = FmtTraits<F>::four;
  static constexpr int SEGS = four ? 2 : 4;        // 16-byte row segments per 64-code unit
  static constexpr int UNROLL = four ? (R == 1 ? 4 : 2) : (R == 1 ? 2 : 1);   // units in flight per lane
  static constexpr int NSC = (F == NVFP8) ? 4 : (F == INT4_AFFINE ? 1 : 2);   // scale words per row per unit
};

// Raw scale words of one row for one unit (64 codes starting at k).
template <int F, int NSC>
__device__ __forceinline__ void load_unit_scales(const uint8_t* scales, int64_t row, int64_t nblk, int64_t k, int K,
                                                 bool ok, int t, uint32_t s[NSC]) {
  #pragma unroll
  for (int i = 0; i < NSC; ++i) s[i] = 0u;
  if (!ok) return;
  const int64_t base = row * nblk;
  if constexpr (F == MXFP4 || F == MXFP8_E4M3 || F == MXFP8_E5M2) {
    s[0] = ldg8(scales + base + k / 32);
    if (k + 32 < K) s[1] = ldg8(scales + base + k / 32 + 1);
  } else if constexpr (F == NVFP4) {
    // the lane's word of segment j lies in block (k + 32 j + 8 t) / 16
    s[0] = ldg8(scales + base + (k + 8 * t) / 16);
    if (k + 32 < K) s[1] = ldg8(scales + base + (k + 32 + 8 * t) / 16);
  } else if constexpr (F == NVFP8) {
    const uint32_t* sp = reinterpret_cast<const uint32_t*>(scales) + base + k / 16;
    #pragma unroll
    for (int i = 0; i < 4; ++i)
      if (k + 16 * i < K) s[i] = ldg32(sp + i);
  } else {
    s[0] = ldg32(reinterpret_cast<const uint32_t*>(scales) + base + k / 64);
  }
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// One warp multiplies a 16-row weight tile (rows g and g+8 per lane) for one
// 64-code unit against the staged activations, into d64 (float32, per column
// block).  wa/wb: the lane's words of the two rows, sa/sb: their scale words.
template <int F, int NB, int SEGS, int NSC>
__device__ __forceinline__ void tile_unit(const uint32_t (&wa)[SEGS], const uint32_t (&wb)[SEGS],
                                          const uint32_t (&sa)[NSC], const uint32_t (&sb)[NSC],
                                          const uint16_t* xs, int xstride, int u, int M, int g, int t,
                                          float (&d64)[NB][4]) {
  constexpr bool FOUR = FmtTraits<F>::four;
  constexpr bool I4 = F == INT4_AFFINE;
  #pragma unroll
  for (int nb = 0; nb < NB; ++nb) d64[nb][0] = d64[nb][1] = d64[nb][2] = d64[nb][3] = 0.0f;
  #pragma unroll
  for (int sgm = 0; sgm < SEGS; ++sgm) {
    if constexpr (FOUR) {
      uint32_t fa[4], fb[4];
      if constexpr (I4) {
        int4x8_f16_biased(wa[sgm], fa);
        int4x8_f16_biased(wb[sgm], fb);
      } else {
        e2m1x8_f16(wa[sgm], fa);
        e2m1x8_f16(wb[sgm], fb);
        if constexpr (F == NVFP4) {
          const uint32_t ca = e4m3_f16x2_splat(sa[sgm]), cb = e4m3_f16x2_splat(sb[sgm]);
          #pragma unroll
          for (int q = 0; q < 4; ++q) {
            fa[q] = hmul2_f16(fa[q], ca);
            fb[q] = hmul2_f16(fb[q], cb);
          }
        }
      }
      #pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int m = min(nb * 8 + g, M - 1);
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + size_t(m) * xstride + u * 64 + sgm * 32 + 8 * t);
        if constexpr (F == MXFP4) {
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_f16(d, fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
          mma_f16(d, fa[2], fb[2], fa[3], fb[3], xv.z, xv.w);
          const float swa = e8m0_f32(sa[sgm]), swb = e8m0_f32(sb[sgm]);
          d64[nb][0] = __fmaf_rn(swa, d[0], d64[nb][0]);
          d64[nb][1] = __fmaf_rn(swa, d[1], d64[nb][1]);
          d64[nb][2] = __fmaf_rn(swb, d[2], d64[nb][2]);
          d64[nb][3] = __fmaf_rn(swb, d[3], d64[nb][3]);
        } else {
          mma_f16(d64[nb], fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
          mma_f16(d64[nb], fa[2], fb[2], fa[3], fb[3], xv.z, xv.w);
        }
      }
    } else {
      uint32_t fa[2], fb[2];
      f8x4_f16<F == MXFP8_E5M2>(wa[sgm], fa);
      f8x4_f16<F == MXFP8_E5M2>(wb[sgm], fb);
      #pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int m = min(nb * 8 + g, M - 1);
        const uint2 xv = *reinterpret_cast<const uint2*>(xs + size_t(m) * xstride + u * 64 + sgm * 16 + 4 * t);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        mma_f16(d, fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
        float swa, swb;
        if constexpr (F == NVFP8) {
          swa = __uint_as_float(sa[sgm]);
          swb = __uint_as_float(sb[sgm]);
        } else {
          swa = e8m0_f32(sa[sgm >> 1]);
          swb = e8m0_f32(sb[sgm >> 1]);
        }
        d64[nb][0] = __fmaf_rn(swa, d[0], d64[nb][0]);
        d64[nb][1] = __fmaf_rn(swa, d[1], d64[nb][1]);
        d64[nb][2] = __fmaf_rn(swb, d[2], d64[nb][2]);
        d64[nb][3] = __fmaf_rn(swb, d[3], d64[nb][3]);
      }
    }
  }
}

template <int F, int NB, int R>
__global__ void __launch_bounds__(WARPS * 32) qgemv_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales, float glob,
                                                           const uint16_t* __restrict__ x, void* __restrict__ out,
                                                           int out_f32, int M, int N, int K, int KS) {
  using C = Cfg<F, R>;
  constexpr bool FOUR = C::four;
  constexpr int SEGS = C::SEGS, U = C::UNROLL, NSC = C::NSC;
  constexpr bool I4 = F == INT4_AFFINE;
  constexpr int ROWS = 16 * R;
  extern __shared__ __align__(16) uint8_t smem[];
  const int xstride = KS + 8;                                   // f16 elements per staged row (+16 B pad)
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);
  float* xsc = reinterpret_cast<float*>(smem + size_t(M) * xstride * 2);   // [M][KS/64] 2^-shift
  float* xsum = xsc + M * (KS / 64);                                        // [M][KS/64] (int4 affine)
  float* red = xsum + (I4 ? M * (KS / 64) : 0);                             // [WARPS][ROWS][8 NB]

  // Let the next kernel in the stream start its own weight traffic now.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * ROWS;
  const int64_t row_bytes = FOUR ? K / 2 : K;
  const int64_t nblk = K / FmtTraits<F>::block;
  const int sbytes = FmtTraits<F>::sbytes;

  // Weights do not depend on the preceding kernel: pull this CTA's rows into L2.
  if (lane == 0) {
    #pragma unroll 1
    for (int rr = warp * (ROWS / WARPS); rr < (warp + 1) * (ROWS / WARPS); ++rr) {
      const int row = row0 + rr;
      if (row < N) {
        prefetch_l2(codes + int64_t(row) * row_bytes, uint32_t(row_bytes));
        const uint32_t sb = uint32_t(nblk * sbytes);
        if ((sb & 15u) == 0 && ((int64_t(row) * nblk * sbytes) & 15) == 0)
          prefetch_l2(scales + int64_t(row) * nblk * sbytes, sb);
      }
    }
  }

  const uint8_t* pA[R];
  const uint8_t* pB[R];
  int rowA[R], rowB[R];
  bool okA[R], okB[R];
  #pragma unroll
  for (int r = 0; r < R; ++r) {
    rowA[r] = row0 + 16 * r + g;
    rowB[r] = rowA[r] + 8;
    okA[r] = rowA[r] < N;
    okB[r] = rowB[r] < N;
    pA[r] = codes + int64_t(okA[r] ? rowA[r] : 0) * row_bytes;
    pB[r] = codes + int64_t(okB[r] ? rowB[r] : 0) * row_bytes;
  }

  float acc[R][NB][4];
  #pragma unroll
  for (int r = 0; r < R; ++r)
    #pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[r][nb][0] = acc[r][nb][1] = acc[r][nb][2] = acc[r][nb][3] = 0.0f;

  uint32_t wa[U][R][SEGS], wb[U][R][SEGS], sa[U][R][NSC], sb[U][R][NSC];

  for (int ks = 0; ks < K; ks += KS) {
    const int kn = K - ks < KS ? K - ks : KS;
    const int units = (kn + 63) / 64;
    auto issue = [&](int i, int slot) {
      const int u = warp + i * WARPS;
      const int64_t k = int64_t(ks) + int64_t(u) * 64;
      const bool ok = u < units;
      #pragma unroll
      for (int r = 0; r < R; ++r) {
        #pragma unroll
        for (int sgm = 0; sgm < SEGS; ++sgm) {
          const int64_t ksg = k + sgm * (FOUR ? 32 : 16);
          const bool v = ok && ksg < K;
          const int64_t off = (FOUR ? ksg / 2 : ksg) + 4 * t;
          wa[slot][r][sgm] = v && okA[r] ? ldg32(pA[r] + off) : 0u;
          wb[slot][r][sgm] = v && okB[r] ? ldg32(pB[r] + off) : 0u;
        }
        load_unit_scales<F, NSC>(scales, rowA[r], nblk, k, K, ok && okA[r], t, sa[slot][r]);
        load_unit_scales<F, NSC>(scales, rowB[r], nblk, k, K, ok && okB[r], t, sb[slot][r]);
      }
    };
    #pragma unroll
    for (int i = 0; i < U; ++i) issue(i, i);

    // The activations may be the preceding kernel's output: wait for it (once).
    if (ks == 0) asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- stage the activations of this K range as scaled f16 -------------
    // 8 lanes per (row, 64-code unit), 8 values each; the shift puts the
    // unit's max |x| in [2^14, 2^15).
    const int tasks = M * units * 8;
    for (int i = threadIdx.x; i < ((tasks + 255) & ~255); i += blockDim.x) {
      const bool live = i < tasks;
      const int m = live ? i / (units * 8) : 0;
      const int rem = live ? i - m * units * 8 : 0;
      const int u = rem >> 3, part = rem & 7;
      const int64_t k = int64_t(ks) + u * 64 + part * 8;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (live && k < K) v = __ldg(reinterpret_cast<const uint4*>(x + int64_t(m) * K + k));
      const uint32_t h[4] = {v.x, v.y, v.z, v.w};
      uint32_t mx = 0;
      #pragma unroll
      for (int j = 0; j < 4; ++j) mx = max(mx, max(h[j] & 0x7FFFu, (h[j] >> 16) & 0x7FFFu));
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
      const int E = int(mx >> 7);
      int sh = (mx == 0u || E == 255) ? 0 : 141 - E;               // 14 - (E - 127)
      sh = sh > 126 ? 126 : sh;
      const float up = __uint_as_float(uint32_t(sh + 127) << 23);
      float f[8];
      #pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[2 * j] = __fmul_rn(__uint_as_float(h[j] << 16), up);
        f[2 * j + 1] = __fmul_rn(__uint_as_float(h[j] & 0xFFFF0000u), up);
      }
      uint32_t o[4];
      if constexpr (I4) {    // stored as (x0,x4) (x1,x5) (x2,x6) (x3,x7), the int4 pairing
        #pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = pack_f16x2(f[j], f[j + 4]);
      } else {
        #pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = pack_f16x2(f[2 * j], f[2 * j + 1]);
      }
      if (live)
        *reinterpret_cast<uint4*>(xs + size_t(m) * xstride + u * 64 + part * 8) = make_uint4(o[0], o[1], o[2], o[3]);
      if constexpr (I4) {    // sum of the staged (rounded) values
        float sm = 0.0f;
        #pragma unroll
        for (int j = 0; j < 4; ++j) sm += f16x2_lo(o[j]) + f16x2_hi(o[j]);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 1);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 2);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 4);
        if (live && part == 0) xsum[m * (KS / 64) + u] = sm;
      }
      if (live && part == 0) xsc[m * (KS / 64) + u] = __uint_as_float(uint32_t(127 - sh) << 23);
    }
    __syncthreads();

    // ---- stream the weights -------------------------------------------------
    #pragma unroll 1
    for (int i0 = 0; warp + i0 * WARPS < units; i0 += U) {
      #pragma unroll
      for (int j = 0; j < U; ++j) {
        const int i = i0 + j;
        const int u = warp + i * WARPS;
        if (u >= units) break;
        #pragma unroll
        for (int r = 0; r < R; ++r) {
          float d64[NB][4];
          tile_unit<F, NB, SEGS, NSC>(wa[j][r], wb[j][r], sa[j][r], sb[j][r], xs, xstride, u, M, g, t, d64);
          #pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const int c0 = min(nb * 8 + 2 * t, M - 1), c1 = min(nb * 8 + 2 * t + 1, M - 1);
            const float x0 = xsc[c0 * (KS / 64) + u], x1 = xsc[c1 * (KS / 64) + u];
            if constexpr (I4) {
              const float sA = bf16bits_f32(sa[j][r][0] & 0xFFFFu), bA = bf16bits_f32(sa[j][r][0] >> 16);
              const float sB = bf16bits_f32(sb[j][r][0] & 0xFFFFu), bB = bf16bits_f32(sb[j][r][0] >> 16);
              const float cA = __fmaf_rn(-1024.0f, sA, bA), cB = __fmaf_rn(-1024.0f, sB, bB);
              const float m0 = xsum[c0 * (KS / 64) + u], m1 = xsum[c1 * (KS / 64) + u];
              d64[nb][0] = __fmaf_rn(sA, d64[nb][0], cA * m0);
              d64[nb][1] = __fmaf_rn(sA, d64[nb][1], cA * m1);
              d64[nb][2] = __fmaf_rn(sB, d64[nb][2], cB * m0);
              d64[nb][3] = __fmaf_rn(sB, d64[nb][3], cB * m1);
            }
            acc[r][nb][0] = __fmaf_rn(x0, d64[nb][0], acc[r][nb][0]);
            acc[r][nb][1] = __fmaf_rn(x1, d64[nb][1], acc[r][nb][1]);
            acc[r][nb][2] = __fmaf_rn(x0, d64[nb][2], acc[r][nb][2]);
            acc[r][nb][3] = __fmaf_rn(x1, d64[nb][3], acc[r][nb][3]);
          }
        }
        issue(i + U, j);   // refill this slot with the unit U ahead
      }
    }
    __syncthreads();
  }

  // acc[r][nb]: c0 = (row 16r+g, col 2t), c1 = (16r+g, 2t+1), c2 = (16r+g+8, 2t), c3 = (16r+g+8, 2t+1).
  constexpr int RC = 8 * NB;
  #pragma unroll
  for (int r = 0; r < R; ++r)
    #pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
      float* rw = red + (size_t(warp) * ROWS + 16 * r + g) * RC + nb * 8 + 2 * t;
      rw[0] = acc[r][nb][0];
      rw[1] = acc[r][nb][1];
      rw[8 * RC] = acc[r][nb][2];
      rw[8 * RC + 1] = acc[r][nb][3];
    }
  __syncthreads();
  for (int i = threadIdx.x; i < ROWS * M; i += blockDim.x) {
    const int r = i % ROWS, m = i / ROWS;
    if (row0 + r >= N) continue;
    float sum = 0.0f;
    #pragma unroll
    for (int w = 0; w < WARPS; ++w) sum += red[(size_t(w) * ROWS + r) * RC + m];
    if constexpr (F == NVFP4) sum *= glob;
    const int64_t o = int64_t(m) * N + row0 + r;
    if (out_f32) static_cast<float*>(out)[o] = sum;
    else static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(sum);
  }
}

// Activations staged per pass: all of K up to 4096 (M <= 8) or 2048 (M > 8).
inline int stage_k(int M, int K) {
  const int cap = M <= 8 ? 4096 : 2048;
  const int k64 = (K + 63) / 64 * 64;
  return k64 < cap ? k64 : cap;
}

inline size_t smem_bytes(int F, int M, int KS, int R, int NB) {
  return size_t(M) * (KS + 8) * 2 + size_t(M) * (KS / 64) * 4 * (F == INT4_AFFINE ? 2 : 1) +
         size_t(WARPS) * 16 * R * 8 * NB * 4;
}

// Launch with programmatic stream serialization: the kernel may start while
// the preceding kernel in the stream finishes (it waits before touching X).
template <typename Kern, typename... Args>
static cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kern, args...);
}

template <int F, int NB, int R>
static cudaError_t launch_nb(const uint8_t* c, const uint8_t* s, float glob, const uint16_t* x, void* out,
                             bool out_f32, int M, int N, int K, cudaStream_t st) {
  static std::atomic<int> attr_done[64];
  const int KS = stage_k(M, K);
  const size_t sm = smem_bytes(F, M, KS, R, NB);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_done[dev].load()) {
    const size_t cap = NB == 1 ? smem_bytes(F, 8, 4096, R, NB) : smem_bytes(F, 16, 2048, R, NB);
    e = cudaFuncSetAttribute(qgemv_kernel<F, NB, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(cap));
    if (e != cudaSuccess) return e;
    attr_done[dev].store(1);
  }
  e = launch_pdl(qgemv_kernel<F, NB, R>, dim3((N + 16 * R - 1) / (16 * R)), dim3(WARPS * 32), sm, st, c, s, glob, x,
                 out, int(out_f32), M, N, K, KS);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Rows per warp: 16 for M <= 2, 32 beyond (each staged activation then serves
// two weight tiles, which keeps staging small next to the weight stream).
template <int F>
static cudaError_t launch_fmt(const void* codes, const void* scales, float glob, const void* x, void* out,
                              bool out_f32, int M, int N, int K, cudaStream_t st) {
  auto c = static_cast<const uint8_t*>(codes);
  auto s = static_cast<const uint8_t*>(scales);
  auto xx = static_cast<const uint16_t*>(x);
  if (M <= 2) return launch_nb<F, 1, 1>(c, s, glob, xx, out, out_f32, M, N, K, st);
  if (M <= 8) return launch_nb<F, 1, 2>(c, s, glob, xx, out, out_f32, M, N, K, st);
  return launch_nb<F, 2, 2>(c, s, glob, xx, out, out_f32, M, N, K, st);
}

}  // namespace gemv

cudaError_t launch_qgemv(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                         bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms) {
  (void)sms;
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return gemv::launch_fmt<MXFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP4: return gemv::launch_fmt<NVFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP8_E4M3: return gemv::launch_fmt<MXFP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP8_E5M2: return gemv::launch_fmt<MXFP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP8: return gemv::launch_fmt<NVFP8>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    default: return gemv::launch_fmt<INT4_AFFINE>(codes, scales, glob, x, out, out_f32, m, n, k, st);
  }
}

}  // namespace qfmt_dev
