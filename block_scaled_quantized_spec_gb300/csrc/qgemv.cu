// Decode GEMV dispatch for 1 <= M <= 16, and the bulk-copy GEMV that serves
// the shapes the two register-direct kernels do not plan for (activations of a
// very long K that exceed their shared-memory slices):
//   out[m, n] = sum_k x[m, k] * dequant(W)[n, k]
// (metaltile PR #250 qgemv commits: output[row] = sum_k dequant(weight[row,k])
// * input[k], and the multi-row qmm; rlx-cpu thunk/ops/quant.rs
// dequant_matmul_nvfp4, whose m == 1 loop streams the packed codes once and
// folds each block scale into a per-block partial sum, and lowp_scaled_matmul,
// which factors both operands' block scales out of each block's sum).
//
// Dispatch: M <= 2 -> qgemv_m2.cuh; 3 <= M <= 16 -> qgemv_mb.cu; otherwise the
// kernel below, which takes K in passes:
//  * a CTA owns 16 (M <= 2) or 32 weight rows; one thread bulk-copies the
//    CTA's code rows for a pass into shared memory with cp.async.bulk on an
//    mbarrier, rows padded by 16 bytes so that the reads below are
//    bank-conflict free;
//  * the launch is programmatic-dependent: the weight copies and the staging
//    of the block scales (float32, or f16 for nvfp4) run while the preceding
//    kernel drains; the CTA waits for that kernel only before its activations;
//  * the 8 warps split K in 64-code units; every lane reads word t of each
//    16-byte row segment (the four lanes of a quad share each scale block);
//  * element codes go to f16 with the hardware conversions (E2M1, E4M3, E5M2 ->
//    f16x2 are exact; int4 becomes the exact f16 1024 + q), and the weights
//    are the 16-row A operand of mma.sync m16n8k16 (f16 in, float32 out);
//  * the activations are staged once per pass in shared memory as f16 with a
//    power-of-two scale per (row, 64-code unit) that puts the unit's largest
//    |x| in [2^14, 2^15): exact for every bf16 value within 2^28 of that
//    maximum;
//  * block scales multiply float32 partial sums (one scale block per MMA k
//    slice), except nvfp4 whose E4M3 micro-scale times the E2M1 value is exact
//    in f16 and is applied before the MMA; the activation scale and the nvfp4
//    global scale follow in float32;
//  * per-warp partial tiles are summed through shared memory; the mbarrier
//    wait is bounded and records an expired wait in a device status word.
#include <cuda_runtime.h>

#include <atomic>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {
namespace gemv {

constexpr int WARPS = 8;
constexpr int THREADS = WARPS * 32;

__device__ __forceinline__ void mma_f16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
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
  static constexpr int BLK = FmtTraits<F>::block;
  static constexpr int SEGS = four ? 2 : 4;        // 16-byte row segments per 64-code unit
  // staged scale words per row per 64-code unit (int4 affine: s and b - 1024 s)
  static constexpr int SPU = is_i4<F>() ? 2 : 64 / BLK;
};

// Staged scale-row stride in 32-bit words: a multiple of 4 plus 4, so the
// eight rows a warp reads at once fall in distinct banks.
template <int F, int R>
__host__ __device__ constexpr int sc_stride(int KS) {
  return ((KS / 64) * Cfg<F, R>::SPU + 3) / 4 * 4 + 4;
}

// Staged code-row stride in bytes: the row's bytes plus 16, so that word t of
// a 16-byte segment in eight consecutive rows falls in distinct banks.
template <int F>
__host__ __device__ constexpr int code_stride(int KS) {
  return (FmtTraits<F>::four ? KS / 2 : KS) + 16;
}

__device__ unsigned int g_gemv_status;

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

template <int F, int NB, int R>
__global__ void __launch_bounds__(THREADS) qgemv_kernel(const uint8_t* __restrict__ codes,
                                                        const uint8_t* __restrict__ scales, float glob,
                                                        const uint16_t* __restrict__ x, void* __restrict__ out,
                                                        int out_f32, int M, int N, int K, int KS, uint64_t limit_ns) {
  using C = Cfg<F, R>;
  constexpr bool FOUR = C::four;
  constexpr int SEGS = C::SEGS, SPU = C::SPU, BLK = C::BLK;
  constexpr bool I4 = is_i4<F>();
  constexpr int ROWS = 16 * R;
  constexpr int RC = 8 * NB;
  extern __shared__ __align__(16) uint8_t smem[];
  const int xstride = KS + 8;                                          // f16 per staged activation row
  const int units_max = KS / 64;
  const int sst = sc_stride<F, R>(KS);
  const int cst = code_stride<F>(KS);
  uint8_t* wsm = smem;                                                 // [ROWS][cst] staged codes
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + size_t(ROWS) * cst);   // [M][KS + 8] f16
  float* xsc = reinterpret_cast<float*>(xs + size_t(M) * xstride);     // [M][KS/64] 2^-shift
  float* xsum = xsc + M * units_max;                                   // [M][KS/64] (int4 affine)
  float* wsc = xsum + (I4 ? M * units_max : 0);                        // [ROWS][sst] staged scales
  float* red = wsc + ROWS * sst;                                       // [WARPS][ROWS][RC]
  __shared__ __align__(8) uint64_t wbar;

  // The next kernel in the stream may launch now.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * ROWS;
  const int64_t row_bytes = FOUR ? K / 2 : K;
  const int64_t nblk = (K + BLK - 1) / BLK;   // int4 affine: a ragged last group
  const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(&wbar));
  const int nrows = N - row0 < ROWS ? N - row0 : ROWS;
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  float acc[R][NB][4];
  #pragma unroll
  for (int r = 0; r < R; ++r)
    #pragma unroll
    for (int nb = 0; nb < NB; ++nb) acc[r][nb][0] = acc[r][nb][1] = acc[r][nb][2] = acc[r][nb][3] = 0.0f;

  bool ok_all = true;
  int pass = 0;
  for (int ks = 0; ks < K; ks += KS, ++pass) {
    const int kn = K - ks < KS ? K - ks : KS;
    const int units = (kn + 63) / 64;
    const uint32_t pbytes = uint32_t(FOUR ? kn / 2 : kn);             // code bytes per row this pass

    // ---- weights of this pass: one bulk copy per row into shared memory ----
    // (they do not come from the preceding kernel, so no wait is needed)
    if (tid == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // earlier generic reads before the overwrite
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(pbytes * uint32_t(nrows))
                   : "memory");
      for (int rr = 0; rr < nrows; ++rr) {
        const uint8_t* src = codes + int64_t(row0 + rr) * row_bytes + (FOUR ? ks / 2 : ks);
        const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(wsm + size_t(rr) * cst));
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     ::"r"(dst), "l"(src), "r"(pbytes), "r"(bar)
                     : "memory");
      }
    }

    // ---- block scales of this pass (float32, f16 pairs for nvfp4) ---------
    {
      const int per_row = units * 64 / BLK;                            // scale entries per row
      const int ntask = ROWS * per_row;
      #pragma unroll 4
      for (int i = tid; i < ntask; i += THREADS) {
        const int rr = i / per_row, e = i - rr * per_row;
        const int row = row0 + rr;
        const int64_t blk = int64_t(ks / BLK) + e;
        const bool ok = row < N && blk < nblk;
        const int64_t gi = int64_t(ok ? row : 0) * nblk + (ok ? blk : 0);
        if constexpr (is_e8m0<F>()) {
          wsc[rr * sst + e] = ok ? e8m0_f32(__ldg(scales + gi)) : 0.0f;
        } else if constexpr (F == NVFP4) {
          wsc[rr * sst + e] = __uint_as_float(ok ? e4m3_f16x2_splat(__ldg(scales + gi)) : 0u);
        } else if constexpr (is_fs8<F>() || is_fp4f<F>()) {
          wsc[rr * sst + e] = ok ? float_scale<F>(scales, gi) : 0.0f;
        } else {
          float sc, bi;
          i4_scale_bias<F>(ok ? i4_word<F>(scales, gi) : 0u, sc, bi);
          wsc[rr * sst + 2 * e] = sc;
          wsc[rr * sst + 2 * e + 1] = __fmaf_rn(-1024.0f, sc, bi);
        }
      }
    }

    // The activations may be the preceding kernel's output: wait for it (once).
    if (ks == 0) asm volatile("griddepcontrol.wait;" ::: "memory");

    // ---- activations of this pass as scaled f16 ---------------------------
    // 8 lanes per (row, 64-code unit), 8 values each; the shift puts the
    // unit's max |x| in [2^14, 2^15).  Four tasks' loads are in flight at once.
    {
      const int tasks = M * units * 8;
      const int per_m = units * 8;
      const int padded = (tasks + THREADS - 1) / THREADS * THREADS;
      for (int i0 = tid; i0 < padded; i0 += 4 * THREADS) {
        uint4 v[4];
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * THREADS;
          const int m = i / per_m, rem = i - m * per_m;
          const int k = ks + (rem >> 3) * 64 + (rem & 7) * 8;
          v[j] = (i < tasks && k < K) ? __ldg(reinterpret_cast<const uint4*>(x + int64_t(m) * K + k))
                                     : make_uint4(0, 0, 0, 0);
        }
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = i0 + j * THREADS;
          if (i0 - tid + j * THREADS >= padded) break;                 // warp-uniform
          const bool live = i < tasks;
          const int m = live ? i / per_m : 0;
          const int rem = live ? i - m * per_m : 0;
          const int u = rem >> 3, part = rem & 7;
          const uint32_t h[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
          uint32_t mx = 0;
          #pragma unroll
          for (int q = 0; q < 4; ++q) mx = max(mx, max(h[q] & 0x7FFFu, (h[q] >> 16) & 0x7FFFu));
          mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
          mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
          mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
          const int E = int(mx >> 7);
          int sh = (mx == 0u || E == 255) ? 0 : 141 - E;               // 14 - (E - 127)
          sh = sh > 126 ? 126 : sh;
          const float up = __uint_as_float(uint32_t(sh + 127) << 23);
          float f[8];
          #pragma unroll
          for (int q = 0; q < 4; ++q) {
            f[2 * q] = __fmul_rn(__uint_as_float(h[q] << 16), up);
            f[2 * q + 1] = __fmul_rn(__uint_as_float(h[q] & 0xFFFF0000u), up);
          }
          uint32_t o[4];
          if constexpr (I4) {    // stored as (x0,x4) (x1,x5) (x2,x6) (x3,x7), the int4 pairing
            #pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = pack_f16x2(f[q], f[q + 4]);
          } else {
            #pragma unroll
            for (int q = 0; q < 4; ++q) o[q] = pack_f16x2(f[2 * q], f[2 * q + 1]);
          }
          if (live)
            *reinterpret_cast<uint4*>(xs + size_t(m) * xstride + u * 64 + part * 8) = make_uint4(o[0], o[1], o[2], o[3]);
          if constexpr (I4) {    // sum of the staged (rounded) values
            float sm = 0.0f;
            #pragma unroll
            for (int q = 0; q < 4; ++q) sm += f16x2_lo(o[q]) + f16x2_hi(o[q]);
            sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 1);
            sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 2);
            sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 4);
            if (live && part == 0) xsum[m * units_max + u] = sm;
          }
          if (live && part == 0) xsc[m * units_max + u] = __uint_as_float(uint32_t(127 - sh) << 23);
        }
      }
    }
    __syncthreads();

    // ---- the weights must have landed (bounded wait) ------------------------
    {
      int ok = 1;
      if (lane == 0) {
        if (!mbar_try_wait(bar, uint32_t(pass & 1))) {
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar, uint32_t(pass & 1)))
            if (globaltimer_ns() - t0 > limit_ns) { ok = 0; break; }
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          atomicOr(&g_gemv_status, 1u);
          // let the copies finish before this CTA's shared memory can be released
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar, uint32_t(pass & 1)) && globaltimer_ns() - t0 < limit_ns) {
          }
        }
        ok_all = false;
      }
    }

    // ---- multiply: each warp takes 64-code units warp, warp + 8, ... ------
    if (ok_all) {
      const uint8_t* wlane = wsm + g * cst + 4 * t;                    // row g of tile 0, lane's word
      const float* scl = wsc + g * sst;
      #pragma unroll 1
      for (int u = warp; u < units; u += WARPS) {
        #pragma unroll
        for (int r = 0; r < R; ++r) {
          const uint8_t* wra = wlane + (16 * r) * cst + (FOUR ? u * 32 : u * 64);
          const uint8_t* wrb = wra + 8 * cst;
          const float* sca = scl + (16 * r) * sst + u * SPU;
          const float* scb = sca + 8 * sst;
          float d64[NB][4];
          #pragma unroll
          for (int nb = 0; nb < NB; ++nb) d64[nb][0] = d64[nb][1] = d64[nb][2] = d64[nb][3] = 0.0f;
          #pragma unroll
          for (int sgm = 0; sgm < SEGS; ++sgm) {
            // a K that ends mid-unit leaves the tail segments unstaged: use zero codes
            const bool in = ks + u * 64 + sgm * (FOUR ? 32 : 16) < K;
            const uint32_t wa = in ? *reinterpret_cast<const uint32_t*>(wra + 16 * sgm) : 0u;
            const uint32_t wb = in ? *reinterpret_cast<const uint32_t*>(wrb + 16 * sgm) : 0u;
            if constexpr (FOUR) {
              uint32_t fa[4], fb[4];
              if constexpr (I4) {
                int4x8_f16_biased(i4_u<F>(wa), fa);
                int4x8_f16_biased(i4_u<F>(wb), fb);
              } else {
                if constexpr (F == MXINT4) {
                  sint4x8_f16(wa, fa);
                  sint4x8_f16(wb, fb);
                } else {
                  e2m1x8_f16(wa, fa);
                  e2m1x8_f16(wb, fb);
                }
                if constexpr (F == NVFP4) {
                  // the lane's word of this segment lies in micro-block 2 sgm + t/2 of the unit
                  const uint32_t ca = __float_as_uint(sca[2 * sgm + (t >> 1)]);
                  const uint32_t cb = __float_as_uint(scb[2 * sgm + (t >> 1)]);
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
                if constexpr (is_mx4<F>() || is_fp4f<F>()) {   // a block scale per segment
                  float d[4] = {0.f, 0.f, 0.f, 0.f};
                  mma_f16(d, fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
                  mma_f16(d, fa[2], fb[2], fa[3], fb[3], xv.z, xv.w);
                  const float swa = sca[sgm], swb = scb[sgm];
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
              elem8x4_f16<F>(wa, fa);
              elem8x4_f16<F>(wb, fb);
              const float swa = sca[16 * sgm / BLK], swb = scb[16 * sgm / BLK];   // the block of this segment
              #pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                const int m = min(nb * 8 + g, M - 1);
                const uint2 xv = *reinterpret_cast<const uint2*>(xs + size_t(m) * xstride + u * 64 + sgm * 16 + 4 * t);
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_f16(d, fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
                d64[nb][0] = __fmaf_rn(swa, d[0], d64[nb][0]);
                d64[nb][1] = __fmaf_rn(swa, d[1], d64[nb][1]);
                d64[nb][2] = __fmaf_rn(swb, d[2], d64[nb][2]);
                d64[nb][3] = __fmaf_rn(swb, d[3], d64[nb][3]);
              }
            }
          }
          // unit epilogue: activation scale (and the int4 affine bias term)
          #pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const int c0 = min(nb * 8 + 2 * t, M - 1), c1 = min(nb * 8 + 2 * t + 1, M - 1);
            const float x0 = xsc[c0 * units_max + u], x1 = xsc[c1 * units_max + u];
            if constexpr (I4) {
              const float m0 = xsum[c0 * units_max + u], m1 = xsum[c1 * units_max + u];
              d64[nb][0] = __fmaf_rn(sca[0], d64[nb][0], sca[1] * m0);
              d64[nb][1] = __fmaf_rn(sca[0], d64[nb][1], sca[1] * m1);
              d64[nb][2] = __fmaf_rn(scb[0], d64[nb][2], scb[1] * m0);
              d64[nb][3] = __fmaf_rn(scb[0], d64[nb][3], scb[1] * m1);
            }
            acc[r][nb][0] = __fmaf_rn(x0, d64[nb][0], acc[r][nb][0]);
            acc[r][nb][1] = __fmaf_rn(x1, d64[nb][1], acc[r][nb][1]);
            acc[r][nb][2] = __fmaf_rn(x0, d64[nb][2], acc[r][nb][2]);
            acc[r][nb][3] = __fmaf_rn(x1, d64[nb][3], acc[r][nb][3]);
          }
        }
      }
    }
    __syncthreads();   // the next pass overwrites the staged codes, scales and activations
  }

  // acc[r][nb]: c0 = (row 16r+g, col 2t), c1 = (16r+g, 2t+1), c2 = (16r+g+8, 2t), c3 = (16r+g+8, 2t+1).
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
  if (!ok_all) return;   // an expired wait leaves this CTA's outputs unwritten (status word set)
  constexpr bool X2 = F == MXFP4X2;                                         // output row = rows 2r + 2r + 1
  constexpr int OR = X2 ? ROWS / 2 : ROWS;                                  // output rows of the CTA
  for (int i = tid; i < OR * M; i += THREADS) {
    const int pr = i % OR, m = i / OR;
    const int r = X2 ? 2 * pr : pr;
    if (row0 + r >= N) continue;
    float sum = 0.0f;
    #pragma unroll
    for (int w = 0; w < WARPS; ++w) {
      sum += red[(size_t(w) * ROWS + r) * RC + m];
      if constexpr (X2) sum += red[(size_t(w) * ROWS + r + 1) * RC + m];    // the residual plane
    }
    if constexpr (F == NVFP4) sum *= glob;
    const int64_t o = X2 ? int64_t(m) * (N / 2) + row0 / 2 + pr : int64_t(m) * N + row0 + r;
    if (out_f32) static_cast<float*>(out)[o] = sum;
    else static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(sum);
  }
}

template <int F, int NB, int R>
inline size_t smem_bytes(int M, int KS) {
  const int units = KS / 64;
  return size_t(16 * R) * code_stride<F>(KS) + size_t(M) * (KS + 8) * 2 +
         size_t(M) * units * 4 * (is_i4<F>() ? 2 : 1) + size_t(16 * R) * sc_stride<F, R>(KS) * 4 +
         size_t(WARPS) * 16 * R * 8 * NB * 4;
}

// Shared memory per CTA is held under this budget (two or more CTAs per SM).
constexpr size_t SMEM_BUDGET = 112 * 1024;

// Codes per pass: the largest multiple of 64 (at most 8192, at most K
// rounded up) whose staged codes, activations and scales fit the budget.
template <int F, int NB, int R>
inline int stage_k(int M, int K) {
  int ks = (K + 63) / 64 * 64;
  ks = ks < 8192 ? ks : 8192;
  while (ks > 64 && smem_bytes<F, NB, R>(M, ks) > SMEM_BUDGET) ks -= 64;
  return ks;
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
  const int KS = stage_k<F, NB, R>(M, K);
  const size_t sm = smem_bytes<F, NB, R>(M, KS);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_done[dev].load()) {
    e = cudaFuncSetAttribute(qgemv_kernel<F, NB, R>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(SMEM_BUDGET));
    if (e != cudaSuccess) return e;
    attr_done[dev].store(1);
  }
  return launch_pdl(qgemv_kernel<F, NB, R>, dim3((N + 16 * R - 1) / (16 * R)), dim3(THREADS), sm, st, c, s, glob, x,
                    out, int(out_f32), M, N, K, KS, wait_limit_ns());
}

// Rows per CTA: 16 for M <= 2, 32 beyond (each staged activation then serves
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

cudaError_t read_and_clear_gemv_status(unsigned int* status) {
  cudaError_t e = cudaMemcpyFromSymbol(status, gemv::g_gemv_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(gemv::g_gemv_status, &zero, sizeof(unsigned int));
}

cudaError_t launch_qgemv(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                         bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms) {
  if (qgemv_m2_fits(fmt, M, K))
    return launch_qgemv_m2(fmt, codes, scales, glob, x, out, out_f32, M, N, K, st, sms);
  if (qgemv_rb_fits(fmt, M, N, K, sms))
    return launch_qgemv_rb(fmt, codes, scales, glob, x, out, out_f32, M, N, K, st, sms);
  if (M >= 3 && qgemv_mb_fits(fmt, M, K))
    return launch_qgemv_mb(fmt, codes, scales, glob, x, out, out_f32, M, N, K, st, sms);
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return gemv::launch_fmt<MXFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP4: return gemv::launch_fmt<NVFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP8_E4M3: return gemv::launch_fmt<MXFP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP8_E5M2: return gemv::launch_fmt<MXFP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP8: return gemv::launch_fmt<NVFP8>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP8_F16: return gemv::launch_fmt<NVFP8_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXINT8: return gemv::launch_fmt<MXINT8>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case INT8: return gemv::launch_fmt<INT8>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case INT8_F16: return gemv::launch_fmt<INT8_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case INT4: return gemv::launch_fmt<INT4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case INT4_F16: return gemv::launch_fmt<INT4_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP4X2: return gemv::launch_fmt<MXFP4X2>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXINT4: return gemv::launch_fmt<MXINT4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP4: return gemv::launch_fmt<FP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP4_F16: return gemv::launch_fmt<FP4_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP8_E4M3: return gemv::launch_fmt<FP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP8_E4M3_F16: return gemv::launch_fmt<FP8_E4M3_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP8_E5M2: return gemv::launch_fmt<FP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP8_E5M2_F16: return gemv::launch_fmt<FP8_E5M2_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    default: return gemv::launch_fmt<INT4_AFFINE>(codes, scales, glob, x, out, out_f32, m, n, k, st);
  }
}

}  // namespace qfmt_dev
