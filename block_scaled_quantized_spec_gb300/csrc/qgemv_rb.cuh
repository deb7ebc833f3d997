// Batch decode GEMV for 3 <= M <= 16 activation rows:
//   out[m, n] = sum_k x[m, k] * dequant(W)[n, k]
// (metaltile PR #250 qgemv commits; rlx-cpu thunk/ops/quant.rs
// lowp_scaled_matmul: per K block, the block's sum of products times its
// scales).
//
// The decode of the weights is what costs on the CUDA cores (E2M1 -> f16 runs
// at ~79 codes per SM and cycle), so one decode serves every activation row:
//  * mma.sync m16n8k16 with the weights as A (16 rows g, g + 8 of a tile) and
//    the activation rows as the 8 columns of B (a second MMA pair for rows
//    8-15): per 32-code block, lane t of a quad holds codes 8t .. 8t + 7 of
//    rows g and g + 8 and two MMAs cover the block, so D holds that block's
//    sums for 16 weight rows x 8 activation rows, which take the block's
//    weight scale and the activations' span scale in float32 (the E4M3 / E5M2
//    / E2M1 / int decodes to f16 are exact; nvfp4 multiplies its E4M3
//    micro-scales into the f16 weights, which is exact too).  nvfp8's float
//    scales come per 16 codes, so there lane t holds codes 4t .. 4t + 3 of
//    each 16-block and each MMA is one 16-block;
//  * the activations are bulk-copied into shared memory once per CTA (one
//    round trip) and each warp turns its k range into f16 in place, with a
//    power-of-two shift per 32 values (the span's largest |x| in [2^14,
//    2^15): exact for every bf16 within 2^29 of it), in the order the lanes'
//    codes pair up; a copy that does not land within the wait limit sets the
//    status word and the CTA stores nothing;
//  * one CTA per SM takes the 16-row tiles b, b + grid, ... (an even share of
//    the launch on every SM), its 16 warps split K; each warp's codes and
//    scales are loaded 16 (8-bit codes: 8) blocks ahead in registers, across
//    tile ends, and the first ones before the dependent wait; the CTA's rows
//    are prefetched into L2 as it starts;
//  * per tile the warps' partial sums meet in shared memory and one thread
//    per output stores it.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {
namespace gemv_rb {

constexpr int WARPS = 16, THREADS = 512;

template <int F>
struct Lay {
  static constexpr bool four = FmtTraits<F>::four;
  static constexpr bool B16 = FmtTraits<F>::block == 16 && !four;   // nvfp8: an MMA per 16-code block
  static constexpr bool I4 = is_i4<F>() || F == MXINT4;              // int4 pairing and span sums of x
  static constexpr bool X2 = F == MXFP4X2;                           // output row = weight rows 2r, 2r + 1
  static constexpr int CW = four ? 1 : 2;                            // code words a lane holds per row and block
  // blocks a warp holds ahead: a lane's 4 (8) bytes a row and block are small
  // loads, so many are in flight (~32 KiB an SM) to cover the memory latency
  static constexpr int PB = four ? 8 : 4;
};

// Staged activation row stride in halfwords: K plus 32 halfwords, so that
// rows start 64 bytes apart modulo 128 (the 8 rows of a B-fragment load fall
// in the two halves of the banks alternately).
__host__ __device__ constexpr int xrow(int K) { return K + 32 + ((K + 32) % 64 == 0 ? 32 : 0); }

inline size_t smem_bytes(int F, int M, int K) {
  const int spans = K / 32;
  const bool i4 = fmt_is_i4(F) || F == MXINT4;
  return size_t(M) * xrow(K) * 2 + 16 + size_t(spans) * 16 * 4 * (i4 ? 2 : 1) + size_t(WARPS) * 16 * 16 * 4 + 8;
}

// A copy that did not land in time (one word per translation unit that
// instantiates the kernel; read through Group<...>::read_status).
static __device__ unsigned int g_rb_status;

__device__ __forceinline__ bool rb_wait(uint32_t bar, uint64_t limit_ns) {
  auto done = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar)
        : "memory");
    return ok != 0u;
  };
  if (done()) return true;
  uint64_t t0, t1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  while (!done()) {
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    if (t1 - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void mma(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                    uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// A lane's 8 codes of one row and block -> four f16x2 in the staged pairing:
// (c0,c1) (c2,c3) (c4,c5) (c6,c7), or for the 4-bit integers (c0,c4) (c1,c5)
// (c2,c6) (c3,c7) holding 1024 + u (u the unsigned nibble).
template <int F>
__device__ __forceinline__ void dec8(const uint32_t (&w)[Lay<F>::CW], uint32_t r[4]) {
  if constexpr (Lay<F>::I4) {
    const uint32_t u = i4_u<F>(w[0]);
    #pragma unroll
    for (int b = 0; b < 4; ++b) r[b] = ((u >> (4 * b)) & 0x000F000Fu) | 0x64006400u;
  } else if constexpr (Lay<F>::four) {
    asm("{.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;}"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
        : "r"(w[0]));
  } else {
    elem8x4_f16<F>(w[0], r);
    elem8x4_f16<F>(w[1], r + 2);
  }
}

// The raw scale words a lane keeps per row and block.
struct BS {
  uint32_t a, b;   // rows g and g + 8 (nvfp8: the first 16-block)
  uint32_t a2, b2; // nvfp8: the second 16-block
};

template <int F, int NB>
__global__ void __launch_bounds__(THREADS, 1) qgemv_rb_kernel(const uint8_t* __restrict__ codes,
                                                             const uint8_t* __restrict__ scales, float glob,
                                                             const uint16_t* __restrict__ x, void* __restrict__ out,
                                                             int out_f32, int M, int N, int K, uint64_t limit_ns,
                                                             int drop) {
  using LY = Lay<F>;
  constexpr int CW = LY::CW, PB = LY::PB;
  constexpr int B = FmtTraits<F>::block, SB = FmtTraits<F>::sbytes;
  extern __shared__ __align__(16) uint8_t smem[];
  const int XR = xrow(K);
  const int spans = K / 32;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                        // [M][XR] f16
  uint4* xzero = reinterpret_cast<uint4*>(xs + size_t(M) * XR);             // 16 zero bytes
  float* xsc = reinterpret_cast<float*>(xzero + 1);                          // [span][16] 2^-shift
  float* xsum = xsc + spans * 16;                                            // [span][16] (int4)
  float* red = xsum + (LY::I4 ? spans * 16 : 0);                             // [warp][16 rows][16 acts]
  uint64_t* xbar = reinterpret_cast<uint64_t*>(red + WARPS * 256);           // the activation copies landed

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int ntiles = (N + 15) / 16;
  const int G = int(gridDim.x);
  const int ntl = (ntiles - int(blockIdx.x) + G - 1) / G;                   // this CTA's tiles b, b + G, ...
  const int bw0 = warp * spans / WARPS, nbw = (warp + 1) * spans / WARPS - bw0;   // this warp's blocks
  const int64_t rowb = LY::four ? K / 2 : K;
  const int64_t srow = int64_t((K + B - 1) / B) * SB;                       // scale bytes a row

  // the CTA's weight rows towards L2
  if (warp == 0 && lane < 16) {
    for (int j = 0; j < ntl; ++j) {
      const int r = (int(blockIdx.x) + j * G) * 16 + lane;
      if (r < N) prefetch_l2(codes + int64_t(r) * rowb, uint64_t(rowb));
    }
  }

  // Items in order: tile ti, block bw0 + j of rows g and g + 8; the k-th
  // item of the warp is held in slot k % PB.  Load position: tile lt, block
  // lj, with the tile's row pointers.
  uint32_t wa[PB][CW], wb[PB][CW];
  BS bs[PB];
  int lt = 0, lj = 0;
  const uint8_t *lca = nullptr, *lcb = nullptr, *lsa = nullptr, *lsb = nullptr;
  auto set_rows = [&]() {
    const int row0 = (int(blockIdx.x) + lt * G) * 16;
    const int ra = min(row0 + g, N - 1), rb = min(row0 + g + 8, N - 1);      // rows past N: never stored
    lca = codes + int64_t(ra) * rowb;
    lcb = codes + int64_t(rb) * rowb;
    lsa = scales + int64_t(ra) * srow;
    lsb = scales + int64_t(rb) * srow;
  };
  auto load_next = [&](int i) {
    if (lt >= ntl) return;
    const int blk = bw0 + lj;
    if constexpr (LY::four) {
      wa[i][0] = __ldg(reinterpret_cast<const uint32_t*>(lca + 16 * blk + 4 * t));
      wb[i][0] = __ldg(reinterpret_cast<const uint32_t*>(lcb + 16 * blk + 4 * t));
    } else if constexpr (LY::B16) {
      wa[i][0] = __ldg(reinterpret_cast<const uint32_t*>(lca + 32 * blk + 4 * t));
      wa[i][1] = __ldg(reinterpret_cast<const uint32_t*>(lca + 32 * blk + 16 + 4 * t));
      wb[i][0] = __ldg(reinterpret_cast<const uint32_t*>(lcb + 32 * blk + 4 * t));
      wb[i][1] = __ldg(reinterpret_cast<const uint32_t*>(lcb + 32 * blk + 16 + 4 * t));
    } else {
      const uint2 va = __ldg(reinterpret_cast<const uint2*>(lca + 32 * blk + 8 * t));
      const uint2 vb = __ldg(reinterpret_cast<const uint2*>(lcb + 32 * blk + 8 * t));
      wa[i][0] = va.x; wa[i][1] = va.y;
      wb[i][0] = vb.x; wb[i][1] = vb.y;
    }
    if constexpr (is_e8m0<F>()) {
      bs[i].a = __ldg(lsa + blk);
      bs[i].b = __ldg(lsb + blk);
    } else if constexpr (F == NVFP4) {                                       // the lane's 16-block: 2 blk + t / 2
      bs[i].a = __ldg(lsa + 2 * blk + (t >> 1));
      bs[i].b = __ldg(lsb + 2 * blk + (t >> 1));
    } else if constexpr (LY::B16) {
      bs[i].a = __float_as_uint(float_scale<F>(lsa, 2 * blk));
      bs[i].a2 = __float_as_uint(float_scale<F>(lsa, 2 * blk + 1));
      bs[i].b = __float_as_uint(float_scale<F>(lsb, 2 * blk));
      bs[i].b2 = __float_as_uint(float_scale<F>(lsb, 2 * blk + 1));
    } else if constexpr (LY::I4) {                                           // int4 affine / sym: per 64
      bs[i].a = i4_word<F>(lsa, blk / 2);
      bs[i].b = i4_word<F>(lsb, blk / 2);
    } else {                                                                 // float scale per 32 or 64
      bs[i].a = __float_as_uint(float_scale<F>(lsa, blk * 32 / B));
      bs[i].b = __float_as_uint(float_scale<F>(lsb, blk * 32 / B));
    }
    if (++lj == nbw) {
      lj = 0;
      if (++lt < ntl) set_rows();
    }
  };
  set_rows();
  #pragma unroll
  for (int i = 0; i < PB; ++i) load_next(i);

  const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(xbar));
  if (tid == 0) {
    *xzero = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // The activations may be the preceding kernel's output: one bulk copy a row.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (warp == 0) {
    if (lane == 0)
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(uint32_t(M) * uint32_t(K) * 2u)
                   : "memory");
    __syncwarp();
    if (lane < M && !drop)
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                   ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(xs + size_t(lane) * XR))),
                   "l"(x + int64_t(lane) * K), "r"(uint32_t(K) * 2u), "r"(bar)
                   : "memory");
  }
  if (!__syncthreads_and(rb_wait(bar, limit_ns))) {
    if (tid == 0) {   // nothing stored; the copies land before the CTA leaves
      atomicOr(&g_rb_status, 1u);
      rb_wait(bar, limit_ns);
    }
    return;
  }

  // ---- this warp's k range to f16 in place: 4 lanes a (row, span) ----------
  {
    const int tasks = M * nbw;                                              // (row, span) pairs of this warp
    int m = (lane >> 2) / nbw, sp = (lane >> 2) % nbw;                       // task lane / 4, then 8 on
    const int dm = 8 / nbw, dsp = 8 % nbw;
    for (int q0 = 0; q0 < tasks; q0 += 8) {
      const bool live = q0 + (lane >> 2) < tasks;
      const uint16_t* src = xs + size_t(live ? m : 0) * XR + 32 * (bw0 + sp);   // the raw bf16 copy
      uint32_t h[4];
      if constexpr (LY::B16) {                                              // values 4t .. 4t+3, 16 + 4t .. 16 + 4t + 3
        const uint2 u0 = live ? *reinterpret_cast<const uint2*>(src + 4 * t) : make_uint2(0u, 0u);
        const uint2 u1 = live ? *reinterpret_cast<const uint2*>(src + 16 + 4 * t) : make_uint2(0u, 0u);
        h[0] = u0.x; h[1] = u0.y; h[2] = u1.x; h[3] = u1.y;
      } else {
        const uint4 u = live ? *reinterpret_cast<const uint4*>(src + 8 * t) : make_uint4(0u, 0u, 0u, 0u);
        h[0] = u.x; h[1] = u.y; h[2] = u.z; h[3] = u.w;
      }
      __syncwarp();                                                         // the span is read before it is rewritten
      // the span's largest |x| (4 lanes), its shift to [2^14, 2^15)
      uint32_t mx = 0;
      #pragma unroll
      for (int j = 0; j < 4; ++j) mx = max(mx, max(h[j] & 0x7FFFu, (h[j] >> 16) & 0x7FFFu));
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      const int E = int(mx >> 7);
      int sh = (mx == 0u || E == 255) ? 0 : 141 - E;                        // 14 - (E - 127)
      sh = sh > 126 ? 126 : sh;
      const float up = __uint_as_float(uint32_t(sh + 127) << 23);
      float f[8];
      #pragma unroll
      for (int j = 0; j < 4; ++j) {
        f[2 * j] = __fmul_rn(__uint_as_float(h[j] << 16), up);
        f[2 * j + 1] = __fmul_rn(__uint_as_float(h[j] & 0xFFFF0000u), up);
      }
      uint32_t o[4];
      if constexpr (LY::I4) {
        #pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = pack_f16x2(f[j], f[j + 4]);
      } else {
        #pragma unroll
        for (int j = 0; j < 4; ++j) o[j] = pack_f16x2(f[2 * j], f[2 * j + 1]);
      }
      if (live) *reinterpret_cast<uint4*>(xs + size_t(m) * XR + 32 * (bw0 + sp) + 8 * t) = make_uint4(o[0], o[1], o[2], o[3]);
      if constexpr (LY::I4) {                                               // the span's sum of staged values
        float sm = 0.0f;
        #pragma unroll
        for (int j = 0; j < 4; ++j) sm += f16x2_lo(o[j]) + f16x2_hi(o[j]);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 1);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 2);
        if (live && t == 0) xsum[(bw0 + sp) * 16 + m] = sm;
      }
      if (live && t == 0) xsc[(bw0 + sp) * 16 + m] = __uint_as_float(uint32_t(127 - sh) << 23);
      m += dm;                                                              // the work item 8 further on
      sp += dsp;
      if (sp >= nbw) {
        sp -= nbw;
        ++m;
      }
    }
  }
  __syncwarp();

  // B fragments: lane (g, t) supplies activation row g (+ 8), or zeros past M
  const uint16_t* xb[NB];
  int xstep[NB];
  #pragma unroll
  for (int c = 0; c < NB; ++c) {
    const int m = 8 * c + g;
    xb[c] = m < M ? xs + size_t(m) * XR + 8 * t + 32 * bw0 : reinterpret_cast<const uint16_t*>(xzero);
    xstep[c] = m < M ? 32 : 0;
  }
  // D columns of this lane: activation rows 2t, 2t + 1 (+ 8)
  float acc[NB][4];
  #pragma unroll
  for (int c = 0; c < NB; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;

  int ct = 0, cj = 0;                                                       // the item computed next
  while (ct < ntl) {
    #pragma unroll
    for (int i = 0; i < PB; ++i) {
      if (ct >= ntl) break;
      uint32_t fa[4], fb[4];
      dec8<F>(wa[i], fa);
      dec8<F>(wb[i], fb);
      if constexpr (F == NVFP4) {                                            // E2M1 x E4M3 is exact in f16
        uint32_t pa, pb;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(pa) : "h"(uint16_t(bs[i].a)));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(pb) : "h"(uint16_t(bs[i].b)));
        pa = prmt(pa, 0u, 0x1010u);
        pb = prmt(pb, 0u, 0x1010u);
        #pragma unroll
        for (int e = 0; e < 4; ++e) {
          fa[e] = mul_f16x2(fa[e], pa);
          fb[e] = mul_f16x2(fb[e], pb);
        }
      }
      // the lane's weight scales of this block
      float qa = 1.0f, qb = 1.0f;
      if constexpr (is_e8m0<F>()) {
        qa = e8m0_f32(bs[i].a);
        qb = e8m0_f32(bs[i].b);
      } else if constexpr (!LY::I4 && !LY::B16 && F != NVFP4) {
        qa = __uint_as_float(bs[i].a);
        qb = __uint_as_float(bs[i].b);
      }
      const int blk = bw0 + cj;
      const float2* scp = reinterpret_cast<const float2*>(xsc + blk * 16);
      const float2* ssp = reinterpret_cast<const float2*>(xsum + blk * 16);
      #pragma unroll
      for (int c = 0; c < NB; ++c) {
        const uint4 xv = *reinterpret_cast<const uint4*>(xb[c] + cj * xstep[c]);
        const float2 xs2 = scp[4 * c + t];                                   // activation rows 8c + 2t, + 1
        float d0[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if constexpr (LY::B16) {                                             // one 16-block an MMA
          float d1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          mma(d0, fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
          mma(d1, fa[2], fb[2], fa[3], fb[3], xv.z, xv.w);
          const float sa = __uint_as_float(bs[i].a), sa2 = __uint_as_float(bs[i].a2);
          const float sb = __uint_as_float(bs[i].b), sb2 = __uint_as_float(bs[i].b2);
          acc[c][0] = __fmaf_rn(xs2.x, __fmaf_rn(sa, d0[0], sa2 * d1[0]), acc[c][0]);
          acc[c][1] = __fmaf_rn(xs2.y, __fmaf_rn(sa, d0[1], sa2 * d1[1]), acc[c][1]);
          acc[c][2] = __fmaf_rn(xs2.x, __fmaf_rn(sb, d0[2], sb2 * d1[2]), acc[c][2]);
          acc[c][3] = __fmaf_rn(xs2.y, __fmaf_rn(sb, d0[3], sb2 * d1[3]), acc[c][3]);
        } else {
          mma(d0, fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
          mma(d0, fa[2], fb[2], fa[3], fb[3], xv.z, xv.w);
          if constexpr (F == MXINT4) {                                       // D = sum x~ (1032 + q)
            const float2 sm = ssp[4 * c + t];
            acc[c][0] = __fmaf_rn(__fmul_rn(qa, xs2.x), __fmaf_rn(-1032.0f, sm.x, d0[0]), acc[c][0]);
            acc[c][1] = __fmaf_rn(__fmul_rn(qa, xs2.y), __fmaf_rn(-1032.0f, sm.y, d0[1]), acc[c][1]);
            acc[c][2] = __fmaf_rn(__fmul_rn(qb, xs2.x), __fmaf_rn(-1032.0f, sm.x, d0[2]), acc[c][2]);
            acc[c][3] = __fmaf_rn(__fmul_rn(qb, xs2.y), __fmaf_rn(-1032.0f, sm.y, d0[3]), acc[c][3]);
          } else if constexpr (LY::I4) {                                     // s D + (b - 1024 s) sum(x~)
            const float2 sm = ssp[4 * c + t];
            float sa, ba, sb, bb;
            i4_scale_bias<F>(bs[i].a, sa, ba);
            i4_scale_bias<F>(bs[i].b, sb, bb);
            ba = __fmaf_rn(-1024.0f, sa, ba);
            bb = __fmaf_rn(-1024.0f, sb, bb);
            acc[c][0] = __fmaf_rn(xs2.x, __fmaf_rn(sa, d0[0], ba * sm.x), acc[c][0]);
            acc[c][1] = __fmaf_rn(xs2.y, __fmaf_rn(sa, d0[1], ba * sm.y), acc[c][1]);
            acc[c][2] = __fmaf_rn(xs2.x, __fmaf_rn(sb, d0[2], bb * sm.x), acc[c][2]);
            acc[c][3] = __fmaf_rn(xs2.y, __fmaf_rn(sb, d0[3], bb * sm.y), acc[c][3]);
          } else {                                                           // (nvfp4: micro-scales in the weights)
            acc[c][0] = __fmaf_rn(__fmul_rn(qa, xs2.x), d0[0], acc[c][0]);
            acc[c][1] = __fmaf_rn(__fmul_rn(qa, xs2.y), d0[1], acc[c][1]);
            acc[c][2] = __fmaf_rn(__fmul_rn(qb, xs2.x), d0[2], acc[c][2]);
            acc[c][3] = __fmaf_rn(__fmul_rn(qb, xs2.y), d0[3], acc[c][3]);
          }
        }
      }
      load_next(i);                                                          // the slot's next item
      if (++cj == nbw) {
        // ---- the tile's last block: partial sums of the warps meet -------------
        const int row0 = (int(blockIdx.x) + ct * G) * 16;
        #pragma unroll
        for (int c = 0; c < NB; ++c) {
          float* rw = red + warp * 256;
          rw[g * 16 + 8 * c + 2 * t] = acc[c][0];
          rw[g * 16 + 8 * c + 2 * t + 1] = acc[c][1];
          rw[(g + 8) * 16 + 8 * c + 2 * t] = acc[c][2];
          rw[(g + 8) * 16 + 8 * c + 2 * t + 1] = acc[c][3];
          acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;
        }
        __syncthreads();
        constexpr int OR = LY::X2 ? 8 : 16;                                  // output rows of the tile
        if (tid < OR * M) {
          const int m = tid / OR, pr = tid % OR;
          const int rr = LY::X2 ? 2 * pr : pr;
          if (row0 + rr < N) {
            float sum = 0.0f;
            #pragma unroll
            for (int w = 0; w < WARPS; ++w) {
              sum += red[w * 256 + rr * 16 + m];
              if constexpr (LY::X2) sum += red[w * 256 + (rr + 1) * 16 + m];   // the residual plane
            }
            if constexpr (F == NVFP4) sum *= glob;
            const int64_t o = LY::X2 ? int64_t(m) * (N / 2) + row0 / 2 + pr : int64_t(m) * N + row0 + rr;
            if (out_f32) static_cast<float*>(out)[o] = sum;
            else static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(sum);
          }
        }
        __syncthreads();
        cj = 0;
        ++ct;
      }
    }
  }
}

template <int F, int NB>
static cudaError_t launch_nb(const void* codes, const void* scales, float glob, const void* x, void* out,
                             bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
  const uint64_t limit = wait_limit_ns();
  const int drop = drop_arrivals();
  static std::atomic<int> attr_done[64];
  const size_t sm = smem_bytes(F, M, K);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_done[dev].load()) {
    e = cudaFuncSetAttribute(qgemv_rb_kernel<F, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(1);
  }
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(unsigned(std::min((N + 15) / 16, sms)));
  lc.blockDim = dim3(THREADS);
  lc.dynamicSmemBytes = sm;
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, qgemv_rb_kernel<F, NB>, static_cast<const uint8_t*>(codes),
                            static_cast<const uint8_t*>(scales), glob, static_cast<const uint16_t*>(x), out,
                            int(out_f32), M, N, K, limit, drop);
}

// The entry points of one group of formats.
template <int... Fs>
struct Group {
  static cudaError_t launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                            bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
    cudaError_t r = cudaErrorInvalidValue;
    (void)((fmt == Fs && ((r = M <= 8 ? launch_nb<Fs, 1>(codes, scales, glob, x, out, out_f32, M, N, K, st, sms)
                                      : launch_nb<Fs, 2>(codes, scales, glob, x, out, out_f32, M, N, K, st, sms)),
                          true)) ||
           ...);
    return r;
  }
  static cudaError_t read_status(unsigned int* status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_rb_status, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_rb_status, &zero, sizeof(unsigned int));
  }
};

using GroupE2M1 = Group<MXFP4, NVFP4, MXFP4X2, MXINT4, FP4, FP4_F16>;
using GroupInt = Group<INT4_AFFINE, INT4, INT4_F16, MXINT8, INT8, INT8_F16>;
using GroupFp8 = Group<MXFP8_E4M3, MXFP8_E5M2, NVFP8, NVFP8_F16, FP8_E4M3, FP8_E4M3_F16, FP8_E5M2, FP8_E5M2_F16>;

cudaError_t e2m1_launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                        bool out_f32, int M, int N, int K, cudaStream_t st, int sms);
cudaError_t intg_launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                        bool out_f32, int M, int N, int K, cudaStream_t st, int sms);
cudaError_t fp8_launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                       bool out_f32, int M, int N, int K, cudaStream_t st, int sms);
cudaError_t e2m1_status(unsigned int* status);
cudaError_t intg_status(unsigned int* status);
cudaError_t fp8_status(unsigned int* status);

}  // namespace gemv_rb
}  // namespace qfmt_dev
