// Batch decode GEMV, 3 <= M <= 16:
//   out[m, n] = sum_k x[m, k] * dequant(W)[n, k]
// (metaltile PR #250 qmm commits: the multi-row decode qmm, one dequantized
// weight tile reused across the batch rows; rlx-cpu thunk/ops/quant.rs
// lowp_scaled_matmul, which applies each block's scale to that block's partial
// sum).
//
// Here the weight stream is shared by up to 16 activation rows, so the
// tensor-core work per weight byte grows with M and the kernel is built for
// throughput rather than for the latency of one launch:
//  * a CTA (4 warps) owns 64 weight rows, 16 per warp, and a K range; K is
//    split over a thread-block cluster of S CTAs so each CTA's activation
//    slice (M x K/S, staged once as f16) fits in shared memory; the S partial
//    sums meet through distributed shared memory, summed in rank order;
//  * each lane reads word t of every 16-byte segment of its two rows (g and
//    g + 8) straight into registers, four 64-byte chunks ahead, so the four
//    lanes of a quad hold one segment and every mma.sync k-slice lies inside
//    one scale block;
//  * codes become f16 with the hardware conversions (int4 as 1024 + q; nvfp4
//    applies its E4M3 micro-scale in f16, exact); all 8 B columns carry
//    activation rows (a second column block for 9 <= M <= 16);
//  * block scales multiply the float32 result of each segment's MMAs; the
//    activations' power-of-two scale (one per 128 values and row) multiplies
//    each chunk's float32 sum; int4 affine adds bias x sum(x) per block;
//  * the launch is programmatic-dependent: weights and scales are requested
//    before waiting on the preceding kernel, the activations after.
#include <cuda_runtime.h>

#include <atomic>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {
namespace gemv_mb {

constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr int ROWS = 16 * WARPS;        // weight rows per CTA
constexpr int XSPAN = 128;              // activations sharing one power-of-two scale
constexpr size_t X_BUDGET = 40 * 1024;  // staged f16 activations per CTA (five CTAs per SM)

// 64-byte chunks per lane in flight: four; two for nvfp8 and int4 affine,
// whose per-chunk scales (eight float32, four scale/bias pairs) stay in registers
template <int F>
constexpr int chunks_in_flight() { return (is_fs8<F>() || is_i4<F>() || is_fp4f<F>()) ? 2 : 4; }

template <int F>
struct Shape {
  static constexpr bool four = FmtTraits<F>::four;
  static constexpr int CODES = four ? 128 : 64;   // codes per row in one 64-byte chunk
  static constexpr int SEG = CODES / 4;           // codes per 16-byte segment
  static constexpr int WORD = SEG / 4;            // codes per 32-bit word (8 or 4)
};

__device__ __forceinline__ void mma_f16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// As above with a zero accumulator input (the first MMA of a scale block).
__device__ __forceinline__ void mma_f16_z(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void mma_bf16_z(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                           uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
      : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// 8 E2M1 codes -> f16x2 (c0,c1) (c2,c3) (c4,c5) (c6,c7).
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

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t ldg_word(const uint8_t* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Staged activation row stride in halfwords for a K range of kr values.  A
// B-operand read covers rb bytes of each of 128 / rb consecutive rows at once
// (64 for the 16-byte reads of the 4-bit formats, 32 for the 8-byte reads of
// the 8-bit ones); rows that start rb bytes apart modulo 128 use disjoint banks.
__host__ __device__ constexpr int xstride(int kr, int rb) {
  const int bytes = 2 * kr;
  const int pad = ((rb - bytes % 128) + 128) % 128;
  return (bytes + pad) / 2;
}

template <int F>
__host__ __device__ constexpr int read_bytes() { return FmtTraits<F>::four ? 64 : 32; }

// 16-byte asynchronous copy global -> shared; pred false zero-fills without
// reading the source.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(pred ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// float at the same shared-memory offset in cluster CTA `rank`
__device__ __forceinline__ float ld_cluster_f32(const float* p, uint32_t rank) {
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  uint32_t r;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(r) : "memory");
  return v;
}

// Shared memory of one CTA: staged activations [M][xst] f16, their scales
// [M][kr/128 + 1] (and int4-affine span sums [M][kr/64 + 1]), the partial tile [64][16].
inline size_t smem_bytes(int F, int M, int kr) {
  const int rb = fmt_is_four(F) ? 64 : 32;
  return size_t(M) * xstride(kr, rb) * 2 + size_t(M) * (kr / XSPAN + 1) * 4 +
         (fmt_is_i4(F) ? size_t(M) * (kr / 64 + 1) * 4 : 0) + size_t(ROWS) * 16 * 4;
}

// Raw scale words a lane keeps per chunk: 2 (rows g, g + 8) for the byte
// scales, 4 for int4 affine (two blocks), 8 for nvfp8 (four float32 blocks).
template <int F>
constexpr int scale_words() { return (is_fs8<F>() || is_fp4f<F>()) ? 8 : (is_i4<F>() ? 4 : 2); }

template <int F, int NB, bool UNI>
__global__ void __launch_bounds__(THREADS, 5) qgemv_mb_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales, float glob,
                                                           const uint16_t* __restrict__ x, void* __restrict__ out,
                                                           int out_f32, int M, int N, int K, int KR) {
  using S = Shape<F>;
  constexpr bool FOUR = S::four, I4 = is_i4<F>();
  constexpr int CODES = S::CODES, SEG = S::SEG;
  constexpr int BLK = FmtTraits<F>::block, SB = FmtTraits<F>::sbytes;
  constexpr int SW = scale_words<F>();
  constexpr int P = chunks_in_flight<F>();
  extern __shared__ __align__(16) uint8_t smem[];
  const int xst = xstride(KR, read_bytes<F>());
  // Row strides of the activation scales and span sums, one float longer than
  // the row: the lanes of a quad read rows 2t and 2t + 1, which then fall in
  // different banks.
  const int nsp = KR / XSPAN + 1, nsm = KR / 64 + 1;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                         // [M][xst] f16
  float* xsc = reinterpret_cast<float*>(xs + size_t(M) * xst);              // [M][nsp] 2^-shift
  float* xsum = xsc + M * nsp;                                              // [M][nsm] (int4 affine)
  float* red = xsum + (I4 ? M * nsm : 0);                                   // [ROWS][16] partial tile

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * ROWS;
  const int k0 = blockIdx.y * KR;
  const int k1 = min(K, k0 + KR);
  const int nch = k1 > k0 ? (k1 - k0 + CODES - 1) / CODES : 0;
  const int ra = row0 + 16 * warp + g, rb = ra + 8;
  const bool va = ra < N, vb = rb < N;                                      // rows past N read row 0, never stored
  const int64_t rowbytes = FOUR ? K / 2 : K;
  const int64_t nblk = (K + BLK - 1) / BLK;   // int4 affine: a ragged last group
  const uint8_t* pa = codes + int64_t(va ? ra : 0) * rowbytes + (FOUR ? k0 / 2 : k0) + 4 * t;
  const uint8_t* pb = codes + int64_t(vb ? rb : 0) * rowbytes + (FOUR ? k0 / 2 : k0) + 4 * t;
  const uint8_t* sra = scales + int64_t(va ? ra : 0) * nblk * SB;
  const uint8_t* srb = scales + int64_t(vb ? rb : 0) * nblk * SB;

  // This CTA's weight rows towards L2 now (rounds after the first read them there).
  if (tid < ROWS && row0 + tid < N && k1 > k0) {
    const uint8_t* p = codes + int64_t(row0 + tid) * rowbytes + (FOUR ? k0 / 2 : k0);
    prefetch_l2(p, uint64_t(FOUR ? (k1 - k0) / 2 : (k1 - k0)));
  }

  uint32_t wa[P][4], wb[P][4];     // word t of the chunk's four segments, rows g and g + 8
  uint32_t sc[P][SW];

  auto load_chunk = [&](int c, int i) {
    #pragma unroll
    for (int sg = 0; sg < 4; ++sg) {
      // UNI: every CTA's K range is whole and a multiple of P chunks
      const bool ok = UNI || (c < nch && k0 + c * CODES + sg * SEG < k1);
      wa[i][sg] = ok ? ldg_word(pa + int64_t(c) * 64 + 16 * sg) : 0u;
      wb[i][sg] = ok ? ldg_word(pb + int64_t(c) * 64 + 16 * sg) : 0u;
    }
    const int kc = k0 + c * CODES;                                          // first k of the chunk
    auto live = [&](int k) { return UNI || (c < nch && k < k1); };
    if constexpr (is_mx4<F>()) {                                            // one E8M0 block per segment
      uint32_t a = 0, b = 0;
      #pragma unroll
      for (int sg = 0; sg < 4; ++sg) {
        const int k = kc + sg * SEG;
        a |= (live(k) ? uint32_t(__ldg(sra + k / 32)) : 127u) << (8 * sg);
        b |= (live(k) ? uint32_t(__ldg(srb + k / 32)) : 127u) << (8 * sg);
      }
      sc[i][0] = a;
      sc[i][1] = b;
    } else if constexpr (F == NVFP4) {                                      // the micro-block of this lane's word
      uint32_t a = 0, b = 0;
      #pragma unroll
      for (int sg = 0; sg < 4; ++sg) {
        const int k = kc + sg * SEG + 8 * t;
        a |= (live(k) ? uint32_t(__ldg(sra + k / 16)) : 0u) << (8 * sg);
        b |= (live(k) ? uint32_t(__ldg(srb + k / 16)) : 0u) << (8 * sg);
      }
      sc[i][0] = a;
      sc[i][1] = b;
    } else if constexpr (is_mx8<F>()) {                                     // segments 0-1 and 2-3 share a block
      uint32_t a = 0, b = 0;
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = kc + h * 32;
        a |= (live(k) ? uint32_t(__ldg(sra + k / 32)) : 127u) << (8 * h);
        b |= (live(k) ? uint32_t(__ldg(srb + k / 32)) : 127u) << (8 * h);
      }
      sc[i][0] = a;
      sc[i][1] = b;
    } else if constexpr (is_fs8<F>() || is_fp4f<F>()) {                     // each segment's block scale
      #pragma unroll
      for (int sg = 0; sg < 4; ++sg) {
        const int k = kc + sg * SEG;
        sc[i][sg] = live(k) ? __float_as_uint(float_scale<F>(sra, k / FmtTraits<F>::block)) : 0u;
        sc[i][4 + sg] = live(k) ? __float_as_uint(float_scale<F>(srb, k / FmtTraits<F>::block)) : 0u;
      }
    } else {                                                                // int4 affine: (scale, bias) per 64
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = kc + h * 64;
        sc[i][h] = live(k) ? i4_word<F>(sra, k / 64) : 0u;
        sc[i][2 + h] = live(k) ? i4_word<F>(srb, k / 64) : 0u;
      }
    }
  };

  #pragma unroll
  for (int i = 0; i < P; ++i) load_chunk(i, i);

  // The activations may be the preceding kernel's output.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- stage the activations [k0, k0 + KR) of all M rows as scaled f16 -----
  // 16 values per task: copied as bf16 by cp.async (every task's copy in
  // flight at once), then converted in place by the same thread; 8 tasks (8
  // consecutive lanes) share one 128-value span and its power-of-two scale.
  {
    const uint32_t xsa = static_cast<uint32_t>(__cvta_generic_to_shared(xs));
    const int per_m = KR / 16;
    const int tasks = M * per_m;
    const int iters = (tasks + THREADS - 1) / THREADS;
    // i / per_m as a multiply-high: exact for i < 16 per_m < 2^32 / per_m
    const uint32_t pm_magic = 0xFFFFFFFFu / uint32_t(per_m) + 1u;
    // Every row group reads the same activation lines: each CTA starts at its
    // own place in the slice (a whole 128-value span, so the groups of 8
    // lanes below stay aligned), spreading the requests over the L2 slices.
    const int rot = 8 * int((blockIdx.x * 37u) % uint32_t(tasks / 8));
    auto task = [&](int i) { return i + rot < tasks ? i + rot : i + rot - tasks; };
    for (int j = 0; j < iters; ++j) {
      const int i = task(tid + j * THREADS);
      if (tid + j * THREADS < tasks) {
        const int m = int(__umulhi(uint32_t(i), pm_magic)), kk = (i - m * per_m) * 16;
        const bool ok = k0 + kk < k1;
        const uint16_t* src = ok ? x + int64_t(m) * K + k0 + kk : x;
        const uint32_t dst = xsa + uint32_t((m * xst + kk) * 2);
        cp_async16(dst, src, ok);
        cp_async16(dst + 16, ok ? src + 8 : x, ok);
      }
    }
    cp_async_wait_all();
    if constexpr (I4) {
      // int4 affine multiplies bf16 activations as given: only the pairing
      // (x0,x4) (x1,x5) (x2,x6) (x3,x7) per 8 values, and float32 sums per 64
      for (int j = 0; j < iters; ++j) {
        const bool live = tid + j * THREADS < tasks;                        // whole 4-lane groups
        const int i = task(tid + j * THREADS);
        const int m = live ? int(__umulhi(uint32_t(i), pm_magic)) : 0;
        const int kk = live ? (i - m * per_m) * 16 : 0;
        uint4* p16 = reinterpret_cast<uint4*>(xs + m * xst + kk);
        const uint4 v0 = live ? p16[0] : make_uint4(0, 0, 0, 0);
        const uint4 v1 = live ? p16[1] : make_uint4(0, 0, 0, 0);
        float sm = 0.0f;
        const uint32_t h[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        #pragma unroll
        for (int q = 0; q < 8; ++q) sm += bf16bits_f32(h[q] & 0xFFFFu) + bf16bits_f32(h[q] >> 16);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 1);
        sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 2);
        if (live) {
          p16[0] = make_uint4(prmt(v0.x, v0.z, 0x5410u), prmt(v0.x, v0.z, 0x7632u), prmt(v0.y, v0.w, 0x5410u),
                              prmt(v0.y, v0.w, 0x7632u));
          p16[1] = make_uint4(prmt(v1.x, v1.z, 0x5410u), prmt(v1.x, v1.z, 0x7632u), prmt(v1.y, v1.w, 0x5410u),
                              prmt(v1.y, v1.w, 0x7632u));
          if ((kk & 63) == 0) xsum[m * nsm + (kk >> 6)] = sm;
        }
      }
    } else {
    for (int j = 0; j < iters; ++j) {
      const bool live = tid + j * THREADS < tasks;                          // whole 8-lane groups
      const int i = task(tid + j * THREADS);
      const int m = live ? int(__umulhi(uint32_t(i), pm_magic)) : 0;
      const int kk = live ? (i - m * per_m) * 16 : 0;
      uint4* p16 = reinterpret_cast<uint4*>(xs + m * xst + kk);
      const uint4 v0 = live ? p16[0] : make_uint4(0, 0, 0, 0);
      const uint4 v1 = live ? p16[1] : make_uint4(0, 0, 0, 0);
      const uint32_t h[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t m2 = 0;
      #pragma unroll
      for (int q = 0; q < 8; ++q) m2 = max_u16x2(m2, h[q] & 0x7FFF7FFFu);
      uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
      mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
      const int E = int(mx >> 7);
      int sh = (mx == 0u || E == 255) ? 0 : 141 - E;                         // max |x| to [2^14, 2^15)
      sh = sh > 126 ? 126 : sh;
      const float up = __uint_as_float(uint32_t(sh + 127) << 23);
      float f[16];
      #pragma unroll
      for (int q = 0; q < 8; ++q) {
        f[2 * q] = __fmul_rn(__uint_as_float(h[q] << 16), up);
        f[2 * q + 1] = __fmul_rn(__uint_as_float(h[q] & 0xFFFF0000u), up);
      }
      uint32_t o[8];
      #pragma unroll
      for (int q = 0; q < 8; ++q) o[q] = pack_f16x2(f[2 * q], f[2 * q + 1]);
      if (live) {
        p16[0] = make_uint4(o[0], o[1], o[2], o[3]);
        p16[1] = make_uint4(o[4], o[5], o[6], o[7]);
      }
      if (live && (kk & (XSPAN - 1)) == 0) xsc[m * nsp + kk / XSPAN] = __uint_as_float(uint32_t(127 - sh) << 23);
    }
    }
  }
  __syncthreads();

  // ---- multiply: chunk by chunk, slot i refilled as soon as it is consumed --
  int mrow[NB], mc0[NB], mc1[NB];            // B row of this lane; activation rows of its D columns
  #pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    mrow[nb] = min(8 * nb + g, M - 1);
    mc0[nb] = min(8 * nb + 2 * t, M - 1);
    mc1[nb] = min(8 * nb + 2 * t + 1, M - 1);
  }
  constexpr int WORD = S::WORD;
  float acc[NB][4];
  #pragma unroll
  for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;
  const int rounds = (nch + P - 1) / P;
  for (int r = 0; r < rounds; ++r) {
    #pragma unroll
    for (int i = 0; i < P; ++i) {
      const int c = r * P + i;
      if (c < nch) {                                                        // uniform over the CTA
        float ac[NB][4], d[NB][4];
        constexpr bool per_seg = is_mx4<F>() || is_fp4f<F>() || is_fs8<F>();  // a scale per segment
        constexpr bool per_pair = is_mx8<F>() || I4;  // a block per two segments
        #pragma unroll
        for (int sg = 0; sg < 4; ++sg) {
          // this segment starts a scale block: its first MMA takes a zero accumulator
          const bool fresh = per_seg || (per_pair && (sg & 1) == 0) || sg == 0;
          const int kx = c * CODES + sg * SEG + WORD * t;                   // this lane's first staged k
          if constexpr (FOUR) {
            uint32_t fa[4], fb[4];
            if constexpr (I4) {
              #pragma unroll
              for (int b = 0; b < 4; ++b) {
                fa[b] = ((i4_u<F>(wa[i][sg]) >> (4 * b)) & 0x000F000Fu) | 0x43004300u;   // bf16 128 + u
                fb[b] = ((i4_u<F>(wb[i][sg]) >> (4 * b)) & 0x000F000Fu) | 0x43004300u;
              }
            } else {
              if constexpr (F == MXINT4) {
                sint4x8_f16(wa[i][sg], fa);
                sint4x8_f16(wb[i][sg], fb);
              } else {
                e2m1x8_f16(wa[i][sg], fa);
                e2m1x8_f16(wb[i][sg], fb);
              }
              if constexpr (F == NVFP4) {                                   // E4M3 micro-scale, exact in f16
                uint32_t s2a, s2b;
                const uint32_t ba = (sc[i][0] >> (8 * sg)) & 0xFFu, bb = (sc[i][1] >> (8 * sg)) & 0xFFu;
                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2a) : "h"(uint16_t(ba | (ba << 8))));
                asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s2b) : "h"(uint16_t(bb | (bb << 8))));
                #pragma unroll
                for (int e = 0; e < 4; ++e) {
                  fa[e] = hmul2_f16(fa[e], s2a);
                  fb[e] = hmul2_f16(fb[e], s2b);
                }
              }
            }
            #pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const uint4 xv = *reinterpret_cast<const uint4*>(xs + mrow[nb] * xst + kx);
              if constexpr (I4) {   // bf16 activations as given, bf16 weights 128 + q (both exact)
                if (fresh) mma_bf16_z(d[nb], fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
                else mma_bf16(d[nb], fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
                mma_bf16(d[nb], fa[2], fb[2], fa[3], fb[3], xv.z, xv.w);
              } else {
                if (fresh) mma_f16_z(d[nb], fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
                else mma_f16(d[nb], fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
                mma_f16(d[nb], fa[2], fb[2], fa[3], fb[3], xv.z, xv.w);
              }
            }
          } else {
            uint32_t fa[2], fb[2];
            elem8x4_f16<F>(wa[i][sg], fa);
            elem8x4_f16<F>(wb[i][sg], fb);
            #pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              const uint2 xv = *reinterpret_cast<const uint2*>(xs + mrow[nb] * xst + kx);
              if (fresh) mma_f16_z(d[nb], fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
              else mma_f16(d[nb], fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
            }
          }
          // block scales on the float32 MMA results (d rows g: e = 0, 1; g + 8: e = 2, 3)
          constexpr bool per_seg = is_mx4<F>() || is_fp4f<F>() || is_fs8<F>();  // a scale per segment
          constexpr bool per_pair = is_mx8<F>() || I4;  // a block per two segments
          if (per_seg || (per_pair && (sg & 1))) {
            const bool first = sg < (per_seg ? 1 : 2);                      // the chunk's first block
            float sa, sb, ba = 0.0f, bb = 0.0f, xm0[NB], xm1[NB];
            if constexpr (is_mx4<F>()) {
              sa = e8m0_f32((sc[i][0] >> (8 * sg)) & 0xFFu);
              sb = e8m0_f32((sc[i][1] >> (8 * sg)) & 0xFFu);
            } else if constexpr (is_fs8<F>() || is_fp4f<F>()) {
              sa = __uint_as_float(sc[i][sg]);
              sb = __uint_as_float(sc[i][4 + sg]);
            } else if constexpr (I4) {                                      // s * D + (b - 128 s) * sum(x)
              const int h = sg >> 1;
              i4_scale_bias<F>(sc[i][h], sa, ba);
              i4_scale_bias<F>(sc[i][2 + h], sb, bb);
              ba = __fmaf_rn(-128.0f, sa, ba);
              bb = __fmaf_rn(-128.0f, sb, bb);
              const int blk = (c * CODES) / 64 + h;
              #pragma unroll
              for (int nb = 0; nb < NB; ++nb) {
                xm0[nb] = xsum[mc0[nb] * nsm + blk];
                xm1[nb] = xsum[mc1[nb] * nsm + blk];
              }
            } else {
              sa = e8m0_f32((sc[i][0] >> (8 * (sg >> 1))) & 0xFFu);
              sb = e8m0_f32((sc[i][1] >> (8 * (sg >> 1))) & 0xFFu);
            }
            #pragma unroll
            for (int nb = 0; nb < NB; ++nb) {
              if constexpr (I4) {
                ac[nb][0] = __fmaf_rn(sa, d[nb][0], first ? ba * xm0[nb] : __fmaf_rn(ba, xm0[nb], ac[nb][0]));
                ac[nb][1] = __fmaf_rn(sa, d[nb][1], first ? ba * xm1[nb] : __fmaf_rn(ba, xm1[nb], ac[nb][1]));
                ac[nb][2] = __fmaf_rn(sb, d[nb][2], first ? bb * xm0[nb] : __fmaf_rn(bb, xm0[nb], ac[nb][2]));
                ac[nb][3] = __fmaf_rn(sb, d[nb][3], first ? bb * xm1[nb] : __fmaf_rn(bb, xm1[nb], ac[nb][3]));
              } else {
                ac[nb][0] = first ? sa * d[nb][0] : __fmaf_rn(sa, d[nb][0], ac[nb][0]);
                ac[nb][1] = first ? sa * d[nb][1] : __fmaf_rn(sa, d[nb][1], ac[nb][1]);
                ac[nb][2] = first ? sb * d[nb][2] : __fmaf_rn(sb, d[nb][2], ac[nb][2]);
                ac[nb][3] = first ? sb * d[nb][3] : __fmaf_rn(sb, d[nb][3], ac[nb][3]);
              }
            }
          }
        }
        // the chunk's activation scale (one power of two per 128 values and row)
        const int span = (c * CODES) / XSPAN;
        #pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          if constexpr (I4) {                                               // activations unscaled
            acc[nb][0] += ac[nb][0];
            acc[nb][1] += ac[nb][1];
            acc[nb][2] += ac[nb][2];
            acc[nb][3] += ac[nb][3];
            continue;
          }
          const float x0 = xsc[mc0[nb] * nsp + span], x1 = xsc[mc1[nb] * nsp + span];
          if constexpr (F == NVFP4) {                                       // micro-scales already applied
            acc[nb][0] = __fmaf_rn(x0, d[nb][0], acc[nb][0]);
            acc[nb][1] = __fmaf_rn(x1, d[nb][1], acc[nb][1]);
            acc[nb][2] = __fmaf_rn(x0, d[nb][2], acc[nb][2]);
            acc[nb][3] = __fmaf_rn(x1, d[nb][3], acc[nb][3]);
          } else {
            acc[nb][0] = __fmaf_rn(x0, ac[nb][0], acc[nb][0]);
            acc[nb][1] = __fmaf_rn(x1, ac[nb][1], acc[nb][1]);
            acc[nb][2] = __fmaf_rn(x0, ac[nb][2], acc[nb][2]);
            acc[nb][3] = __fmaf_rn(x1, ac[nb][3], acc[nb][3]);
          }
        }
      }
      if (r + 1 < rounds) load_chunk((r + 1) * P + i, i);                  // slot i is free
    }
  }

  // ---- this CTA's partial tile, then the cluster's sum in rank order -------
  #pragma unroll
  for (int nb = 0; nb < NB; ++nb)
    #pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int rr = 16 * warp + g + (e >= 2 ? 8 : 0), col = 8 * nb + 2 * t + (e & 1);
      red[rr * 16 + col] = acc[nb][e];
    }
  cluster_sync();
  {
    uint32_t rank, csize;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
    const int rpr = ROWS / int(csize);                                      // rows reduced by this CTA
    constexpr bool X2 = F == MXFP4X2;                                       // output row = rows 2r + 2r + 1
    const uint32_t m_magic = 0xFFFFFFFFu / uint32_t(M) + 1u;                // i / M, exact for i < 2^16
    for (int i = tid; i < (X2 ? rpr / 2 : rpr) * M; i += THREADS) {
      const int iq = int(__umulhi(uint32_t(i), m_magic));
      const int rr = int(rank) * rpr + (X2 ? 2 * iq : iq), m = i - iq * M;
      if (row0 + rr >= N) continue;
      float sum = 0.0f;
      for (uint32_t q = 0; q < csize; ++q) {
        sum += ld_cluster_f32(red + rr * 16 + m, q);
        if constexpr (X2) sum += ld_cluster_f32(red + (rr + 1) * 16 + m, q);   // the residual plane
      }
      if constexpr (F == NVFP4) sum *= glob;
      const int64_t o = X2 ? int64_t(m) * (N / 2) + (row0 + rr) / 2 : int64_t(m) * N + row0 + rr;
      if (out_f32) static_cast<float*>(out)[o] = sum;
      else static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(sum);
    }
  }
  cluster_sync();   // no CTA leaves while the others still read its partial tile
}

// The K split: the smallest cluster size S in {1, 2, 4, 8} whose per-CTA K
// range (rounded up to 128) keeps the staged activations within X_BUDGET and
// gives at least four CTAs per SM (shorter K ranges per warp, fewer rounds).
inline bool plan(int F, int M, int N, int K, int sms, int* S, int* KR) {
  const int rb = fmt_is_four(F) ? 64 : 32;
  const int row_ctas = (N + ROWS - 1) / ROWS;
  for (int s = 1; s <= 8; s *= 2) {
    const int kr = ((K + s - 1) / s + XSPAN - 1) / XSPAN * XSPAN;
    const bool fits = size_t(M) * xstride(kr, rb) * 2 <= X_BUDGET;
    if (fits && (row_ctas * s >= 4 * sms || s == 8 || kr == XSPAN)) {
      *S = s;
      *KR = kr;
      return true;
    }
  }
  return false;
}

template <int F, int NB, bool UNI>
static cudaError_t launch_nb(const void* codes, const void* scales, float glob, const void* x, void* out,
                             bool out_f32, int M, int N, int K, int S, int KR, cudaStream_t st) {
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = 1;
  at[1].val.clusterDim.y = unsigned(S);
  at[1].val.clusterDim.z = 1;
  lc.gridDim = dim3((N + ROWS - 1) / ROWS, S);
  lc.blockDim = dim3(THREADS);
  lc.dynamicSmemBytes = smem_bytes(F, M, KR);
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, qgemv_mb_kernel<F, NB, UNI>, static_cast<const uint8_t*>(codes),
                            static_cast<const uint8_t*>(scales), glob, static_cast<const uint16_t*>(x), out,
                            int(out_f32), M, N, K, KR);
}

template <int F>
static cudaError_t launch_fmt(const void* codes, const void* scales, float glob, const void* x, void* out,
                              bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
  int S = 1, KR = 0;
  if (!plan(F, M, N, K, sms, &S, &KR)) return cudaErrorInvalidValue;
  const bool uni = S * KR == K && (KR / Shape<F>::CODES) % chunks_in_flight<F>() == 0;
  if (M <= 8)
    return uni ? launch_nb<F, 1, true>(codes, scales, glob, x, out, out_f32, M, N, K, S, KR, st)
               : launch_nb<F, 1, false>(codes, scales, glob, x, out, out_f32, M, N, K, S, KR, st);
  return uni ? launch_nb<F, 2, true>(codes, scales, glob, x, out, out_f32, M, N, K, S, KR, st)
             : launch_nb<F, 2, false>(codes, scales, glob, x, out, out_f32, M, N, K, S, KR, st);
}

}  // namespace gemv_mb

bool qgemv_mb_fits(int fmt, int64_t M, int64_t K) {
  int S = 0, KR = 0;
  return M >= 1 && M <= 16 && K <= (int64_t(1) << 24) && gemv_mb::plan(fmt, int(M), 1, int(K), 1, &S, &KR);
}

cudaError_t launch_qgemv_mb(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                            bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms) {
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return gemv_mb::launch_fmt<MXFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case NVFP4: return gemv_mb::launch_fmt<NVFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXFP8_E4M3: return gemv_mb::launch_fmt<MXFP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXFP8_E5M2: return gemv_mb::launch_fmt<MXFP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case NVFP8: return gemv_mb::launch_fmt<NVFP8>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case NVFP8_F16: return gemv_mb::launch_fmt<NVFP8_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXINT8: return gemv_mb::launch_fmt<MXINT8>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case INT8: return gemv_mb::launch_fmt<INT8>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case INT8_F16: return gemv_mb::launch_fmt<INT8_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case INT4: return gemv_mb::launch_fmt<INT4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case INT4_F16: return gemv_mb::launch_fmt<INT4_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXFP4X2: return gemv_mb::launch_fmt<MXFP4X2>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXINT4: return gemv_mb::launch_fmt<MXINT4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP4: return gemv_mb::launch_fmt<FP4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP4_F16: return gemv_mb::launch_fmt<FP4_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP8_E4M3: return gemv_mb::launch_fmt<FP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP8_E4M3_F16: return gemv_mb::launch_fmt<FP8_E4M3_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP8_E5M2: return gemv_mb::launch_fmt<FP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP8_E5M2_F16: return gemv_mb::launch_fmt<FP8_E5M2_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    default: return gemv_mb::launch_fmt<INT4_AFFINE>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
  }
}

}  // namespace qfmt_dev
