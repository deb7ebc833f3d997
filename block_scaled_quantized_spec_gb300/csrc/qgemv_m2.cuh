// Decode GEMV for one or two activation rows (M <= 2):
//   out[m, n] = sum_k x[m, k] * dequant(W)[n, k]
// (metaltile PR #250 qgemv commits: output[row] = sum_k dequant(weight[row,k])
// * input[k]; rlx-cpu thunk/ops/quant.rs dequant_matmul_nvfp4, whose m == 1
// loop streams the packed codes once and applies each block scale to that
// block's partial sum).
//
// At M = 1 a launch moves a few MB and its time is set by how soon the weight
// bytes are requested and how little work is left once the activations exist.
// So:
//  * every lane loads its weight spans straight into registers with 16-byte
//    loads at the top of the kernel (a CTA owns 16 weight rows; its 8 warps
//    take 64-byte column chunks of those rows in turn), together with the
//    block scales it will need, before waiting on the preceding kernel (the
//    launch is programmatic-dependent; the weights are not that kernel's
//    output).  Chunks past the first round are prefetched into L2;
//  * the activations are staged once per CTA in shared memory as f16 with a
//    power-of-two scale per 32 values (the span's largest |x| goes to
//    [2^14, 2^15): exact for every bf16 value within 2^29 of that maximum);
//  * a lane's 16-byte span (32 four-bit or 16 eight-bit codes) is converted to
//    f16 with the hardware conversions (E2M1/E4M3/E5M2 -> f16x2 are exact,
//    int4 becomes the exact f16 1024 + q) and is the lane's share of the A
//    operand of mma.sync m16n8k16.  The B operand is zero except in column t
//    (activation row 0) and t + 4 (row 1) of the lanes that supply quad lane
//    t's k positions, so D column t collects exactly quad lane t's span: one
//    scale block per column, scaled once per chunk in float32 (nvfp4 applies
//    its E4M3 micro-scales to the f16 weights instead: E2M1 x E4M3 is exact in
//    f16; its FP32 global scale is applied at the end);
//  * per-warp sums meet in shared memory; one thread per output stores it.
//
// The same kernel serves three more forms of the decode step (template MODE):
// expert-routed rows over a stacked weight (PR #250, MoE gather-qmm), up to
// four weight matrices sharing the activations (the batched Q/K/V and 4-way
// GEMVs) and an RMSNorm of the activations fused in front (the fused
// RMSNorm + GEMV); see the description beside `Extra` below.
//
// This header holds the kernel and its launchers; qgemv_m2_<group>.cu
// instantiate them for a group of formats each (compiled in parallel) and
// qgemv_m2.cu routes a format to its group.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {
namespace gemv_m2 {

constexpr int WARPS = 8;
constexpr int THREADS = WARPS * 32;
// chunks per warp held in registers at a time: four 64-byte chunks (the whole
// of a 4096-wide fp4 row share); the E8M0 8-bit formats hold eight
template <int F>
constexpr int chunks_in_flight() { return is_mx8<F>() ? 8 : 4; }
// with W warps per CTA: 4-warp CTAs hold twice the 4-bit chunks per warp
template <int F, int W>
constexpr int chunks_per_warp() { return (W == 4 && FmtTraits<F>::four) ? 2 * chunks_in_flight<F>() : chunks_in_flight<F>(); }
constexpr size_t SMEM_LIMIT = 96 * 1024;

template <int F>
struct Shape {
  static constexpr bool four = FmtTraits<F>::four;
  static constexpr int CODES = four ? 128 : 64;   // codes per row in one 64-byte chunk
  static constexpr int LANE = CODES / 4;           // codes in a lane's 16-byte span
};

__device__ __forceinline__ void mma_f16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8 E2M1 codes -> f16x2 (c0,c1) (c2,c3) (c4,c5) (c6,c7) (low code in the low half).
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

__device__ __forceinline__ uint32_t word(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}

// The four f16x2 fragments of activations 8q .. 8q+7 of a lane's span, in the
// order the staged activations use: E2M1 and 8-bit codes (8q, 8q+1) ..
// (8q+6, 8q+7); int4 the biased pairs (q_{8q+b}, q_{8q+b+4}), b = 0..3.
template <int F>
__device__ __forceinline__ void frags8(const uint4& v, int q, uint32_t r[4]) {
  if constexpr (F == MXFP4 || F == NVFP4 || is_fp4f<F>()) {
    e2m1x8_f16(word(v, q), r);
  } else if constexpr (is_i4<F>() || F == MXINT4) {
    const uint32_t w = i4_u<F>(word(v, q));
    #pragma unroll
    for (int b = 0; b < 4; ++b) r[b] = ((w >> (4 * b)) & 0x000F000Fu) | 0x64006400u;
  } else {
    elem8x4_f16<F>(word(v, 2 * q), r);
    elem8x4_f16<F>(word(v, 2 * q + 1), r + 2);
  }
}

// E8M0 byte j of w as float32 when 1 <= byte <= 254 (the biased exponent
// moved into place); bytes 0 and 255 take e8m0_f32.
template <int J>
__device__ __forceinline__ float e8m0_fast(uint32_t w) {
  return __uint_as_float(J == 3 ? (w >> 1) & 0x7F800000u : (w << (23 - 8 * J)) & 0x7F800000u);
}

__device__ __forceinline__ bool has_byte_00_or_ff(uint32_t w) {
  const uint32_t z = (w - 0x01010101u) & ~w & 0x80808080u;
  const uint32_t f = (~w - 0x01010101u) & w & 0x80808080u;
  return (z | f) != 0u;
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint4 ldg_stream(const uint8_t* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Halfword offset of activation k in a staged row: 8 halfwords of padding
// after every 32 values keep the B-operand reads of a warp in distinct banks.
__host__ __device__ constexpr int xoff(int k) { return k + (k >> 5) * 8; }

// Staged activation row stride in halfwords: the padded row rounded so that
// consecutive rows start 64 bytes apart modulo 128 (rows 0 and 1 then use
// disjoint banks).
__host__ __device__ constexpr int xstride(int K) {
  const int h = xoff(K);
  const int bytes = 2 * h;
  const int pad = ((64 - bytes % 128) + 128) % 128;
  return h + pad / 2;
}

inline size_t smem_bytes(int F, int M, int K, int warps = WARPS) {
  const int spans = K / 32;
  return size_t(M) * xstride(K) * 2 + 64 + size_t(M) * spans * 4 * ((fmt_is_i4(F) || F == MXINT4) ? 2 : 1) +
         size_t(warps) * 2 * 16 * 4 + size_t(warps) * 2 * 4;
}

// STAGE: row strides of the weight and scale copies in shared memory (a
// 64-byte offset between rows puts rows g and g + 1 in different halves of
// the banks; 16 bytes between scale rows spread rows 0-7 over the banks).
__host__ __device__ constexpr int64_t stage_wstride(int64_t rowbytes) { return rowbytes + 64; }
__host__ __device__ constexpr int64_t stage_sstride(int64_t srowbytes) { return (srowbytes + 15) / 16 * 16 + 16; }
constexpr int STAGE_WARPS = 16;                                              // two groups of 8, one per tile
inline size_t stage_offset(int F, int M, int K) { return (smem_bytes(F, M, K, STAGE_WARPS) + 127) / 128 * 128; }
constexpr int STAGE_ROWS = 32;                                              // two 16-row tiles
constexpr size_t STAGE_SMEM_LIMIT = 112 * 1024;                             // two CTAs an SM
inline size_t stage_smem_bytes(int F, int M, int K, int64_t rowbytes, int64_t srowbytes) {
  return stage_offset(F, M, K) + STAGE_ROWS * size_t(stage_wstride(rowbytes)) +
         STAGE_ROWS * size_t(stage_sstride(srowbytes)) + 16;
}

// Bounded wait for the phase of the given parity of a shared-memory mbarrier.
__device__ __forceinline__ bool mbar_wait_parity(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  auto done = [&]() {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
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

// Per-chunk scale words a D-holding lane keeps: the weight block scales of
// the two columns it holds, for rows g and g + 8 (raw encodings).
struct ChunkScales {
  uint32_t a0, a1, b0, b1;
};

// Rows whose expert index lies outside [0, E) in an expert-routed launch (one
// word per translation unit that instantiates the kernel; read through
// Group<...>::read_status).
static __device__ unsigned int g_gather_status;

// Launch forms beyond the plain product (bits of MODE):
//  * GATHER, the expert-routed form (one activation row per blockIdx.y, M =
//    1): the row's weights are rows [e N, e N + N) of the stacked matrix, e =
//    eidx[blockIdx.y], read once the preceding kernel has completed (it may be
//    the router that wrote them), so the weight requests wait for it too;
//  * BATCH: up to four weight matrices share the activations (the Q/K/V and
//    4-way projections); the CTAs of matrix i are [tile0[i], tile0[i + 1]);
//  * GATE (with RMS): the gated RMSNorm: x * gamma * silu(gate) is staged
//    (silu(z) = z / (1 + e^-z), gate a bf16 [M, K] tensor read with X); the
//    root mean square stays that of x;
//  * RMS: the activations are RMS-normalised on the way in: x * gamma is
//    staged, sum(x^2) is gathered over the CTA (whose warps cover all of K),
//    and 1 / sqrt(mean(x^2) + eps) multiplies each output.
//  * STAGE: one 16-warp CTA per SM takes two 16-row tiles (tile b and
//    b + grid), one per group of 8 warps; the 32 weight rows and their scale
//    rows are bulk-copied into shared memory as the kernel starts (L2
//    evict-first: read once) and the lanes read their spans from there.  Two
//    such CTAs fit on an SM, so every CTA of the next launch of a decode
//    chain starts, and requests its weights, while this launch still runs --
//    exactly one beside each of this launch's, which keeps the launch's work
//    even over the SMs (with two 16-row CTAs an SM most of the next launch
//    starts only as this launch's CTAs leave; with smaller CTAs the scheduler
//    stacks up to four of one launch on an SM).  Group 0 stages the
//    activations for both.  A copy that does not land within the wait limit
//    sets bit 1 of the status word and the CTA stores nothing.
constexpr int GATHER = 1, BATCH = 2, RMS = 4, GATE = 8, STAGE = 16;
struct Extra {
  const int32_t* eidx;          // GATHER
  int E;
  int count;                    // BATCH
  const uint8_t* codes[4];
  const uint8_t* scales[4];
  float glob[4];
  void* out[4];
  int n[4];
  int tile0[5];
  const uint16_t* gamma;        // RMS: bf16 [K]
  const uint16_t* gate;         // GATE: bf16 [M, K]
  float eps;
  uint64_t limit_ns;            // STAGE: the copies' wait limit
  int drop;                     // STAGE fault hook: the copies are not issued, so the wait expires
};

template <int F, int MR, bool UNI, int W, int MODE = 0>
__global__ void __launch_bounds__(32 * W, W == 4 ? 3 : 2) qgemv_m2_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales, float glob,
                                                           const uint16_t* __restrict__ x, void* __restrict__ out,
                                                           int out_f32, int M, int N, int K, const Extra ex) {
  (void)glob;   // nvfp4's global scale; the other formats have none
  using S = Shape<F>;
  constexpr bool STG = (MODE & STAGE) != 0;
  constexpr int P = STG ? 2 : chunks_per_warp<F, W>();
  constexpr int WARPS = W;
  constexpr int GROUPS = STG ? 2 : 1;                                       // STAGE: a warp group per tile
  constexpr int WK = W / GROUPS;                                            // warps sharing a tile's K range
  constexpr bool FOUR = S::four, I4 = is_i4<F>() || F == MXINT4;   // int4 pairing, span sums of x
  constexpr bool X2 = F == MXFP4X2;                                         // output row = rows 2r + 2r + 1
  constexpr int CODES = S::CODES, LANE = S::LANE;
  extern __shared__ __align__(16) uint8_t smem[];
  const int xst = xstride(K);
  const int spans = K / 32;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem);                         // [M][xst] f16
  uint16_t* xzero = xs + size_t(M) * xst;                                   // 32 zero halfwords
  float* xsc = reinterpret_cast<float*>(xzero + 32);                        // [M][spans] 2^-shift
  float* xsum = xsc + M * spans;                                            // [M][spans] (int4 affine)
  float* red = xsum + (I4 ? M * spans : 0);                                 // [WARPS][2][16]
  float* rss = red + WARPS * 2 * 16;                                        // [WARPS][2] (RMS)

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kw = warp % WK, jt = warp / WK;                                 // K-range warp, tile group
  const int g = lane >> 2, t = lane & 3;
  int row0 = blockIdx.x * 16;
  // STAGE: the weight and scale rows of this CTA in shared memory
  const int64_t stage_rowb = FmtTraits<F>::four ? K / 2 : K;
  const int64_t stage_srowb = int64_t((K + FmtTraits<F>::block - 1) / FmtTraits<F>::block) * FmtTraits<F>::sbytes;
  uint8_t* wsm = smem + ((reinterpret_cast<uintptr_t>(rss + WARPS * 2) - reinterpret_cast<uintptr_t>(smem) + 127) & ~uintptr_t(127));
  uint8_t* ssm = wsm + STAGE_ROWS * stage_wstride(stage_rowb);
  uint64_t* wbar = reinterpret_cast<uint64_t*>(ssm + STAGE_ROWS * stage_sstride(stage_srowb));
  const int tile1 = int(blockIdx.x) + int(gridDim.x);                       // STAGE: the second tile
  const int stage_tiles = STG && tile1 < (N + 15) / 16 ? 2 : 1;
  if constexpr (STG) {
    if (warp == 0) {
      const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(wbar));
      const int nr0 = min(16, N - row0), nr1 = stage_tiles > 1 ? min(16, N - 16 * tile1) : 0;
      if (lane == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"(uint32_t(nr0 + nr1) * uint32_t(stage_rowb + stage_srowb))
                     : "memory");
      }
      __syncwarp();
      uint64_t pol;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
      const int r = lane & 15;
      const bool sc = lane >= 16;
      #pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int base = j == 0 ? row0 : 16 * tile1;
        if (r < (j == 0 ? nr0 : nr1) && !ex.drop) {
          const uint8_t* src = sc ? scales + int64_t(base + r) * stage_srowb : codes + int64_t(base + r) * stage_rowb;
          uint8_t* dst = sc ? ssm + (16 * j + r) * stage_sstride(stage_srowb) : wsm + (16 * j + r) * stage_wstride(stage_rowb);
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
              ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))), "l"(src),
              "r"(uint32_t(sc ? stage_srowb : stage_rowb)), "r"(bar), "l"(pol)
              : "memory");
        }
      }
    }
  }
  if constexpr ((MODE & BATCH) != 0) {    // this CTA's matrix: unrolled selects, no indexed parameters
    int i = 0;
    #pragma unroll
    for (int j = 1; j < 4; ++j) i += (j < ex.count && int(blockIdx.x) >= ex.tile0[j]) ? 1 : 0;
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (j == i) {
        codes = ex.codes[j];
        scales = ex.scales[j];
        glob = ex.glob[j];
        out = ex.out[j];
        N = ex.n[j];
        row0 = (int(blockIdx.x) - ex.tile0[j]) * 16;
      }
    }
  }
  if constexpr ((MODE & GATHER) != 0) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t m = blockIdx.y;
    const int e = __ldg(ex.eidx + m);
    x += m * K;
    out = static_cast<uint8_t*>(out) + m * (X2 ? N / 2 : N) * (out_f32 ? 4 : 2);
    if (e < 0 || e >= ex.E) {                                               // a zero row, and the status bit
      constexpr int OR = X2 ? 8 : 16;                                       // output rows of the tile
      const int o0 = X2 ? row0 / 2 : row0;
      if (tid < OR && o0 + tid < (X2 ? N / 2 : N)) {
        if (out_f32) static_cast<float*>(out)[o0 + tid] = 0.0f;
        else static_cast<__nv_bfloat16*>(out)[o0 + tid] = __float2bfloat16_rn(0.0f);
      }
      if (tid == 0) atomicOr(&g_gather_status, 1u);
      return;
    }
    codes += int64_t(e) * N * (FmtTraits<F>::four ? K / 2 : K);
    scales += int64_t(e) * N * ((K + FmtTraits<F>::block - 1) / FmtTraits<F>::block) * FmtTraits<F>::sbytes;
  }
  int ra = row0 + g, rb = row0 + g + 8;
  bool va = ra < N, vb = rb < N;
  const int64_t rowbytes = FOUR ? K / 2 : K;
  const uint8_t* pa = STG ? wsm + g * stage_wstride(rowbytes) + 16 * t : codes + int64_t(va ? ra : 0) * rowbytes + 16 * t;
  const uint8_t* pb =
      STG ? wsm + (g + 8) * stage_wstride(rowbytes) + 16 * t : codes + int64_t(vb ? rb : 0) * rowbytes + 16 * t;
  const int nchunk = (K + CODES - 1) / CODES;
  const int mine = nchunk > kw ? (nchunk - kw + WK - 1) / WK : 0;            // chunks of this warp
  const int a0 = (2 * t) & 3;                                                 // first column's quad lane
  const int64_t nblk = (K + FmtTraits<F>::block - 1) / FmtTraits<F>::block;   // int4 affine: a ragged last group

  uint4 wa[P], wb[P];
  ChunkScales cs[P];
  uint32_t ms[P];      // nvfp4: this lane's two E4M3 micro-scales, row g (low half) and row g + 8

  // Rows past N read row 0 (their outputs are never stored).  UNI: every
  // warp's chunks are whole and in range (K a multiple of 8 chunks, the chunk
  // count per warp a multiple of P), so the loads carry no predicates and
  // paired E8M0 bytes come in one 16-bit load.
  constexpr bool uni = UNI;
  constexpr int SB = FmtTraits<F>::sbytes;
  const uint8_t* sra = STG ? ssm + g * stage_sstride(nblk * SB) : scales + int64_t(va ? ra : 0) * nblk * SB;   // row g's
  const uint8_t* srb = STG ? ssm + (g + 8) * stage_sstride(nblk * SB) : scales + int64_t(vb ? rb : 0) * nblk * SB;
  constexpr bool GL = !STG;                                                 // scale reads: global (else shared)

  // chunk slot i of round r: codes of rows g and g + 8 and their scales
  auto load_chunk = [&](int r, int i) {
    const int c = kw + WK * (r * P + i);
    const int ks = c * CODES + LANE * t;                                     // this lane's first k
    const int k0 = c * CODES + LANE * a0;                                    // quad lane a0's first k
    const bool live = uni || r * P + i < mine;
    const bool kin = uni || (live && ks < K);
    const bool c0 = uni || (live && k0 < K), c1 = uni || (live && k0 + LANE < K);
    if constexpr (STG) {
      wa[i] = kin ? *reinterpret_cast<const uint4*>(pa + c * 64) : make_uint4(0, 0, 0, 0);
      wb[i] = kin ? *reinterpret_cast<const uint4*>(pb + c * 64) : make_uint4(0, 0, 0, 0);
    } else {
      wa[i] = kin ? ldg_stream(pa + int64_t(c) * 64) : make_uint4(0, 0, 0, 0);
      wb[i] = kin ? ldg_stream(pb + int64_t(c) * 64) : make_uint4(0, 0, 0, 0);
    }
    // the block (or pair of blocks) of quad lanes a0 and a0 + 1 in this chunk;
    // a block outside the matrix reads as E8M0 127 / zero (its D column is zero)
    if constexpr (is_mx4<F>()) {
      const int e = k0 / 32;                                                  // even
      if (uni) {
        const uint32_t pa2 = ld_ro<GL>(reinterpret_cast<const uint16_t*>(sra) + e / 2);
        const uint32_t pb2 = ld_ro<GL>(reinterpret_cast<const uint16_t*>(srb) + e / 2);
        cs[i].a0 = prmt(pa2, pb2, 0x5410u);                                   // four E8M0 bytes
      } else {
        const uint32_t x0 = c0 ? ld_ro<GL>(sra + e) : 127u;
        const uint32_t x1 = c1 ? ld_ro<GL>(sra + e + 1) : 127u;
        const uint32_t x2 = c0 ? ld_ro<GL>(srb + e) : 127u;
        const uint32_t x3 = c1 ? ld_ro<GL>(srb + e + 1) : 127u;
        cs[i].a0 = x0 | (x1 << 8) | (x2 << 16) | (x3 << 24);
      }
      cs[i].a1 = cs[i].b0 = cs[i].b1 = 0u;
    } else if constexpr (is_mx8<F>()) {
      const int e = k0 / 32;                                                  // a0, a0 + 1 share it
      const uint32_t x0 = c0 ? ld_ro<GL>(sra + e) : 127u;
      const uint32_t x2 = c0 ? ld_ro<GL>(srb + e) : 127u;
      cs[i].a0 = prmt(x0, x2, 0x1410u) | 0x7F007F00u;                         // bytes 0 and 2 used, 1 and 3 = 127
      cs[i].a1 = cs[i].b0 = cs[i].b1 = 0u;
    } else if constexpr (is_fs8<F>() || is_fp4f<F>()) {
      constexpr int B = FmtTraits<F>::block;                                  // 16 (nvfp8), 32 (mxfp4x2), 64 (int8)
      const int e = k0 / B;
      cs[i].a0 = c0 ? __float_as_uint(float_scale<F, GL>(sra, e)) : 0u;
      cs[i].b0 = c0 ? __float_as_uint(float_scale<F, GL>(srb, e)) : 0u;
      if constexpr (B <= LANE) {                                              // quad lane a0 + 1: the next block
        cs[i].a1 = c1 ? __float_as_uint(float_scale<F, GL>(sra, e + 1)) : 0u;
        cs[i].b1 = c1 ? __float_as_uint(float_scale<F, GL>(srb, e + 1)) : 0u;
      } else {                                                                // a0, a0 + 1 share it
        cs[i].a1 = c1 ? cs[i].a0 : 0u;
        cs[i].b1 = c1 ? cs[i].b0 : 0u;
      }
    } else if constexpr (is_i4<F>()) {
      const int e = k0 / 64;                                                  // a0, a0 + 1 share it
      cs[i].a0 = c0 ? i4_word<F, GL>(sra, e) : 0u;
      cs[i].b0 = c0 ? i4_word<F, GL>(srb, e) : 0u;
      cs[i].a1 = cs[i].b1 = 0u;
    } else {   // NVFP4: the lane's own two micro-blocks, one 16-bit pair per row
      const int e = ks / 32;                                                  // pair index (16-code blocks / 2)
      const uint32_t ma = kin ? ld_ro<GL>(reinterpret_cast<const uint16_t*>(sra) + e) : 0u;
      const uint32_t mb2 = kin ? ld_ro<GL>(reinterpret_cast<const uint16_t*>(srb) + e) : 0u;
      ms[i] = prmt(ma, mb2, 0x5410u);
      cs[i].a0 = cs[i].a1 = cs[i].b0 = cs[i].b1 = 0u;
    }
  };
  auto load_round = [&](int r) {
    #pragma unroll
    for (int i = 0; i < P; ++i) load_chunk(r, i);
  };

  const int rounds = (mine + P - 1) / P;
  if constexpr (!STG) load_round(0);
  // chunks past the first round: start them towards L2 now
  if (!STG && rounds > 1 && tid < 16 && row0 + tid < N) {
    const int64_t first = int64_t(WARPS) * P * 64;
    if (rowbytes > first) {
      const uint8_t* p = codes + int64_t(row0 + tid) * rowbytes + first;
      const uint32_t n = uint32_t(rowbytes - first);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(n) : "memory");
    }
  }

  // Any E8M0 scale byte of this round equal to 0 or 255 sends the warp down the exact decode.
  bool exact = false;
  if constexpr (is_e8m0<F>() && !STG) {
    bool sp = false;
    #pragma unroll
    for (int i = 0; i < P; ++i) sp |= has_byte_00_or_ff(cs[i].a0);
    exact = __any_sync(0xFFFFFFFFu, sp);
  }
  if (tid < 16) reinterpret_cast<uint32_t*>(xzero)[tid] = 0u;
  __syncthreads();

  // The activations may be the preceding kernel's output.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- stage this warp's activations: the k ranges of its own chunks --------
  // 16 values per task, tasks 2s and 2s+1 (lanes l and l^1) share a 32-span;
  // the span's shift puts its largest |x| in [2^14, 2^15).
  float ssq[2] = {0.0f, 0.0f};                                               // RMS: this lane's sum of x^2 per row
  if (jt == 0) {
    constexpr int TPC = CODES / 16;                                            // tasks per chunk and row
    const int per_m = mine * TPC;
    const int tasks = M * per_m;
    // TIF tasks per lane and pass are in flight together (a round's worth)
    constexpr int TIF = (MR * P * TPC + 31) / 32;
    for (int j0 = 0; j0 < tasks; j0 += 32 * TIF) {
      uint4 v[TIF][2];
      uint4 zv[(MODE & GATE) != 0 ? TIF : 1][2];                            // GATE: the gate's 16 values
      int kk[TIF], mm[TIF];
      bool lv[TIF];
      #pragma unroll
      for (int u = 0; u < TIF; ++u) {
        const int j = j0 + lane + 32 * u;
        const int m = j >= per_m ? 1 : 0;
        const int rem = j - m * per_m;
        const int c = kw + WK * (rem / TPC);
        const int k = c * CODES + (rem % TPC) * 16;
        lv[u] = j < tasks && k < K;
        kk[u] = k;
        mm[u] = m;
        const uint4* src = reinterpret_cast<const uint4*>(x + int64_t(m) * K + k);
        v[u][0] = lv[u] ? __ldg(src) : make_uint4(0, 0, 0, 0);
        v[u][1] = lv[u] ? __ldg(src + 1) : make_uint4(0, 0, 0, 0);
        if constexpr ((MODE & GATE) != 0) {   // requested with the activations
          const uint4* zp = reinterpret_cast<const uint4*>(ex.gate + int64_t(m) * K + k);
          zv[u][0] = lv[u] ? __ldg(zp) : make_uint4(0, 0, 0, 0);
          zv[u][1] = lv[u] ? __ldg(zp + 1) : make_uint4(0, 0, 0, 0);
        }
      }
      #pragma unroll
      for (int u = 0; u < TIF; ++u) {
        if (j0 + 32 * u >= tasks) break;                                       // uniform over the warp
        const bool live = lv[u];
        const int m = mm[u], k = kk[u];
        const uint32_t h[8] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w};
        float f[16];
        int sh;
        if constexpr ((MODE & RMS) != 0) {
          // x * gamma (exact in float32), its span maximum, and this row's sum of x^2
          const uint4* gp = reinterpret_cast<const uint4*>(ex.gamma + k);
          const uint4 g0 = live ? __ldg(gp) : make_uint4(0, 0, 0, 0), g1 = live ? __ldg(gp + 1) : make_uint4(0, 0, 0, 0);
          const uint32_t gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          uint32_t mx = 0;
          float sq = 0.0f;
          #pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float x0 = __uint_as_float(h[q] << 16), x1 = __uint_as_float(h[q] & 0xFFFF0000u);
            f[2 * q] = __fmul_rn(x0, __uint_as_float(gw[q] << 16));
            f[2 * q + 1] = __fmul_rn(x1, __uint_as_float(gw[q] & 0xFFFF0000u));
            if constexpr ((MODE & GATE) != 0) {
              const uint32_t zw = q < 4 ? word(zv[u][0], q) : word(zv[u][1], q - 4);
              const float za = __uint_as_float(zw << 16), zb = __uint_as_float(zw & 0xFFFF0000u);
              // silu(z) = z / (1 + e^-z): CUDA's fast exponential and the IEEE reciprocal
              // (e^-z = inf for z far below zero gives a reciprocal of 0, silu -0)
              f[2 * q] = __fmul_rn(f[2 * q], __fmul_rn(za, __frcp_rn(__fadd_rn(1.0f, __expf(-za)))));
              f[2 * q + 1] = __fmul_rn(f[2 * q + 1], __fmul_rn(zb, __frcp_rn(__fadd_rn(1.0f, __expf(-zb)))));
            }
            sq = __fmaf_rn(x0, x0, sq);
            sq = __fmaf_rn(x1, x1, sq);
            mx = max(mx, __float_as_uint(f[2 * q]) & 0x7FFFFFFFu);
            mx = max(mx, __float_as_uint(f[2 * q + 1]) & 0x7FFFFFFFu);
          }
          if (m == 0) ssq[0] += sq;
          else ssq[1] += sq;
          mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));                   // the other half of the span
          const int E = int(mx >> 23);
          sh = (mx == 0u || E == 255) ? 0 : 141 - E;                           // 14 - (E - 127)
          sh = sh > 126 ? 126 : (sh < -126 ? -126 : sh);
        } else {
          uint32_t m2 = 0;
          #pragma unroll
          for (int q = 0; q < 8; ++q) m2 = max_u16x2(m2, h[q] & 0x7FFF7FFFu);
          uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
          mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));                   // the other half of the span
          const int E = int(mx >> 7);
          sh = (mx == 0u || E == 255) ? 0 : 141 - E;                           // 14 - (E - 127)
          sh = sh > 126 ? 126 : sh;
          #pragma unroll
          for (int q = 0; q < 8; ++q) {
            f[2 * q] = __uint_as_float(h[q] << 16);
            f[2 * q + 1] = __uint_as_float(h[q] & 0xFFFF0000u);
          }
        }
        const float up = __uint_as_float(uint32_t(sh + 127) << 23);
        #pragma unroll
        for (int q = 0; q < 16; ++q) f[q] = __fmul_rn(f[q], up);
        uint32_t o[8];
        if constexpr (I4) {   // per 8 values: (x0,x4) (x1,x5) (x2,x6) (x3,x7), the int4 pairing
          #pragma unroll
          for (int q = 0; q < 4; ++q) {
            o[q] = pack_f16x2(f[q], f[q + 4]);
            o[4 + q] = pack_f16x2(f[8 + q], f[12 + q]);
          }
        } else {
          #pragma unroll
          for (int q = 0; q < 8; ++q) o[q] = pack_f16x2(f[2 * q], f[2 * q + 1]);
        }
        if (live) {
          uint4* dst = reinterpret_cast<uint4*>(xs + size_t(m) * xst + xoff(k));
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
        if constexpr (I4) {   // span sum of the staged (rounded) values
          float sm = 0.0f;
          #pragma unroll
          for (int q = 0; q < 8; ++q) sm += f16x2_lo(o[q]) + f16x2_hi(o[q]);
          sm += __shfl_xor_sync(0xFFFFFFFFu, sm, 1);
          if (live && (k & 16) == 0) xsum[m * spans + k / 32] = sm;
        }
        if (live && (k & 16) == 0) xsc[m * spans + k / 32] = __uint_as_float(uint32_t(127 - sh) << 23);
      }
    }
  }
  __syncwarp();

  if constexpr (STG) {   // the weight copies requested at the start (bounded wait; the CTA agrees)
    const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(wbar));
    if (!__syncthreads_and(mbar_wait_parity(bar, 0, ex.limit_ns))) {
      if (tid == 0) {   // nothing stored; the copies land before the CTA leaves
        atomicOr(&g_gather_status, 2u);
        mbar_wait_parity(bar, 0, ex.limit_ns);
      }
      return;
    }
  }

  // B-operand lanes: (g == t) supplies activation row 0, (g == t + 4) row 1.
  const int mb = g == t ? 0 : (g == t + 4 ? 1 : -1);
  const bool bl = mb >= 0 && mb < M;
  const int md = (t >> 1) < M ? (t >> 1) : M - 1;   // the activation row of this lane's D columns

  const bool tile_live = jt < stage_tiles;
  if (tile_live) {
  if constexpr (STG) {   // tile jt's rows in shared memory
    row0 = jt == 0 ? int(blockIdx.x) * 16 : 16 * tile1;
    ra = row0 + g;
    rb = ra + 8;
    va = ra < N;
    vb = rb < N;
    pa = wsm + (16 * jt + g) * stage_wstride(rowbytes) + 16 * t;
    pb = pa + 8 * stage_wstride(rowbytes);
    sra = ssm + (16 * jt + g) * stage_sstride(nblk * SB);
    srb = sra + 8 * stage_sstride(nblk * SB);
    load_round(0);
    if constexpr (is_e8m0<F>()) {
      bool sp = false;
      #pragma unroll
      for (int i = 0; i < P; ++i) sp |= has_byte_00_or_ff(cs[i].a0);
      exact = __any_sync(0xFFFFFFFFu, sp);
    }
  }

  float acc_a = 0.0f, acc_b = 0.0f;
  for (int r = 0; r < rounds; ++r) {
    if (r > 0) {   // this round's chunks were requested while the previous round computed
      if constexpr (is_e8m0<F>()) {
        bool sp = false;
        #pragma unroll
        for (int i = 0; i < P; ++i) sp |= has_byte_00_or_ff(cs[i].a0);
        exact = __any_sync(0xFFFFFFFFu, sp);
      }
    }
    // Chunks advance in pairs (two independent accumulator chains per warp);
    // a chunk past the end of this warp's share has zero codes, zero
    // activations and zero scales and adds nothing.
    #pragma unroll
    for (int ip = 0; ip < P; ip += 2) {
    int xo[2];
    float d[2][4];
    uint32_t sa0[2], sa1[2], sb0[2], sb1[2];
    #pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
      const int i = ip + ii;
      const int c = kw + WK * (r * P + i);
      const int ks = c * CODES + LANE * t;
      xo[ii] = (bl && r * P + i < mine && ks < K) ? mb * xst + xoff(ks) : M * xst;   // M * xst: the zero block
      d[ii][0] = d[ii][1] = d[ii][2] = d[ii][3] = 0.0f;
      if constexpr (F == NVFP4) {
        // E4M3 pair -> f16x2 (s0, s1), then splat each
        uint32_t pa2, pb2;
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(pa2) : "h"(uint16_t(ms[i] & 0xFFFFu)));
        asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(pb2) : "h"(uint16_t(ms[i] >> 16)));
        sa0[ii] = prmt(pa2, 0u, 0x1010u);
        sa1[ii] = prmt(pa2, 0u, 0x3232u);
        sb0[ii] = prmt(pb2, 0u, 0x1010u);
        sb1[ii] = prmt(pb2, 0u, 0x3232u);
      }
    }
    #pragma unroll
    for (int q = 0; q < LANE / 8; ++q) {                                       // 8 activations, two MMAs
      #pragma unroll
      for (int ii = 0; ii < 2; ++ii) {
        const int i = ip + ii;
        const uint4 xv = *reinterpret_cast<const uint4*>(xs + xo[ii] + 8 * q);
        uint32_t fa[4], fb[4];
        frags8<F>(wa[i], q, fa);
        frags8<F>(wb[i], q, fb);
        if constexpr (F == NVFP4) {                                            // codes 0-15 / 16-31 of the span
          const uint32_t ca = q < 2 ? sa0[ii] : sa1[ii], cb = q < 2 ? sb0[ii] : sb1[ii];
          #pragma unroll
          for (int e = 0; e < 4; ++e) {
            fa[e] = hmul2_f16(fa[e], ca);
            fb[e] = hmul2_f16(fb[e], cb);
          }
        }
        mma_f16(d[ii], fa[0], fb[0], fa[1], fb[1], xv.x, xv.y);
        mma_f16(d[ii], fa[2], fb[2], fa[3], fb[3], xv.z, xv.w);
      }
    }
    #pragma unroll
    for (int ii = 0; ii < 2; ++ii) {
      const int i = ip + ii;
      // D columns 2t, 2t+1 hold quad lanes a0, a0 + 1 of activation row md
      const int c = kw + WK * (r * P + i);
      const int k0 = c * CODES + LANE * a0;
      const int s0 = min(k0 / 32, spans - 1), s1 = min((k0 + LANE) / 32, spans - 1);
      const float x0s = xsc[md * spans + s0], x1s = xsc[md * spans + s1];
      if constexpr (is_mx4<F>()) {
        const uint32_t w4 = cs[i].a0;
        float q0, q1, q2, q3;
        if (exact) {
          q0 = e8m0_f32(w4 & 0xFFu); q1 = e8m0_f32((w4 >> 8) & 0xFFu);
          q2 = e8m0_f32((w4 >> 16) & 0xFFu); q3 = e8m0_f32(w4 >> 24);
        } else {
          q0 = e8m0_fast<0>(w4); q1 = e8m0_fast<1>(w4); q2 = e8m0_fast<2>(w4); q3 = e8m0_fast<3>(w4);
        }
        if constexpr (F == MXINT4) {
          // D = sum_k x~ (1024 + u) with u = q + 8: the span's sum is D - 1032 sum(x~);
          // a span past K (a chunk slot past the warp's share, or the second span
          // of the last chunk) has zero activations, so D = 0, and no sum either
          const float m0 = k0 < K ? xsum[md * spans + s0] : 0.0f;
          const float m1 = k0 + LANE < K ? xsum[md * spans + s1] : 0.0f;
          d[ii][0] = __fmaf_rn(-1032.0f, m0, d[ii][0]);
          d[ii][1] = __fmaf_rn(-1032.0f, m1, d[ii][1]);
          d[ii][2] = __fmaf_rn(-1032.0f, m0, d[ii][2]);
          d[ii][3] = __fmaf_rn(-1032.0f, m1, d[ii][3]);
        }
        acc_a = __fmaf_rn(__fmul_rn(q0, x0s), d[ii][0], acc_a);
        acc_a = __fmaf_rn(__fmul_rn(q1, x1s), d[ii][1], acc_a);
        acc_b = __fmaf_rn(__fmul_rn(q2, x0s), d[ii][2], acc_b);
        acc_b = __fmaf_rn(__fmul_rn(q3, x1s), d[ii][3], acc_b);
      } else if constexpr (is_mx8<F>()) {
        const uint32_t w4 = cs[i].a0;
        const float qa = exact ? e8m0_f32(w4 & 0xFFu) : e8m0_fast<0>(w4);
        const float qb = exact ? e8m0_f32((w4 >> 16) & 0xFFu) : e8m0_fast<2>(w4);
        const float ca = __fmul_rn(qa, x0s), cb = __fmul_rn(qb, x0s);
        acc_a = __fmaf_rn(ca, d[ii][0] + d[ii][1], acc_a);
        acc_b = __fmaf_rn(cb, d[ii][2] + d[ii][3], acc_b);
      } else if constexpr (is_fs8<F>() || is_fp4f<F>()) {
        acc_a = __fmaf_rn(__fmul_rn(__uint_as_float(cs[i].a0), x0s), d[ii][0], acc_a);
        acc_a = __fmaf_rn(__fmul_rn(__uint_as_float(cs[i].a1), x1s), d[ii][1], acc_a);
        acc_b = __fmaf_rn(__fmul_rn(__uint_as_float(cs[i].b0), x0s), d[ii][2], acc_b);
        acc_b = __fmaf_rn(__fmul_rn(__uint_as_float(cs[i].b1), x1s), d[ii][3], acc_b);
      } else if constexpr (is_i4<F>()) {
        // sum_k x~ (1024 + u): s * D + (b - 1024 s) * sum(x~), then the span's 2^-shift
        // a second span past K (a ragged last group of 32) adds no bias term
        const float m0 = xsum[md * spans + s0], m1 = k0 + LANE < K ? xsum[md * spans + s1] : 0.0f;
        float sa, ba, sb, bb;
        i4_scale_bias<F>(cs[i].a0, sa, ba);
        i4_scale_bias<F>(cs[i].b0, sb, bb);
        ba = __fmaf_rn(-1024.0f, sa, ba);
        bb = __fmaf_rn(-1024.0f, sb, bb);
        acc_a = __fmaf_rn(x0s, __fmaf_rn(sa, d[ii][0], ba * m0), acc_a);
        acc_a = __fmaf_rn(x1s, __fmaf_rn(sa, d[ii][1], ba * m1), acc_a);
        acc_b = __fmaf_rn(x0s, __fmaf_rn(sb, d[ii][2], bb * m0), acc_b);
        acc_b = __fmaf_rn(x1s, __fmaf_rn(sb, d[ii][3], bb * m1), acc_b);
      } else {   // NVFP4: micro-scales already applied; the span shifts remain
        acc_a = __fmaf_rn(x0s, d[ii][0], acc_a);
        acc_a = __fmaf_rn(x1s, d[ii][1], acc_a);
        acc_b = __fmaf_rn(x0s, d[ii][2], acc_b);
        acc_b = __fmaf_rn(x1s, d[ii][3], acc_b);
      }
    }
    // the pair's registers are free: request the same slots of the next round
    if (r + 1 < rounds) {
      load_chunk(r + 1, ip);
      load_chunk(r + 1, ip + 1);
    }
    }
  }

  // lanes t and t ^ 1 hold the two column pairs of the same activation row
  acc_a += __shfl_xor_sync(0xFFFFFFFFu, acc_a, 1);
  acc_b += __shfl_xor_sync(0xFFFFFFFFu, acc_b, 1);
  if ((t & 1) == 0) {
    red[(warp * 2 + (t >> 1)) * 16 + g] = acc_a;
    red[(warp * 2 + (t >> 1)) * 16 + g + 8] = acc_b;
  }
  }   // tile_live
  if constexpr ((MODE & RMS) != 0) {
    #pragma unroll
    for (int mm = 0; mm < 2; ++mm) {
      float v = ssq[mm];
      #pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
      if (lane == 0) rss[warp * 2 + mm] = v;
    }
  }
  __syncthreads();
  constexpr int OR = X2 ? 8 : 16;                                           // output rows of the tile
  const int gt = tid - jt * 32 * WK;                                        // thread of the tile's group
  if (tile_live && gt < OR * M) {
    const int m = gt / OR, pr = gt % OR;
    const int rr = X2 ? 2 * pr : pr;
    if (row0 + rr < N) {
      float sum = 0.0f;
      #pragma unroll
      for (int w = jt * WK; w < jt * WK + WK; ++w) {
        sum += red[(w * 2 + m) * 16 + rr];
        if constexpr (X2) sum += red[(w * 2 + m) * 16 + rr + 1];             // the residual plane
      }
      if constexpr (F == NVFP4) sum *= glob;
      if constexpr ((MODE & RMS) != 0) {
        float ss = 0.0f;
        #pragma unroll
        for (int w = 0; w < WARPS; ++w) ss += rss[w * 2 + m];
        sum *= rsqrtf(__fadd_rn(__fdiv_rn(ss, float(K)), ex.eps));
      }
      const int64_t o = X2 ? int64_t(m) * (N / 2) + row0 / 2 + pr : int64_t(m) * N + row0 + rr;
      if (out_f32) static_cast<float*>(out)[o] = sum;
      else static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(sum);
    }
  }
}

template <int F, int MR, bool UNI, int W = 8, int MODE = 0>
static cudaError_t launch_mr(const void* codes, const void* scales, float glob, const void* x, void* out,
                              bool out_f32, int M, int N, int K, cudaStream_t st, const Extra& ex = Extra{},
                              int tiles = 0, int rows = 1) {
  static std::atomic<int> attr_done[64];
  const size_t sm = (MODE & STAGE) != 0
                        ? stage_smem_bytes(F, M, K, FmtTraits<F>::four ? K / 2 : K,
                                           int64_t((K + FmtTraits<F>::block - 1) / FmtTraits<F>::block) *
                                               FmtTraits<F>::sbytes)
                        : smem_bytes(F, M, K, W);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_done[dev].load()) {
    e = cudaFuncSetAttribute(qgemv_m2_kernel<F, MR, UNI, W, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int((MODE & STAGE) != 0 ? STAGE_SMEM_LIMIT : SMEM_LIMIT));
    if (e != cudaSuccess) return e;
    attr_done[dev].store(1);
  }
  Extra exl = ex;
  exl.limit_ns = wait_limit_ns();
  exl.drop = drop_arrivals();
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(tiles > 0 ? tiles : (N + 15) / 16, rows);
  lc.blockDim = dim3(32 * W);
  lc.dynamicSmemBytes = sm;
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, qgemv_m2_kernel<F, MR, UNI, W, MODE>, static_cast<const uint8_t*>(codes),
                            static_cast<const uint8_t*>(scales), glob, static_cast<const uint16_t*>(x), out,
                            int(out_f32), M, N, K, exl);
}

// The staged-weight form (STAGE) where it pays and fits: a launch of at most
// two CTAs an SM (a larger grid streams its weights anyway), four CTAs'
// copies within an SM's shared memory, and 16-byte aligned rows.
template <int F>
static bool stage_fits(const void* codes, const void* scales, int M, int N, int K, int sms) {
  // measured (decode chains of 4096 x 4096 layers): faster for the E2M1
  // formats (mxfp4 3.30 against 3.42 us, fp4 3.30 against 3.68 us), slower
  // for mxint4, whose int4 pairing needs more registers than a 16-warp CTA has
  if constexpr (!(F == MXFP4 || F == NVFP4 || F == FP4 || F == FP4_F16)) return false;
  const int64_t rowb = FmtTraits<F>::four ? K / 2 : K;
  const int64_t srowb = int64_t((K + FmtTraits<F>::block - 1) / FmtTraits<F>::block) * FmtTraits<F>::sbytes;
  return (N + 15) / 16 <= 2 * sms && rowb % 16 == 0 && srowb % 16 == 0 &&
         (reinterpret_cast<uintptr_t>(codes) & 15u) == 0 && (reinterpret_cast<uintptr_t>(scales) & 15u) == 0 &&
         stage_smem_bytes(F, M, K, rowb, srowb) <= STAGE_SMEM_LIMIT;
}

// 8-warp CTAs (two per SM); E2M1 formats whose grid exceeds two CTAs per SM
// use 4-warp CTAs holding all eight chunks of a 4096-wide row share (three
// per SM: fewer, longer warps; measured faster for nvfp4 at N = 14336, not for
// int4 affine).
template <int F>
static cudaError_t launch_fmt(const void* codes, const void* scales, float glob, const void* x, void* out,
                              bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
  constexpr int CODES = Shape<F>::CODES;
  const int nchunk = (K + CODES - 1) / CODES;
  const bool wide = (F == MXFP4 || F == NVFP4) && (N + 15) / 16 > 2 * sms;
  if (wide) {
    const bool uni = K % (4 * CODES) == 0 && (nchunk / 4) % chunks_per_warp<F, 4>() == 0;
    if (M == 1)
      return uni ? launch_mr<F, 1, true, 4>(codes, scales, glob, x, out, out_f32, M, N, K, st)
                 : launch_mr<F, 1, false, 4>(codes, scales, glob, x, out, out_f32, M, N, K, st);
    return uni ? launch_mr<F, 2, true, 4>(codes, scales, glob, x, out, out_f32, M, N, K, st)
               : launch_mr<F, 2, false, 4>(codes, scales, glob, x, out, out_f32, M, N, K, st);
  }
  const bool uni = K % (WARPS * CODES) == 0 && (nchunk / WARPS) % chunks_in_flight<F>() == 0;
  // the staged form holds two chunks a warp at a time: whole rounds of two
  const bool stage_uni = K % (WARPS * CODES) == 0 && (nchunk / WARPS) % 2 == 0;
  if (stage_uni && stage_fits<F>(codes, scales, M, N, K, sms)) {
    const int grid = std::min((N + 15) / 16, sms);   // one CTA an SM, two tiles where there are enough
    return M == 1 ? launch_mr<F, 1, true, STAGE_WARPS, STAGE>(codes, scales, glob, x, out, out_f32, M, N, K, st,
                                                              Extra{}, grid)
                  : launch_mr<F, 2, true, STAGE_WARPS, STAGE>(codes, scales, glob, x, out, out_f32, M, N, K, st,
                                                              Extra{}, grid);
  }
  if (M == 1)
    return uni ? launch_mr<F, 1, true>(codes, scales, glob, x, out, out_f32, M, N, K, st)
               : launch_mr<F, 1, false>(codes, scales, glob, x, out, out_f32, M, N, K, st);
  return uni ? launch_mr<F, 2, true>(codes, scales, glob, x, out, out_f32, M, N, K, st)
             : launch_mr<F, 2, false>(codes, scales, glob, x, out, out_f32, M, N, K, st);
}

// Expert-routed rows: one single-row GEMV per activation row (blockIdx.y).
template <int F>
static cudaError_t launch_gather_fmt(const void* codes, const void* scales, float glob, const void* x,
                                     const int32_t* eidx, void* out, bool out_f32, int M, int N, int K, int E,
                                     cudaStream_t st) {
  constexpr int CODES = Shape<F>::CODES;
  const int nchunk = (K + CODES - 1) / CODES;
  const bool uni = K % (WARPS * CODES) == 0 && (nchunk / WARPS) % chunks_in_flight<F>() == 0;
  Extra ex{};
  ex.eidx = eidx;
  ex.E = E;
  return uni ? launch_mr<F, 1, true, 8, GATHER>(codes, scales, glob, x, out, out_f32, 1, N, K, st, ex, 0, M)
             : launch_mr<F, 1, false, 8, GATHER>(codes, scales, glob, x, out, out_f32, 1, N, K, st, ex, 0, M);
}

// Up to four weight matrices sharing the activations (BATCH), optionally
// behind a fused RMSNorm (RMS), or one matrix behind the RMSNorm.
template <int F, int MODE>
static cudaError_t launch_multi_fmt(const Extra& ex, const void* x, bool out_f32, int M, int K, int tiles,
                                    cudaStream_t st) {
  constexpr int CODES = Shape<F>::CODES;
  const int nchunk = (K + CODES - 1) / CODES;
  const bool uni = K % (WARPS * CODES) == 0 && (nchunk / WARPS) % chunks_in_flight<F>() == 0;
  const void* c0 = ex.codes[0];
  const void* s0 = ex.scales[0];
  if (M == 1)
    return uni ? launch_mr<F, 1, true, 8, MODE>(c0, s0, ex.glob[0], x, ex.out[0], out_f32, M, ex.n[0], K, st, ex, tiles)
               : launch_mr<F, 1, false, 8, MODE>(c0, s0, ex.glob[0], x, ex.out[0], out_f32, M, ex.n[0], K, st, ex, tiles);
  return uni ? launch_mr<F, 2, true, 8, MODE>(c0, s0, ex.glob[0], x, ex.out[0], out_f32, M, ex.n[0], K, st, ex, tiles)
             : launch_mr<F, 2, false, 8, MODE>(c0, s0, ex.glob[0], x, ex.out[0], out_f32, M, ex.n[0], K, st, ex, tiles);
}


// The entry points of one group of formats: a switch over Fs by fold.
template <int... Fs>
struct Group {
  static bool has(int fmt) { return ((fmt == Fs) || ...); }
  static cudaError_t launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                            bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
    cudaError_t r = cudaErrorInvalidValue;
    (void)((fmt == Fs && ((r = launch_fmt<Fs>(codes, scales, glob, x, out, out_f32, M, N, K, st, sms)), true)) || ...);
    return r;
  }
  static cudaError_t gather(int fmt, const void* codes, const void* scales, float glob, const void* x,
                            const int32_t* eidx, void* out, bool out_f32, int M, int N, int K, int E,
                            cudaStream_t st) {
    cudaError_t r = cudaErrorInvalidValue;
    (void)((fmt == Fs &&
            ((r = launch_gather_fmt<Fs>(codes, scales, glob, x, eidx, out, out_f32, M, N, K, E, st)), true)) || ...);
    return r;
  }
  static cudaError_t multi(int fmt, int mode, const Extra& ex, const void* x, bool out_f32, int M, int K, int tiles,
                           cudaStream_t st) {
    cudaError_t r = cudaErrorInvalidValue;
    (void)((fmt == Fs && ((r = mode == (BATCH | RMS) ? launch_multi_fmt<Fs, BATCH | RMS>(ex, x, out_f32, M, K, tiles, st)
                             : mode == (RMS | GATE) ? launch_multi_fmt<Fs, RMS | GATE>(ex, x, out_f32, M, K, tiles, st)
                             : mode == RMS         ? launch_multi_fmt<Fs, RMS>(ex, x, out_f32, M, K, tiles, st)
                                                   : launch_multi_fmt<Fs, BATCH>(ex, x, out_f32, M, K, tiles, st)),
                           true)) || ...);
    return r;
  }
  static cudaError_t read_status(unsigned int* status) {
    cudaError_t e = cudaMemcpyFromSymbol(status, g_gather_status, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_gather_status, &zero, sizeof(unsigned int));
  }
};

// The groups, one translation unit each.
using GroupE2M1 = Group<MXFP4, NVFP4, MXFP4X2, MXINT4, FP4, FP4_F16>;
using GroupInt = Group<INT4_AFFINE, INT4, INT4_F16, MXINT8, INT8, INT8_F16>;
using GroupFp8 = Group<MXFP8_E4M3, MXFP8_E5M2, NVFP8, NVFP8_F16, FP8_E4M3, FP8_E4M3_F16, FP8_E5M2, FP8_E5M2_F16>;

#define QFMT_M2_GROUP_API(G)                                                                                    \
  cudaError_t G##_launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out, \
                         bool out_f32, int M, int N, int K, cudaStream_t st, int sms);                          \
  cudaError_t G##_gather(int fmt, const void* codes, const void* scales, float glob, const void* x,            \
                         const int32_t* eidx, void* out, bool out_f32, int M, int N, int K, int E,              \
                         cudaStream_t st);                                                                      \
  cudaError_t G##_multi(int fmt, int mode, const Extra& ex, const void* x, bool out_f32, int M, int K,          \
                        int tiles, cudaStream_t st);                                                            \
  cudaError_t G##_status(unsigned int* status);
QFMT_M2_GROUP_API(e2m1)
QFMT_M2_GROUP_API(intg)
QFMT_M2_GROUP_API(fp8)
#undef QFMT_M2_GROUP_API

#define QFMT_M2_GROUP_DEF(G, T)                                                                                 \
  cudaError_t G##_launch(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out, \
                         bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {                         \
    return T::launch(fmt, codes, scales, glob, x, out, out_f32, M, N, K, st, sms);                              \
  }                                                                                                             \
  cudaError_t G##_gather(int fmt, const void* codes, const void* scales, float glob, const void* x,            \
                         const int32_t* eidx, void* out, bool out_f32, int M, int N, int K, int E,              \
                         cudaStream_t st) {                                                                     \
    return T::gather(fmt, codes, scales, glob, x, eidx, out, out_f32, M, N, K, E, st);                         \
  }                                                                                                             \
  cudaError_t G##_multi(int fmt, int mode, const Extra& ex, const void* x, bool out_f32, int M, int K,          \
                        int tiles, cudaStream_t st) {                                                           \
    return T::multi(fmt, mode, ex, x, out_f32, M, K, tiles, st);                                                \
  }                                                                                                             \
  cudaError_t G##_status(unsigned int* status) { return T::read_status(status); }

}  // namespace gemv_m2
}  // namespace qfmt_dev
