// Prefill GEMM on the block-scaled tensor cores (tcgen05.mma kind::mxf8f6f4),
// the weights fed as stored, M > 16:
//   out[M, N] = X[M, K] (bf16) . dequant(W[N, K])^T, float32 accumulation,
// for the MX formats whose element the hardware reads directly: mxfp4 (E2M1),
// mxfp8 E4M3 and E5M2, each with an E8M0 scale per 32 along K.
//
// The block-factored value it computes is rlx-cpu thunk/ops/quant.rs
// lowp_scaled_matmul: per K block, acc += (a_s . b_s) . sum_k dec(a) dec(b),
// with both operands block-scaled; metaltile PR #250 names Blackwell tcgen05
// scaled-MMA (MXFP) as the CUDA payoff of its formats.  Here the activation
// side is made block-scaled exactly enough for the bf16 contract:
//
//  * xquant (one kernel) splits X into two MXFP8 E4M3 terms per block of 32:
//      s1 = 2^e1, the smallest power of two with amax(x) <= 448 s1;
//      hi = E4M3_rne_sat(x / s1);  r = x - hi s1 (exact in float32);
//      s2 = 2^e2 from amax(r) the same way;  lo = E4M3_rne_sat(r / s2).
//    A bf16 value has 8 significant bits and hi keeps the top 4 (rounded), so
//    r has at most 3 and hi s1 + lo s2 = x exactly whenever hi and lo are
//    normal E4M3 values (x within 2^14 of its block's largest); smaller values
//    carry an absolute error below 2^-21 amax of the block.  The codes go to
//    the workspace as [M, K] bytes (hi, then lo) and the scales as 512-byte
//    atoms of 128 rows x 4 K blocks (umma::sf_atom_offset), the layout
//    tcgen05.cp copies into tensor memory.
//  * the GEMM kernel, CTA tile 128 (M) x 256 (N), K step 128, three stages:
//      warp 0  one thread issues TMA loads of the hi and lo X tiles and the W
//              code tile (128B-swizzled, K-major; E2M1 codes through the
//              16U4_ALIGN16B type, which places 16 codes in each 16-byte
//              unit's low 8 bytes, the layout kind::mxf8f6f4 reads for E2M1)
//              and bulk-copies the two X scale atoms; it owns the TMEM
//              allocation;
//      warp 1  walks the stages as a warp (lane 0 waits on the barriers and
//              broadcasts the outcome, so the stage addresses stay
//              warp-uniform); one elected lane copies the stage's scale
//              atoms into tensor memory (tcgen05.cp .32x128b.warpx4) and
//              issues, per K block of 32, two MMAs into one accumulator:
//              hi . W under (s1, s_w) and lo . W under (s2, s_w).  Issued
//              from a single lane's branch, each tcgen05 instruction cost
//              ~67 cycles of the issuing thread; from the converged warp ~50;
//      warp 2  gathers the stage's W scales (one 32-bit word = 4 K blocks per
//              row) into two scale atoms in shared memory;
//      warps 4-7 drain the accumulator (tcgen05.ld) and store bf16/float32.
//
// The same kernel serves the quantized-activation products: one E4M3 term
// (W . A8, kind::mxf8f6f4), and the all-FP4 product (W . A4: X packed in W's
// FP4 family, both operands E2M1 two codes to a byte: MXFP4 on kind::mxf4
// with two E8M0 scales per row and instruction, or NVFP4 on kind::mxf4nvf4
// with four UE4M3 scales and the two tensors' globals in the epilogue), each
// optionally on tall 256-row tiles.
//
// Every mbarrier wait is bounded; on expiry the kernel records it in the
// device status word, lets issued copies and MMAs land, frees its tensor
// memory and exits without writing its tile.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "decode.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace qfmt_dev {

__device__ unsigned int g_mx_status;

namespace mx {

using namespace tc;

constexpr int BM = 128, BN_MAX = 256, BK = 128;   // BK: K elements (= bytes of an 8-bit code row) per stage
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * BK;              // 16 KiB: one X term
constexpr int B_BYTES = BN_MAX * BK;          // 32 KiB: up to 256 rows of 128 codes (E2M1: 16 in each 16-byte unit)
constexpr int SF_BYTES = 512;                 // one scale atom: 128 rows x 4 K blocks
constexpr int STAGE_BYTES = 2 * A_BYTES + B_BYTES;
constexpr int SF_STAGE = 4 * SF_BYTES;        // hi atom, lo atom, two W atoms (rows 0-127, 128-255)
constexpr int SF_STAGE_A4 = 8 * SF_BYTES;     // all-FP4 form: two K atoms each of two X tiles and two W row groups
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGES * SF_STAGE + 256;
constexpr int SMEM_BYTES_A4 = 1024 + STAGES * STAGE_BYTES + STAGES * SF_STAGE_A4 + 256;
constexpr int SF_STAGE_NV = 16 * SF_BYTES;    // nvfp4 all-FP4: four K atoms of each X tile, eight of W
constexpr int SMEM_BYTES_NV = 1024 + STAGES * STAGE_BYTES + STAGES * SF_STAGE_NV + 256;
constexpr int THREADS = 256;
constexpr int TMEM_COLS = 512;                // accumulator 256 columns + 16 scale columns a stage
constexpr int SF_COL0 = 256;

// Workspace layout (bytes) for M rows and K columns: hi codes, lo codes, hi
// scale atoms, lo scale atoms; each part 1024-byte aligned.
struct WsLayout {
  size_t hi, lo, sf_hi, sf_lo, total;
};
inline size_t align1k(size_t v) { return (v + 1023) & ~size_t(1023); }
inline WsLayout ws_layout(int64_t M, int64_t K) {
  WsLayout w;
  const size_t codes = size_t(M) * size_t(K);
  const size_t sf = size_t((M + BM - 1) / BM) * size_t(K / BK) * SF_BYTES;
  w.hi = 0;
  w.lo = align1k(codes);
  w.sf_hi = w.lo + align1k(codes);
  w.sf_lo = w.sf_hi + align1k(sf);
  w.total = w.sf_lo + align1k(sf);
  return w;
}

// --------------------------------------------------------------- xquant ---

// E8M0 exponent of the smallest power of two s with amax <= 448 s, from the
// float32 bits of amax (>= 0, finite): amax = 1.m 2^E fits 448 2^(E-8) =
// 1.75 2^E when 1.m <= 1.75, else takes 2^(E-7); below 2^-119 the smallest
// scale 2^-127 already fits.  Returns the biased byte (e + 127).
__device__ __forceinline__ uint32_t e8m0_for_e4m3(float amax) {
  const uint32_t a = __float_as_uint(amax);
  if (a >= 0x7F800000u) return 255u;                       // Inf / NaN in the block: a NaN scale
  if (a < 0x04000000u) return 0u;
  const int e = int(a >> 23) - 127 - 8 + ((a & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  return uint32_t(min(max(e, -127), 127) + 127);
}

// 2^-(b - 127) as a float32 (b <= 254): the exact reciprocal of the scale.
__device__ __forceinline__ float e8m0_recip(uint32_t b) {
  const int e = 127 - int(b);                               // exponent of the reciprocal, -127 .. 127
  return e >= -126 ? __uint_as_float(uint32_t(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// Two float32 -> two E4M3 bytes (round to nearest even, saturating to +-448),
// `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t h;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
  return h;
}

// Two E4M3 bytes (low byte first) -> their values as float32 (exact).
__device__ __forceinline__ void e4m3x2_f32(uint32_t two, float& lo, float& hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(uint16_t(two)));
  lo = __half2float(__ushort_as_half(uint16_t(r & 0xFFFFu)));
  hi = __half2float(__ushort_as_half(uint16_t(r >> 16)));
}

// One block of 32 bf16 activations (16 words, value 2i in the low half of
// word i) -> hi and lo E4M3 codes (8 words each, code i in byte i % 4 of word
// i / 4) and their E8M0 scale bytes c1, c2 (see the file comment).
__device__ __forceinline__ void split_block(const uint32_t (&w)[16], uint32_t& c1, uint32_t& c2, uint32_t (&hi)[8],
                                            uint32_t (&lo)[8]) {
  float v[32];
  float amax = 0.0f;
  #pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    amax = fmaxf(amax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
  }
  // an infinity gives the block the NaN scale (255); a NaN element (which
  // fmaxf passes over) stays a NaN code: either way its outputs are NaN
  c1 = e8m0_for_e4m3(amax);
  const float s1 = e8m0_f32(c1), r1 = c1 == 255u ? 0.0f : e8m0_recip(c1);
  float ramax = 0.0f;
  #pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t h = e4m3x2(__fmul_rn(v[2 * i], r1), __fmul_rn(v[2 * i + 1], r1));
    float h0, h1;
    e4m3x2_f32(h, h0, h1);
    v[2 * i] = __fmaf_rn(-h0, s1, v[2 * i]);               // exact residuals
    v[2 * i + 1] = __fmaf_rn(-h1, s1, v[2 * i + 1]);
    ramax = fmaxf(ramax, fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1])));
    if (i & 1) hi[i >> 1] |= h << 16;
    else hi[i >> 1] = h;
  }
  c2 = c1 == 255u ? 255u : e8m0_for_e4m3(ramax);
  const float r2 = c2 == 255u ? 0.0f : e8m0_recip(c2);
  #pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint32_t l = e4m3x2(__fmul_rn(v[2 * i], r2), __fmul_rn(v[2 * i + 1], r2));
    if (i & 1) lo[i >> 1] |= l << 16;
    else lo[i >> 1] = l;
  }
}

__device__ __forceinline__ void load_block(const __nv_bfloat16* src, uint32_t (&w)[16]) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  #pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = __ldg(s4 + i);
    w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
  }
}

// One warp per (row, 32 consecutive blocks of 32): lane l takes block b0 + l.
// Rows past M (up to the 128-row tile) get neutral scale words only.
// Grouped rows (row_of != nullptr): workspace row m holds activation row
// row_of[m] (-1: a padding row, zero), for m below *total (the routing
// kernel's output).
__global__ void __launch_bounds__(256) xquant_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ ws,
                                                     WsLayout lay, int M, int K, const int* __restrict__ row_of,
                                                     const int* __restrict__ total) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nblk = K / 32, chunks = (nblk + 31) / 32;
  const int mpad = (M + BM - 1) / BM * BM;
  const int m = warp / chunks, b = (warp - m * chunks) * 32 + lane;
  if (m >= mpad) return;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (row_of && m >= __ldg(total)) return;
  const int src = row_of ? __ldg(row_of + m) : m;
  const bool live = b < nblk;
  uint32_t c1 = 127u, c2 = 127u;
  if (live && m < M) {
    uint32_t w[16], hi[8], lo[8];
    if (src >= 0) load_block(x + int64_t(src) * K + int64_t(b) * 32, w);
    else for (int i = 0; i < 16; ++i) w[i] = 0u;
    split_block(w, c1, c2, hi, lo);
    uint4* dh = reinterpret_cast<uint4*>(ws + lay.hi + size_t(m) * K + size_t(b) * 32);
    uint4* dl = reinterpret_cast<uint4*>(ws + lay.lo + size_t(m) * K + size_t(b) * 32);
    dh[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    dh[1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    dl[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    dl[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  }
  // four blocks of one row share a 32-bit scale cell of the atom
  uint32_t w1 = c1, w2 = c2;
  #pragma unroll
  for (int d = 1; d < 4; ++d) {
    w1 |= __shfl_down_sync(0xFFFFFFFFu, c1, d) << (8 * d);
    w2 |= __shfl_down_sync(0xFFFFFFFFu, c2, d) << (8 * d);
  }
  if (live && (lane & 3) == 0) {
    const size_t atom = size_t(m / BM) * size_t(K / BK) + size_t(b / 4);
    const uint32_t off = umma::sf_atom_offset(uint32_t(m % BM), 0);
    *reinterpret_cast<uint32_t*>(ws + lay.sf_hi + atom * SF_BYTES + off) = w1;
    *reinterpret_cast<uint32_t*>(ws + lay.sf_lo + atom * SF_BYTES + off) = w2;
  }
}

// ----------------------------------------------------------------- GEMM ---

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Both operands E2M1 packed two codes to a byte, K 64 an instruction, four
// UE4M3 scales of each row (one a block of 16: the whole scale cell).
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// Both operands E2M1 packed two codes to a byte, K 64 an instruction, two
// E8M0 scales of each row (the scale cell's bytes from the descriptor's id).
__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

struct MxParams {
  const uint8_t* wscales;   // [N, K/32] E8M0 (grouped: [E N, K/32])
  const uint8_t* sf_hi;     // X scale atoms (workspace)
  const uint8_t* sf_lo;
  void* out;
  int M, N, K;
  int out_f32;
  int kb_per;               // K steps per split (grid z = the splits of one cluster)
  uint64_t limit_ns;
  int drop_arrivals;
  // grouped rows (expert-routed): nullptr otherwise.  route_off[0..E] are the
  // 128-aligned row offsets of each expert's segment of the workspace rows,
  // row_of[m] the activation (and output) row of workspace row m (-1: padding)
  const int* route_off;
  const int* row_of;
  int E;
  // nvfp4 all-FP4 form: the output is scaled by the weight's global times the
  // activation's (computed on the device, read after the dependent wait)
  float gw;
  const float* gx;
};

template <int F> constexpr uint32_t b_type() {
  return F == MXFP4 ? umma::F8F6F4_E2M1 : (F == MXFP8_E5M2 ? umma::F8F6F4_E5M2 : umma::F8F6F4_E4M3);
}

// BN: the tile's N (256, or 224 where that fills the waves of 152 SMs better).
// TWO: the activations as two E4M3 terms (hi + lo, two MMAs per block), else
// one (the quantized-activation product: one MMA per block).
// TALL (one term only): a CTA takes two 128-row M tiles (256 x BN) into two
// accumulators sharing each stage's W tile, the second X tile in the stage
// memory the lo term uses otherwise: 60 KiB land per K step for twice the
// output of a 44 KiB single-tile step.  Tensor memory: accumulators at
// columns 0 and 256, the stages' scale slots at 224, 240 and 480.
// A4 (one term, mxfp4 weights): the all-FP4 product.  The activation tile is
// E2M1 packed two to a byte like the weights, and both enter kind::mxf4 as
// stored: a stage's 128-byte rows hold 256 codes (K 64 an instruction), so it
// carries twice the K of an 8-bit stage in the same bytes, with two K atoms
// of scales per tile.  Tensor memory: 32 scale columns a stage slot (X tile 0
// at +0 / +4, tile 1 at +8 / +12, W at +16 .. +31: rows 0-127 and 128-255 of
// K atom 0, then of K atom 1); with tall tiles only two slots fit (columns
// 224 and 480) and a slot is refilled once the MMAs of the stage before last
// have completed.
// NV (with A4; nvfp4 weights): the NVFP4 form, kind::mxf4nvf4 with UE4M3
// scales per 16 values.  A K step carries 16 blocks a row: four scale cells,
// so four K atoms for the X tile and eight for W (48 columns a slot at 256 +
// 48 s: X at +0 .. +15, then W's row groups 0 and 1 of K atom a at +16 + 8a
// and +20 + 8a); each MMA reads a whole cell.  With tall tiles a step's 64
// scale columns fit once, split over the two gaps beside the accumulators
// (X tiles at 224 .. 255, W at 480 .. 511): the slot is refilled after the
// MMAs of the step before have completed.  The epilogue multiplies by the two
// tensors' globals.
// A K split runs its splits as a cluster along z; each split's float32
// partial tile goes to its drained stage memory and the cluster sums them
// through distributed shared memory in rank order.
template <int F, int BN, bool TWO = true, bool TALL = false, bool A4 = false, bool NV = false>
__global__ void __launch_bounds__(THREADS, 1) qgemm_mx_kernel(const __grid_constant__ CUtensorMap xhi_map,
                                                              const __grid_constant__ CUtensorMap xlo_map,
                                                              const __grid_constant__ CUtensorMap w_map,
                                                              const MxParams p) {
  static_assert(BN % 32 == 0 && BN <= BN_MAX && BN > 128, "two W scale atoms a stage");
  static_assert(!TALL || (!TWO && BN == 224), "tall tiles: one term, 224 columns");
  static_assert(!A4 || (!TWO && F == (NV ? NVFP4 : MXFP4)), "the all-FP4 form: one E2M1 activation term");
  static_assert(!NV || A4, "the NVFP4 form is an all-FP4 form");
  // bytes a stage's copies deliver: the two X tiles (terms, or M halves), the
  // W codes (E2M1 through 16U4_ALIGN16B: the 8 data bytes of every 16-byte
  // unit, the gaps are not written; packed A4 tiles: every byte) and the X
  // scale atoms (A4: two K atoms a tile)
  constexpr int TERMS = (TWO || TALL) ? 2 : 1;
  constexpr int XA = NV ? 4 : (A4 ? 2 : 1);
  constexpr int X2 = NV ? 12 : XA;                  // scale atoms of the second X tile (NV: after W's)
  constexpr int SFS = NV ? SF_STAGE_NV : (A4 ? SF_STAGE_A4 : SF_STAGE);
  constexpr uint32_t TX_BYTES =
      TERMS * (A_BYTES + XA * SF_BYTES) + ((F == MXFP4 && !A4) ? BN * BK / 2 : BN * BK);
  constexpr int PSTRIDE = BN + 4;                 // floats per partial-tile row (K split)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sf_area = smem + STAGES * STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sf_area + STAGES * SFS);
  // bars[0..S): stage copies landed (TMA and bulk bytes), [S..2S): stage W scales written (the scale warp),
  // [2S..3S): stage empty (MMA commit), [3S]: accumulator done
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 3 * STAGES + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM * (TALL ? 2 : 1);
  // grouped rows: the tile's expert (its weights are rows [e N, e N + N) of the
  // stacked matrix); tiles past the last segment have nothing to do (every CTA
  // of a K-split cluster shares blockIdx.y, so a cluster leaves whole)
  int wrow0 = 0;
  if (p.route_off) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the routing kernel's tables
    if (m0 >= __ldg(p.route_off + p.E)) return;
    int e = 0;
    while (e + 1 < p.E && __ldg(p.route_off + e + 1) <= m0) ++e;
    wrow0 = e * p.N;
  }
  const int nk = p.K / (A4 ? 2 * BK : BK);        // K steps (A4: 256 codes in a 128-byte row)
  const int katoms = p.K / (NV ? 64 : BK);          // scale atoms (4 K blocks) along a row
  const int j0 = blockIdx.z * p.kb_per, j1 = min(nk, j0 + p.kb_per);   // this split's K steps
  const int nloc = j1 - j0;
  const bool split_k = gridDim.z > 1;
  const uint32_t sbase = smem_u32(smem), sfbase = smem_u32(sf_area), bar0 = smem_u32(bars);
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto sf_full = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  const uint32_t done_bar = bar0 + 8u * (3 * STAGES);
  auto a_hi = [&](int s) { return sbase + uint32_t(s * STAGE_BYTES); };
  auto a_lo = [&](int s) { return sbase + uint32_t(s * STAGE_BYTES + A_BYTES); };
  auto b_tile = [&](int s) { return sbase + uint32_t(s * STAGE_BYTES + 2 * A_BYTES); };
  // i: 0 hi, 1 lo, 2-3 W (A4: 0-1 X tile 0, 2-3 X tile 1, 4-7 W; two K atoms
  // each; NV: 0-3 X, 4-11 W: K atom a, row group g at 4 + 2a + g)
  auto sf_s = [&](int s, int i) { return sfbase + uint32_t(s * SFS + i * SF_BYTES); };
  auto fail = [&]() {
    *abort_flag = 1u;
    atomicOr(&g_mx_status, 1u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(sf_full(s), 1);
      mbar_init(empty(s), 1);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xhi_map)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xlo_map)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&w_map)) : "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32((const void*)tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      // the first stages' W tiles do not depend on the preceding kernel: in
      // flight before the dependent wait (each stage's barrier takes the
      // whole step's bytes now; its X parts follow after the wait)
      const int pre = nloc < STAGES ? nloc : STAGES;
      for (int i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(full(i), TX_BYTES);
        tma_load_2d(b_tile(i), &w_map, (j0 + i) * BK, wrow0 + n0, full(i));
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");   // the workspace comes from the preceding xquant
      // the X scale atoms of this tile's 128-row M tile(s); a second M half
      // past M has none (its rows are zeros and stored nowhere): the first
      // half's atoms stand in
      const size_t mt0 = TALL ? size_t(2 * blockIdx.y) : size_t(blockIdx.y);
      const uint8_t* sfh = p.sf_hi + mt0 * size_t(katoms) * SF_BYTES;
      const uint8_t* sfl = TALL ? (m0 + BM < p.M ? sfh + size_t(katoms) * SF_BYTES : sfh)
                                : p.sf_lo + size_t(blockIdx.y) * size_t(katoms) * SF_BYTES;
      int issued = pre;
      for (int i = 0; i < nloc; ++i) {
        const int s = i % STAGES, j = j0 + i;
        const uint32_t ph = (i / STAGES) & 1;
        if (*abort_flag) break;
        if (i >= pre) {
          if (!mbar_wait(empty(s), ph ^ 1u, p.limit_ns)) { fail(); break; }
          mbar_arrive_expect_tx(full(s), TX_BYTES);
          tma_load_2d(b_tile(s), &w_map, j * BK, wrow0 + n0, full(s));
        }
        tma_load_2d(a_hi(s), &xhi_map, j * BK, m0, full(s));
        if constexpr (TWO) tma_load_2d(a_lo(s), &xlo_map, j * BK, m0, full(s));
        if constexpr (TALL) tma_load_2d(a_lo(s), &xhi_map, j * BK, m0 + BM, full(s));   // the second M half
        bulk_load(sf_s(s, 0), sfh + size_t(j) * XA * SF_BYTES, XA * SF_BYTES, full(s));
        if constexpr (TWO || TALL) bulk_load(sf_s(s, X2), sfl + size_t(j) * XA * SF_BYTES, XA * SF_BYTES, full(s));
        issued = i + 1 > pre ? i + 1 : pre;
      }
      // every issued copy lands before the CTA may exit
      for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
        if (!mbar_wait(full(i % STAGES), (i / STAGES) & 1, p.limit_ns)) fail();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The warp walks the loop together (lane 0 waits, the outcome is
    // broadcast), so the stage addresses are warp-uniform; one elected lane
    // issues the tensor-core instructions.
    const bool leader = elect_one();
    constexpr uint32_t BT = b_type<F>();
    // scale slots in tensor memory: one a stage, but two for A4 tall tiles
    constexpr int SLOTS = (A4 && TALL) ? (NV ? 1 : 2) : STAGES;
    for (int i = 0; i < nloc; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      int go = 1;
      if (lane == 0) {
        go = *abort_flag == 0u;
        if (go && !(mbar_wait(full(s), ph, p.limit_ns) && mbar_wait(sf_full(s), ph, p.limit_ns))) {
          fail();
          go = 0;
        }
        if constexpr (SLOTS < STAGES) {
          // the slot's previous user, step i - SLOTS: its MMAs (which read the
          // slot) complete before the slot is copied over.  Its commit is the
          // newest phase of that stage's empty barrier this thread has issued.
          if (go && i >= SLOTS) {
            const int pi = i - SLOTS;
            if (!mbar_wait(empty(pi % STAGES), uint32_t(pi / STAGES) & 1u, p.limit_ns)) {
              fail();
              go = 0;
            }
          }
        }
      }
      if (!__shfl_sync(0xFFFFFFFFu, go, 0)) break;
      tc_fence_after();
      const uint64_t dh = desc_sw128(a_hi(s)), dl = desc_sw128(a_lo(s)), db = desc_sw128(b_tile(s));
      if (leader) {
        if constexpr (NV && TALL) {
          // X tile 0 atoms at 224 + 4a, tile 1 at 240 + 4a, W (row group g, K atom a) at 480 + 8a + 4g
          const uint32_t xs = tmem + 224u, wsl = tmem + 480u;
          #pragma unroll
          for (int a = 0; a < 4; ++a) {
            tmem_cp_sf(xs + uint32_t(4 * a), umma::smem_desc_sf32x16(sf_s(s, a)));
            tmem_cp_sf(xs + uint32_t(16 + 4 * a), umma::smem_desc_sf32x16(sf_s(s, 12 + a)));
          }
          #pragma unroll
          for (int a = 0; a < 8; ++a) tmem_cp_sf(wsl + uint32_t(4 * a), umma::smem_desc_sf32x16(sf_s(s, 4 + a)));
          constexpr uint32_t id = umma::idesc_mxf4nvf4(BM, BN);
          #pragma unroll
          for (int kk = 0; kk < 4; ++kk) {   // K 64 (+32 bytes) an instruction: the whole cell of K atom kk
            mma_mxf4nvf4(tmem, dh + uint64_t(2 * kk), db + uint64_t(2 * kk), id, xs + 4u * kk, wsl + 8u * kk,
                         (i | kk) != 0);
            mma_mxf4nvf4(tmem + 256u, dl + uint64_t(2 * kk), db + uint64_t(2 * kk), id, xs + 16u + 4u * kk,
                         wsl + 8u * kk, (i | kk) != 0);
          }
        } else if constexpr (NV) {
          const uint32_t slot = tmem + uint32_t(BN_MAX + 48 * s);
          #pragma unroll
          for (int a = 0; a < 12; ++a) tmem_cp_sf(slot + uint32_t(4 * a), umma::smem_desc_sf32x16(sf_s(s, a)));
          constexpr uint32_t id = umma::idesc_mxf4nvf4(BM, BN);
          #pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // K 64 (+32 bytes) an instruction: the whole cell of K atom kk
            mma_mxf4nvf4(tmem, dh + uint64_t(2 * kk), db + uint64_t(2 * kk), id, slot + 4u * kk, slot + 16u + 8u * kk,
                         (i | kk) != 0);
        } else if constexpr (A4) {
          const uint32_t slot = tmem + uint32_t(TALL ? ((i % SLOTS) == 0 ? 224 : 480) : BN_MAX + 32 * s);
          #pragma unroll
          for (int a = 0; a < 8; ++a)
            if (TALL || a < 2 || a >= 4) tmem_cp_sf(slot + uint32_t(4 * a), umma::smem_desc_sf32x16(sf_s(s, a)));
          #pragma unroll
          for (int kk = 0; kk < 4; ++kk) {   // K 64 (+32 bytes) an instruction: K atom kk / 2, bytes 2 (kk % 2) + 0, 1
            const uint32_t a = uint32_t(kk >> 1), sid = 2u * uint32_t(kk & 1);
            const uint32_t id = umma::idesc_mxf4(BM, BN, sid, sid);
            mma_mxf4(tmem, dh + uint64_t(2 * kk), db + uint64_t(2 * kk), id, slot + 4u * a, slot + 16u + 8u * a,
                     (i | kk) != 0);
            if constexpr (TALL)
              mma_mxf4(tmem + 256u, dl + uint64_t(2 * kk), db + uint64_t(2 * kk), id, slot + 8u + 4u * a,
                       slot + 16u + 8u * a, (i | kk) != 0);
          }
        } else {
          // hi (first M half): +0, lo (second M half): +4, W: +8 (rows 0-127), +12 (128-255)
          const uint32_t sfc = tmem + uint32_t(TALL ? (s < 2 ? 224 + 16 * s : 480) : SF_COL0 + 16 * s);
          tmem_cp_sf(sfc + 0, umma::smem_desc_sf32x16(sf_s(s, 0)));
          if constexpr (TWO || TALL) tmem_cp_sf(sfc + 4, umma::smem_desc_sf32x16(sf_s(s, 1)));
          tmem_cp_sf(sfc + 8, umma::smem_desc_sf32x16(sf_s(s, 2)));
          tmem_cp_sf(sfc + 12, umma::smem_desc_sf32x16(sf_s(s, 3)));
          #pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {   // +32 bytes along K per instruction
            const uint32_t id = umma::idesc_mxf8f6f4(umma::F8F6F4_E4M3, BT, BM, BN, uint32_t(kk), uint32_t(kk));
            mma_mx(tmem, dh + uint64_t(2 * kk), db + uint64_t(2 * kk), id, sfc + 0, sfc + 8, (i | kk) != 0);
            if constexpr (TWO) mma_mx(tmem, dl + uint64_t(2 * kk), db + uint64_t(2 * kk), id, sfc + 4, sfc + 8, 1u);
            if constexpr (TALL)
              mma_mx(tmem + 256u, dl + uint64_t(2 * kk), db + uint64_t(2 * kk), id, sfc + 4, sfc + 8, (i | kk) != 0);
          }
        }
        mma_commit(empty(s));
      }
      __syncwarp();
    }
    if (leader) mma_commit(done_bar);
  } else if (warp == 2) {
    // ------------------------------------------- W scales -> scale atoms
    // lane l gathers rows n0 + l + 32 i (i = 0..7): the 4 E8M0 bytes of K
    // blocks 4j..4j+3 are one aligned 32-bit word of the row (K % 128 == 0);
    // an A4 step takes two consecutive words (K % 256 == 0); an NV step the
    // 16 E4M3 bytes of its 16 blocks, four words
    const int row_words = p.K / (NV ? 64 : 128);
    const uint32_t* ws32 = reinterpret_cast<const uint32_t*>(p.wscales);
    using SW = typename std::conditional<NV, uint4, uint2>::type;
    auto load = [&](int i, SW (&v)[8]) {
      #pragma unroll
      for (int t = 0; t < 8; ++t) {
        const int r = lane + 32 * t, n = n0 + r;
        const bool in = i < nloc && r < BN && n < p.N;
        const uint32_t* row = ws32 + int64_t(wrow0 + n) * row_words;
        if constexpr (NV) v[t] = in ? __ldg(reinterpret_cast<const uint4*>(row) + j0 + i) : make_uint4(0u, 0u, 0u, 0u);
        else if constexpr (A4) v[t] = in ? __ldg(reinterpret_cast<const uint2*>(row) + j0 + i) : make_uint2(0u, 0u);
        else v[t] = make_uint2(in ? __ldg(row + j0 + i) : 0u, 0u);
      }
    };
    SW cur[8], nxt[8];
    load(0, cur);
    load(1, nxt);
    for (int i = 0; i < nloc; ++i) {
      const int s = i % STAGES;
      const uint32_t ph = (i / STAGES) & 1;
      int ok = 1;
      if (lane == 0) ok = (*abort_flag == 0u) && mbar_wait(empty(s), ph ^ 1u, p.limit_ns);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0 && *abort_flag == 0u) fail();
        break;
      }
      SW nx2[8];
      load(i + 2, nx2);
      #pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint32_t off = umma::sf_atom_offset(uint32_t(lane + 32 * (t % 4)), 0);
        if constexpr (NV) {   // K atom a of row group t / 4 at 4 + 2a + t / 4
          const uint32_t w4[4] = {cur[t].x, cur[t].y, cur[t].z, cur[t].w};
          #pragma unroll
          for (int a = 0; a < 4; ++a) {
            const uint32_t dst = sf_s(s, 4 + 2 * a + t / 4) + off;
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(dst), "r"(w4[a]) : "memory");
          }
        } else {
          const uint32_t dst = sf_s(s, (A4 ? 4 : 2) + t / 4) + off;   // row group t / 4
          asm volatile("st.shared.u32 [%0], %1;" ::"r"(dst), "r"(cur[t].x) : "memory");
          if constexpr (A4) {   // K atom 1 of the step
            const uint32_t dst1 = sf_s(s, 6 + t / 4) + off;
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(dst1), "r"(cur[t].y) : "memory");
          }
        }
        cur[t] = nxt[t];
        nxt[t] = nx2[t];
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0 && !p.drop_arrivals) mbar_arrive(sf_full(s));
    }
  }
  if (warp >= 4 || (TALL && warp < 4)) {
    // --------------------------------------------------------------- epilogue
    // warps 4-7 drain accumulator 0; with tall tiles warps 0-3, done with
    // their roles, drain accumulator 1 at the same time (a warp reads the
    // tensor-memory lanes of its own quadrant, warp % 4)
    __syncwarp();
    int ok = 1;
    if (lane == 0) ok = mbar_wait(done_bar, 0, p.limit_ns);
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok && lane == 0) fail();
    tc_fence_after();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int q = warp & 3;
    float gsc = 1.0f;                               // NV: the two globals (the activation's from the quantizer)
    if constexpr (NV) gsc = __fmul_rn(p.gw, *p.gx);
    const int hf0 = (TALL && warp < 4) ? 1 : 0;
    #pragma unroll 1
    for (int hf = hf0; hf < hf0 + 1; ++hf) {        // this warp's accumulator: an M half of a tall tile
    // the output row of this lane's accumulator row (grouped: through row_of)
    int m = m0 + hf * BM + q * 32 + lane;
    if (p.route_off) m = m < __ldg(p.route_off + p.E) ? __ldg(p.row_of + m) : -1;
    const bool live = ok && *abort_flag == 0u && m >= 0;
    #pragma unroll 1
    for (int cb = 0; cb < BN / 32; ++cb) {
      uint32_t r[32];
      tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(hf * 256 + cb * 32), r);
      if constexpr (NV) {
        #pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(__fmul_rn(__uint_as_float(r[j]), gsc));
      }
      if (split_k) {   // this split's partial tile into the drained stage memory
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(smem) + (q * 32 + lane) * PSTRIDE + cb * 32);
        #pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                               __uint_as_float(r[4 * j + 3]));
        continue;
      }
      const int nb = n0 + cb * 32;
      if (!live || m >= p.M || nb >= p.N) continue;
      const int ncols = p.N - nb < 32 ? p.N - nb : 32;
      if (p.out_f32) {
        float* o = static_cast<float*>(p.out) + int64_t(m) * p.N + nb;
        if (ncols == 32 && (p.N & 3) == 0) {
          #pragma unroll
          for (int j = 0; j < 8; ++j)
            reinterpret_cast<float4*>(o)[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                                          __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        } else {
          #pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncols) o[j] = __uint_as_float(r[j]);
        }
      } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + int64_t(m) * p.N + nb;
        if (ncols == 32 && (p.N & 7) == 0) {
          #pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t h[4];
            #pragma unroll
            for (int t = 0; t < 4; ++t)
              h[t] = f32_to_bf16bits(__uint_as_float(r[8 * j + 2 * t])) |
                     (f32_to_bf16bits(__uint_as_float(r[8 * j + 2 * t + 1])) << 16);
            reinterpret_cast<uint4*>(o)[j] = make_uint4(h[0], h[1], h[2], h[3]);
          }
        } else {
          #pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < ncols) o[j] = __float2bfloat16_rn(__uint_as_float(r[j]));
        }
      }
    }
    }   // hf
  }

  if (split_k) {
    // The splits of one tile form a cluster: each CTA sums a slice of the tile
    // over the cluster's partial tiles (rank order) and stores it; a CTA whose
    // wait expired holds no valid partial, and then no CTA writes its slice.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    cluster_sync();
    uint32_t rank, csize;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
    uint32_t any_abort = 0u;
    for (uint32_t r = 0; r < csize; ++r) any_abort |= ld_cluster_u32(smem_u32((const void*)abort_flag), r);
    constexpr int E = BM * (BN / 4);                       // float4 elements of the tile
    const int e0 = int(rank) * E / int(csize), e1 = any_abort ? e0 : (int(rank) + 1) * E / int(csize);
    for (int e = e0 + int(threadIdx.x); e < e1; e += THREADS) {
      const int row = e / (BN / 4), c4 = e - row * (BN / 4);
      int m = m0 + row;
      const int n = n0 + 4 * c4;
      if (p.route_off) m = m < __ldg(p.route_off + p.E) ? __ldg(p.row_of + m) : -1;
      if (m < 0 || m >= p.M || n >= p.N) continue;
      const uint32_t sa = sbase + uint32_t((row * PSTRIDE + 4 * c4) * 4);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t r = 0; r < csize; ++r) {
        const float4 w = ld_cluster_f32x4(sa, r);
        v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
      }
      const float f4[4] = {v.x, v.y, v.z, v.w};
      const bool vec = n + 4 <= p.N && (p.N & 3) == 0;
      if (p.out_f32) {
        float* o = static_cast<float*>(p.out) + int64_t(m) * p.N + n;
        if (vec) *reinterpret_cast<float4*>(o) = v;
        else for (int j = 0; j < 4 && n + j < p.N; ++j) o[j] = f4[j];
      } else {
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + int64_t(m) * p.N + n;
        if (vec) {
          *reinterpret_cast<uint2*>(o) = make_uint2(f32_to_bf16bits(v.x) | (f32_to_bf16bits(v.y) << 16),
                                                    f32_to_bf16bits(v.z) | (f32_to_bf16bits(v.w) << 16));
        } else {
          for (int j = 0; j < 4 && n + j < p.N; ++j) o[j] = __float2bfloat16_rn(f4[j]);
        }
      }
    }
    cluster_sync();   // no CTA leaves while the others still read its partial tile
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ------------------------------------------------------------------ host ---

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// A K-major [rows, K] map with 128-element x `box_rows` boxes, 128B swizzle.
static bool make_map(EncodeTiledFn enc, CUtensorMap* map, CUtensorMapDataType dt, const void* base, int64_t K,
                     int64_t rows, int64_t row_bytes, uint32_t box_rows) {
  const cuuint64_t gdim[2] = {cuuint64_t(K), cuuint64_t(rows)};
  const cuuint64_t gstride[1] = {cuuint64_t(row_bytes)};
  const cuuint32_t box[2] = {cuuint32_t(BK), box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

static std::atomic<uint64_t> g_limit_ns{2000000000ull};
static std::atomic<int> g_drop{0};
static std::atomic<int> g_force_bn{0}, g_force_s{0};   // plan overrides for measurements (0: the planner's)
static std::atomic<int> g_force_tall{0};                // quantized-activation GEMM: 0 plan, 1 no tall tiles, 2 tall where allowed
static std::atomic<int> g_gemv_off{0}, g_gemv_s{0};     // decode GEMV: off (mma.sync GEMVs), forced K split

// Tile width and K split, by the estimated time in K steps of one CTA:
// waves of co-resident tiles (a split tile runs as a cluster of S CTAs, and
// clusters are placed whole, so the device holds fewer of them at once) times
// the K steps of a split plus, for a split, ~6 K steps of partial-tile
// reduction in every wave.  A 224-wide tile's K step costs ~0.95 of a
// 256-wide one (the step waits on the X tiles, whose size it shares).
// Measured on 2048 x 4096 x 4096, 4096 x 11008 x 4096 and 128..512 x N.
// No split may be left empty.
struct MxPlan {
  int BN, S;
};

template <int F, int BN, bool TWO = true, bool TALL = false, bool A4 = false, bool NV = false>
static cudaError_t set_smem(int dev) {
  static std::atomic<int> done[64];
  if (dev < 0 || dev >= 64 || done[dev].load()) return cudaSuccess;
  cudaError_t e =
      cudaFuncSetAttribute(qgemm_mx_kernel<F, BN, TWO, TALL, A4, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           NV ? SMEM_BYTES_NV : (A4 ? SMEM_BYTES_A4 : SMEM_BYTES));
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(qgemm_mx_kernel<F, BN, TWO, TALL, A4, NV>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1);
  if (e == cudaSuccess) done[dev].store(1);
  return e;
}

// Clusters of S CTAs (of this kernel's shared memory) the device holds at once.
template <int F>
static int cluster_capacity(int dev, int S, int sms) {
  static std::atomic<int> cache[64][5];
  if (S == 1 || dev < 0 || dev >= 64) return sms;
  int v = cache[dev][S].load();
  if (v > 0) return v;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = unsigned(S);
  lc.gridDim = dim3(1, 1, unsigned(S));
  lc.blockDim = dim3(THREADS);
  lc.dynamicSmemBytes = SMEM_BYTES;
  lc.attrs = at;
  lc.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, qgemm_mx_kernel<F, 256>, &lc) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = sms / S;
  }
  cache[dev][S].store(n);
  return n;
}

template <int F>
static MxPlan plan_mx(int dev, int M, int N, int K, int sms) {
  const int nk = K / BK;
  const int64_t mtiles = (M + BM - 1) / BM;
  MxPlan best{256, 1};
  double best_cost = 1e300;
  for (int bn : {256, 224}) {
    const int64_t tiles = int64_t((N + bn - 1) / bn) * mtiles;
    for (int s = 1; s <= 4; ++s) {
      const int per = (nk + s - 1) / s;
      if (s > 1 && (s - 1) * per >= nk) continue;
      const int64_t cap = cluster_capacity<F>(dev, s, sms);
      const int64_t waves = (tiles + cap - 1) / cap;
      const double cost = double(waves) * (per + (s > 1 ? 6.0 : 0.0)) * (bn == 224 ? 0.95 : 1.0);
      if (cost < best_cost - 1e-9) {
        best_cost = cost;
        best = {bn, s};
      }
    }
  }
  return best;
}

template <int F, int BN, bool TWO = true, bool TALL = false, bool A4 = false, bool NV = false>
static cudaError_t launch_tile(const CUtensorMap& mhi, const CUtensorMap& mlo, const CUtensorMap& mw, MxParams prm,
                               int M, int N, int S, cudaStream_t st) {
  const int nk = prm.K / (A4 ? 2 * BK : BK);
  prm.kb_per = (nk + S - 1) / S;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = 1;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = unsigned(S);
  constexpr int TM = TALL ? 2 * BM : BM;
  lc.gridDim = dim3((N + BN - 1) / BN, (M + TM - 1) / TM, S);
  lc.blockDim = dim3(THREADS);
  lc.dynamicSmemBytes = NV ? SMEM_BYTES_NV : (A4 ? SMEM_BYTES_A4 : SMEM_BYTES);
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, qgemm_mx_kernel<F, BN, TWO, TALL, A4, NV>, mhi, mlo, mw, prm);
}

template <int F>
static cudaError_t launch_fmt(const void* codes, const void* scales, const void* x, void* out, bool out_f32, int M,
                              int N, int K, void* ws, cudaStream_t st, int sms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = set_smem<F, 256>(dev)) != cudaSuccess || (e = set_smem<F, 224>(dev)) != cudaSuccess) return e;
  MxPlan pl = plan_mx<F>(dev, M, N, K, sms > 0 ? sms : 1);
  if (g_force_bn.load() == 224 || g_force_bn.load() == 256) pl.BN = g_force_bn.load();
  if (g_force_s.load() >= 1 && g_force_s.load() <= 4 && (g_force_s.load() - 1) * ((K / BK + g_force_s.load() - 1) / g_force_s.load()) < K / BK)
    pl.S = g_force_s.load();
  const WsLayout lay = ws_layout(M, K);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  // activations -> hi / lo MXFP8 terms (one warp per row and 1024 columns)
  {
    const int mpad = (M + BM - 1) / BM * BM;
    const int64_t warps = int64_t(mpad) * ((K / 32 + 31) / 32);
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.gridDim = dim3(unsigned((warps + 7) / 8));
    lc.blockDim = dim3(256);
    lc.stream = st;
    lc.attrs = at;
    lc.numAttrs = 1;
    e = cudaLaunchKernelEx(&lc, xquant_kernel, static_cast<const __nv_bfloat16*>(x), w8, lay, M, K,
                           static_cast<const int*>(nullptr), static_cast<const int*>(nullptr));
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mhi, mlo, mw;
  if (!make_map(enc, &mhi, CU_TENSOR_MAP_DATA_TYPE_UINT8, w8 + lay.hi, K, M, K, BM) ||
      !make_map(enc, &mlo, CU_TENSOR_MAP_DATA_TYPE_UINT8, w8 + lay.lo, K, M, K, BM))
    return cudaErrorInvalidValue;
  const bool ok = F == MXFP4
                      ? make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, codes, K, N, K / 2, uint32_t(pl.BN))
                      : make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K, N, K, uint32_t(pl.BN));
  if (!ok) return cudaErrorInvalidValue;
  MxParams prm{};
  prm.wscales = static_cast<const uint8_t*>(scales);
  prm.sf_hi = w8 + lay.sf_hi;
  prm.sf_lo = w8 + lay.sf_lo;
  prm.out = out;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.out_f32 = out_f32 ? 1 : 0;
  prm.kb_per = K / BK;
  prm.limit_ns = g_limit_ns.load();
  prm.drop_arrivals = g_drop.load();
  if (pl.BN == 224) return launch_tile<F, 224>(mhi, mlo, mw, prm, M, N, pl.S, st);
  return launch_tile<F, 256>(mhi, mlo, mw, prm, M, N, pl.S, st);
}

// The quantized-activation product (both operands block-scaled): X packed to
// MXFP8 E4M3 by the packer's rule into the workspace (codes, then scale
// atoms), then one MMA per block.
inline size_t a8_codes_bytes(int64_t M, int64_t K) { return align1k(size_t(M) * size_t(K)); }
inline size_t a8_workspace_bytes(int64_t M, int64_t K) {
  return a8_codes_bytes(M, K) + align1k(size_t((M + BM - 1) / BM) * size_t(K / BK) * SF_BYTES);
}

template <int F>
static cudaError_t launch_a8(const void* codes, const void* scales, const void* x, void* out, bool out_f32, int M,
                             int N, int K, void* ws, cudaStream_t st, int sms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = set_smem<F, 256>(dev)) != cudaSuccess || (e = set_smem<F, 256, false>(dev)) != cudaSuccess ||
      (e = set_smem<F, 224, false>(dev)) != cudaSuccess)
    return e;
  MxPlan pl = plan_mx<F>(dev, M, N, K, sms > 0 ? sms : 1);
  if (g_force_bn.load() == 224 || g_force_bn.load() == 256) pl.BN = g_force_bn.load();
  if (g_force_s.load() >= 1 && g_force_s.load() <= 4 && (g_force_s.load() - 1) * ((K / BK + g_force_s.load() - 1) / g_force_s.load()) < K / BK)
    pl.S = g_force_s.load();
  // tall tiles (256 x 224, one CTA for two M tiles) without a K split, where
  // they still give every SM a tile
  const int ft = g_force_tall.load();
  const int64_t tall_ctas = int64_t((N + 223) / 224) * ((M + 2 * BM - 1) / (2 * BM));
  const bool tall = ft != 1 && pl.S == 1 && M > BM && (ft == 2 || tall_ctas >= int64_t(sms > 0 ? sms : 1));
  const uint32_t wbox = tall ? 224u : uint32_t(pl.BN);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  if ((e = launch_quantize_e4m3_atoms(x, w8, w8 + a8_codes_bytes(M, K), M, K, st)) != cudaSuccess) return e;
  CUtensorMap mx8, mw;
  if (!make_map(enc, &mx8, CU_TENSOR_MAP_DATA_TYPE_UINT8, w8, K, M, K, BM)) return cudaErrorInvalidValue;
  const bool ok = F == MXFP4 ? make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, codes, K, N, K / 2, wbox)
                             : make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K, N, K, wbox);
  if (!ok) return cudaErrorInvalidValue;
  MxParams prm{};
  prm.wscales = static_cast<const uint8_t*>(scales);
  prm.sf_hi = w8 + a8_codes_bytes(M, K);
  prm.sf_lo = prm.sf_hi;
  prm.out = out;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.out_f32 = out_f32 ? 1 : 0;
  prm.kb_per = K / BK;
  prm.limit_ns = g_limit_ns.load();
  prm.drop_arrivals = g_drop.load();
  if (tall) {
    if ((e = set_smem<F, 224, false, true>(dev)) != cudaSuccess) return e;
    return launch_tile<F, 224, false, true>(mx8, mx8, mw, prm, M, N, 1, st);
  }
  if (pl.BN == 224) return launch_tile<F, 224, false>(mx8, mx8, mw, prm, M, N, pl.S, st);
  return launch_tile<F, 256, false>(mx8, mx8, mw, prm, M, N, pl.S, st);
}

// The all-FP4 product: X packed to MXFP4 by the packer's rule into the
// workspace (codes [M, K/2], then scale atoms), mxfp4 weights, one kind::mxf4
// MMA per 64 K.  Both operand tiles are plain bytes to the copy engine (two
// codes a byte, as stored).  K a multiple of 256 (one step).
inline size_t a4_codes_bytes(int64_t M, int64_t K) { return align1k(size_t(M) * size_t(K / 2)); }
inline size_t a4_workspace_bytes(int64_t M, int64_t K) {
  return a4_codes_bytes(M, K) + align1k(size_t((M + BM - 1) / BM) * size_t(K / BK) * SF_BYTES);
}
// nvfp4: codes, scale atoms of 64 K each, then the quantizer's partial maxima
// and, in the last word of that part, the activation's global.
inline size_t nv_atoms_bytes(int64_t M, int64_t K) {
  return align1k(size_t((M + BM - 1) / BM) * size_t(K / 64) * SF_BYTES);
}
inline size_t nv_global_offset(int64_t M, int64_t K) {
  return a4_codes_bytes(M, K) + nv_atoms_bytes(M, K) + 4 * 1024;
}
inline size_t nv_workspace_bytes(int64_t M, int64_t K) {
  return a4_codes_bytes(M, K) + nv_atoms_bytes(M, K) + align1k(4 * 1025);
}

static cudaError_t launch_a4(const void* codes, const void* scales, const void* x, void* out, bool out_f32, int M,
                             int N, int K, void* ws, cudaStream_t st, int sms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = set_smem<MXFP4, 256, false, false, true>(dev)) != cudaSuccess ||
      (e = set_smem<MXFP4, 224, false, false, true>(dev)) != cudaSuccess)
    return e;
  // the planner counts K steps: an A4 step holds 256 codes, an 8-bit one 128
  const int nk = K / (2 * BK);
  MxPlan pl = plan_mx<MXFP4>(dev, M, N, K / 2, sms > 0 ? sms : 1);
  if (g_force_bn.load() == 224 || g_force_bn.load() == 256) pl.BN = g_force_bn.load();
  const int fs = g_force_s.load();
  if (fs >= 1 && fs <= 4 && (fs - 1) * ((nk + fs - 1) / fs) < nk) pl.S = fs;
  const int ft = g_force_tall.load();
  const int64_t tall_ctas = int64_t((N + 223) / 224) * ((M + 2 * BM - 1) / (2 * BM));
  const bool tall = ft != 1 && pl.S == 1 && M > BM && (ft == 2 || tall_ctas >= int64_t(sms > 0 ? sms : 1));
  const uint32_t wbox = tall ? 224u : uint32_t(pl.BN);
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  if ((e = launch_quantize_mxfp4_atoms(x, w8, w8 + a4_codes_bytes(M, K), M, K, st)) != cudaSuccess) return e;
  CUtensorMap mx4, mw;
  if (!make_map(enc, &mx4, CU_TENSOR_MAP_DATA_TYPE_UINT8, w8, K / 2, M, K / 2, BM) ||
      !make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K / 2, N, K / 2, wbox))
    return cudaErrorInvalidValue;
  MxParams prm{};
  prm.wscales = static_cast<const uint8_t*>(scales);
  prm.sf_hi = w8 + a4_codes_bytes(M, K);
  prm.sf_lo = prm.sf_hi;
  prm.out = out;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.out_f32 = out_f32 ? 1 : 0;
  prm.kb_per = nk;
  prm.limit_ns = g_limit_ns.load();
  prm.drop_arrivals = g_drop.load();
  if (tall) {
    if ((e = set_smem<MXFP4, 224, false, true, true>(dev)) != cudaSuccess) return e;
    return launch_tile<MXFP4, 224, false, true, true>(mx4, mx4, mw, prm, M, N, 1, st);
  }
  if (pl.BN == 224) return launch_tile<MXFP4, 224, false, false, true>(mx4, mx4, mw, prm, M, N, pl.S, st);
  return launch_tile<MXFP4, 256, false, false, true>(mx4, mx4, mw, prm, M, N, pl.S, st);
}

// The all-FP4 product over nvfp4 weights: X packed to NVFP4 (the packer's
// rule over the whole X: two kernels, the amax then the codes), single tiles.
static cudaError_t launch_a4_nv(const void* codes, const void* scales, float gw, const void* x, void* out,
                                bool out_f32, int M, int N, int K, void* ws, cudaStream_t st, int sms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = set_smem<NVFP4, 256, false, false, true, true>(dev)) != cudaSuccess ||
      (e = set_smem<NVFP4, 224, false, false, true, true>(dev)) != cudaSuccess)
    return e;
  const int nk = K / (2 * BK);
  MxPlan pl = plan_mx<MXFP4>(dev, M, N, K / 2, sms > 0 ? sms : 1);
  if (g_force_bn.load() == 224 || g_force_bn.load() == 256) pl.BN = g_force_bn.load();
  const int fs = g_force_s.load();
  if (fs >= 1 && fs <= 4 && (fs - 1) * ((nk + fs - 1) / fs) < nk) pl.S = fs;
  // tall tiles (one scale slot, see the kernel) where they still give every SM a tile
  const int ft = g_force_tall.load();
  const int64_t tall_ctas = int64_t((N + 223) / 224) * ((M + 2 * BM - 1) / (2 * BM));
  const bool tall = ft != 1 && pl.S == 1 && M > BM && (ft == 2 || tall_ctas >= int64_t(sms > 0 ? sms : 1));
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  uint8_t* atoms = w8 + a4_codes_bytes(M, K);
  float* partials = reinterpret_cast<float*>(atoms + nv_atoms_bytes(M, K));
  float* gx = reinterpret_cast<float*>(w8 + nv_global_offset(M, K));
  if ((e = launch_quantize_nvfp4_atoms(x, w8, atoms, partials, gx, M, K, st)) != cudaSuccess) return e;
  CUtensorMap mx4, mw;
  if (!make_map(enc, &mx4, CU_TENSOR_MAP_DATA_TYPE_UINT8, w8, K / 2, M, K / 2, BM) ||
      !make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K / 2, N, K / 2, tall ? 224u : uint32_t(pl.BN)))
    return cudaErrorInvalidValue;
  MxParams prm{};
  prm.wscales = static_cast<const uint8_t*>(scales);
  prm.sf_hi = atoms;
  prm.sf_lo = atoms;
  prm.out = out;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.out_f32 = out_f32 ? 1 : 0;
  prm.kb_per = nk;
  prm.limit_ns = g_limit_ns.load();
  prm.drop_arrivals = g_drop.load();
  prm.gw = gw;
  prm.gx = gx;
  if (tall) {
    if ((e = set_smem<NVFP4, 224, false, true, true, true>(dev)) != cudaSuccess) return e;
    return launch_tile<NVFP4, 224, false, true, true, true>(mx4, mx4, mw, prm, M, N, 1, st);
  }
  if (pl.BN == 224) return launch_tile<NVFP4, 224, false, false, true, true>(mx4, mx4, mw, prm, M, N, pl.S, st);
  return launch_tile<NVFP4, 256, false, false, true, true>(mx4, mx4, mw, prm, M, N, pl.S, st);
}

// ------------------------------------------------- expert-grouped rows ---
//
// MoE rows routed to one expert run through the GEMM together (rlx-cpu
// thunk/ops/quant.rs lowp_scaled_grouped_matmul; metaltile PR #250's MoE
// gather-qmm): a routing kernel buckets the rows by expert into segments of
// whole 128-row tiles (route_off[e] .. route_off[e + 1], padding rows -1 in
// row_of), the activation split reads its rows through row_of, and each GEMM
// tile takes its expert's weight rows, so every expert's weights stream
// once per 128 rows routed to it.

// One CTA: counts per expert, 128-aligned segment offsets, then each row's
// slot (rows keep no particular order inside a segment: each output row is
// computed on its own).  A row whose expert index lies outside [0, E) gets a
// zero output row and status bit 2.
__global__ void __launch_bounds__(1024) route_kernel(const int32_t* __restrict__ idx, int M, int E,
                                                     int* __restrict__ off, int* __restrict__ row_of,
                                                     void* __restrict__ out, int N, int out_f32) {
  extern __shared__ int sh[];
  int* cnt = sh;
  int* cur = sh + E;
  int* poff = sh + 2 * E;            // E + 1
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the router may be the preceding kernel
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = cur[e] = 0;
  __syncthreads();
  for (int r = tid; r < M; r += blockDim.x) {
    const int e = __ldg(idx + r);
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);
    } else {
      atomicOr(&g_mx_status, 2u);
      for (int n = 0; n < N; ++n) {
        if (out_f32) static_cast<float*>(out)[int64_t(r) * N + n] = 0.0f;
        else static_cast<__nv_bfloat16*>(out)[int64_t(r) * N + n] = __float2bfloat16_rn(0.0f);
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    int p = 0;
    for (int e = 0; e < E; ++e) {
      poff[e] = p;
      p += (cnt[e] + BM - 1) / BM * BM;
    }
    poff[E] = p;
  }
  __syncthreads();
  for (int e = tid; e <= E; e += blockDim.x) off[e] = poff[e];
  for (int m = tid; m < poff[E]; m += blockDim.x) row_of[m] = -1;
  __syncthreads();
  for (int r = tid; r < M; r += blockDim.x) {
    const int e = __ldg(idx + r);
    if (e >= 0 && e < E) row_of[poff[e] + atomicAdd(&cur[e], 1)] = r;
  }
}

constexpr int ROUTE_MAX_E = 1024;

// Workspace rows: every segment rounded up to whole 128-row tiles.
inline int64_t grouped_rows(int64_t M, int64_t E) { return (M + 127 * std::min<int64_t>(E, M) + BM - 1) / BM * BM; }

struct GroupedLayout {
  size_t off, row_of, total;
  WsLayout x;     // relative to `base`
  size_t base;
};
inline GroupedLayout grouped_layout(int64_t M, int64_t K, int64_t E) {
  GroupedLayout g;
  const int64_t R = grouped_rows(M, E);
  g.off = 0;
  g.row_of = align1k(size_t(E + 1) * 4);
  g.base = g.row_of + align1k(size_t(R) * 4);
  g.x = ws_layout(R, K);
  g.total = g.base + g.x.total;
  return g;
}

template <int F>
static cudaError_t launch_grouped(const void* codes, const void* scales, const void* x, const int32_t* idx, void* out,
                                  bool out_f32, int M, int N, int K, int E, void* ws, cudaStream_t st, int sms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = set_smem<F, 256>(dev)) != cudaSuccess || (e = set_smem<F, 224>(dev)) != cudaSuccess) return e;
  const GroupedLayout gl = grouped_layout(M, K, E);
  const int R = int(grouped_rows(M, E));
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  int* off = reinterpret_cast<int*>(w8 + gl.off);
  int* row_of = reinterpret_cast<int*>(w8 + gl.row_of);
  uint8_t* xb = w8 + gl.base;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  {
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(1);
    lc.blockDim = dim3(1024);
    lc.dynamicSmemBytes = size_t(3 * E + 1) * sizeof(int);
    lc.stream = st;
    lc.attrs = pdl;
    lc.numAttrs = 1;
    e = cudaLaunchKernelEx(&lc, route_kernel, idx, M, E, off, row_of, out, N, int(out_f32));
    if (e != cudaSuccess) return e;
  }
  {
    const int64_t warps = int64_t(R) * ((K / 32 + 31) / 32);
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(unsigned((warps + 7) / 8));
    lc.blockDim = dim3(256);
    lc.stream = st;
    lc.attrs = pdl;
    lc.numAttrs = 1;
    e = cudaLaunchKernelEx(&lc, xquant_kernel, static_cast<const __nv_bfloat16*>(x), xb, gl.x, R, K,
                           static_cast<const int*>(row_of), static_cast<const int*>(off + E));
    if (e != cudaSuccess) return e;
  }
  const MxPlan pl = plan_mx<F>(dev, R, N, K, sms > 0 ? sms : 1);
  CUtensorMap mhi, mlo, mw;
  if (!make_map(enc, &mhi, CU_TENSOR_MAP_DATA_TYPE_UINT8, xb + gl.x.hi, K, R, K, BM) ||
      !make_map(enc, &mlo, CU_TENSOR_MAP_DATA_TYPE_UINT8, xb + gl.x.lo, K, R, K, BM))
    return cudaErrorInvalidValue;
  const int64_t wrows = int64_t(E) * N;
  const bool ok = F == MXFP4
                      ? make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, codes, K, wrows, K / 2, uint32_t(pl.BN))
                      : make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K, wrows, K, uint32_t(pl.BN));
  if (!ok) return cudaErrorInvalidValue;
  MxParams prm{};
  prm.wscales = static_cast<const uint8_t*>(scales);
  prm.sf_hi = xb + gl.x.sf_hi;
  prm.sf_lo = xb + gl.x.sf_lo;
  prm.out = out;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.out_f32 = out_f32 ? 1 : 0;
  prm.kb_per = K / BK;
  prm.limit_ns = g_limit_ns.load();
  prm.drop_arrivals = g_drop.load();
  prm.route_off = off;
  prm.row_of = row_of;
  prm.E = E;
  // the grid covers R rows of tiles; the tiles past the routed segments leave at once
  if (pl.BN == 224) return launch_tile<F, 224>(mhi, mlo, mw, prm, R, N, pl.S, st);
  return launch_tile<F, 256>(mhi, mlo, mw, prm, R, N, pl.S, st);
}

// ------------------------------------------------ decode GEMV, M <= 16 ---
//
// The same block-scaled MMA with the roles set for a decode step: A = a tile
// of 128 weight rows over KC columns (TMA-loaded as stored before the
// dependent wait, like every weight read here), B = the activations split
// in the CTA into hi and lo E4M3 rows (row 2m = hi of activation row m, row
// 2m + 1 its lo; the MMA's N is 16 for M <= 8, 32 for M <= 16), D = 128 x N
// float32 in tensor memory, out[m][n] = D[n][2m] + D[n][2m + 1].  Nothing is
// decoded on the ALUs.  K may be split over a cluster of S CTAs (KC = K / S <=
// 512); the partial columns meet through distributed shared memory.
constexpr int GV_THREADS = 128, GV_ROWS = 128, GV_KC_MAX = 512;
constexpr int GV_SLABS = GV_KC_MAX / BK;                    // 128-column slabs per CTA, at most
constexpr int GV_W_BYTES = GV_SLABS * GV_ROWS * BK;        // 64 KiB
constexpr int GV_X_BYTES = GV_SLABS * 32 * BK;             // 16 KiB (N up to 32)
constexpr int GV_SMEM = 1024 + GV_W_BYTES + GV_X_BYTES + 2 * GV_SLABS * SF_BYTES + 128;
constexpr int GV_TMEM_COLS = 64;                           // D 0-31, W scales 32-47, X scales 48-63

struct GvParams {
  const uint8_t* wscales;        // [N, K/32] E8M0
  const __nv_bfloat16* x;        // [M, K]
  void* out;                     // [M, N]
  int M, N, K, KC;
  int out_f32;
  uint64_t limit_ns;
};

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

template <int F, int NP>
__global__ void __launch_bounds__(GV_THREADS) qgemv_mx_kernel(const __grid_constant__ CUtensorMap w_map,
                                                              const GvParams p) {
  static_assert(NP == 16 || NP == 32, "the MMA's N: two rows per activation row");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* wt = smem;                                     // [slab][128 rows x 128 B], 128B-swizzled
  uint8_t* xt = wt + GV_W_BYTES;                          // [slab][NP rows x 128 B], 128B-swizzled
  uint8_t* sfa = xt + GV_X_BYTES;                         // [slab] W scale atoms
  uint8_t* sfb = sfa + GV_SLABS * SF_BYTES;               // [slab] X scale atoms
  uint64_t* bars = reinterpret_cast<uint64_t*>(sfb + GV_SLABS * SF_BYTES);   // [0]: W landed, [1]: MMAs done
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 2);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  float* part = reinterpret_cast<float*>(wt);             // [128][17] partial sums (the drained W tile)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = gridDim.x, split = blockIdx.x;            // K split = the cluster along x
  const int n0 = blockIdx.y * GV_ROWS, k0 = split * p.KC;
  const int nsl = p.KC / BK;
  const uint32_t w_bar = smem_u32(bars), done_bar = w_bar + 8u;
  auto fail = [&]() {
    *abort_flag = 1u;
    atomicOr(&g_mx_status, 1u);
  };

  if (tid == 0) {
    mbar_init(w_bar, 1);
    mbar_init(done_bar, 1);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&w_map)) : "memory");
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32((const void*)tmem_slot)),
                 "r"(GV_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- the weights (not the preceding kernel's output): before the wait ---
  if (tid == 0) {
    mbar_arrive_expect_tx(w_bar, uint32_t(nsl) * (F == MXFP4 ? GV_ROWS * BK / 2 : GV_ROWS * BK));
    for (int j = 0; j < nsl; ++j) tma_load_2d(smem_u32(wt + j * GV_ROWS * BK), &w_map, k0 + j * BK, n0, w_bar);
  }
  {
    // row tid's E8M0 scales: one 32-bit word = 4 blocks of a slab
    const int n = n0 + tid;
    const uint32_t* ws32 = reinterpret_cast<const uint32_t*>(p.wscales) + int64_t(n) * (p.K / 128) + k0 / 128;
    for (int j = 0; j < nsl; ++j) {
      const uint32_t v = n < p.N ? __ldg(ws32 + j) : 0u;
      *reinterpret_cast<uint32_t*>(sfa + j * SF_BYTES + umma::sf_atom_offset(uint32_t(tid), 0)) = v;
    }
  }

  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- the activations: split into hi / lo E4M3 rows of the B tile ----------
  {
    const int bps = p.KC / 32;                                  // blocks per row in this split
    for (int task = tid; task < p.M * bps; task += GV_THREADS) {
      const int m = task / bps, b = task - m * bps;
      uint32_t w[16], hi[8], lo[8], c1, c2;
      load_block(p.x + int64_t(m) * p.K + k0 + 32 * b, w);
      split_block(w, c1, c2, hi, lo);
      const int j = b >> 2, c = (b & 3) * 2;                    // slab, first 16-byte chunk of the 128-byte row
      uint8_t* slab = xt + j * NP * BK;
      const int rh = 2 * m, rl = 2 * m + 1;
      *reinterpret_cast<uint4*>(slab + tc::sw128_off(rh, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(slab + tc::sw128_off(rh, c + 1)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
      *reinterpret_cast<uint4*>(slab + tc::sw128_off(rl, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4*>(slab + tc::sw128_off(rl, c + 1)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
      sfb[j * SF_BYTES + umma::sf_atom_offset(uint32_t(rh), uint32_t(b & 3))] = uint8_t(c1);
      sfb[j * SF_BYTES + umma::sf_atom_offset(uint32_t(rl), uint32_t(b & 3))] = uint8_t(c2);
    }
  }
  fence_proxy_async();                                          // generic stores -> tensor-core reads
  __syncthreads();

  if (warp == 0) {
    // the converged warp waits (lane 0) and one elected lane issues
    int wok = 1;
    if (lane == 0) wok = mbar_wait(w_bar, 0, p.limit_ns);
    wok = __shfl_sync(0xFFFFFFFFu, wok, 0);
    const bool leader = elect_one();
    if (!wok) {
      if (leader) fail();
    } else {
      tc_fence_after();
      if (leader) {
        for (int j = 0; j < nsl; ++j) {
          tmem_cp_sf(tmem + 32u + 4u * j, umma::smem_desc_sf32x16(smem_u32(sfa + j * SF_BYTES)));
          tmem_cp_sf(tmem + 48u + 4u * j, umma::smem_desc_sf32x16(smem_u32(sfb + j * SF_BYTES)));
        }
        for (int j = 0; j < nsl; ++j) {
          const uint64_t da = desc_sw128(smem_u32(wt + j * GV_ROWS * BK)), db = desc_sw128(smem_u32(xt + j * NP * BK));
          #pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk) {
            const uint32_t id =
                umma::idesc_mxf8f6f4(b_type<F>(), umma::F8F6F4_E4M3, GV_ROWS, NP, uint32_t(kk), uint32_t(kk));
            mma_mx(tmem, da + uint64_t(2 * kk), db + uint64_t(2 * kk), id, tmem + 32u + 4u * j, tmem + 48u + 4u * j,
                   (j | kk) != 0);
          }
        }
      }
      __syncwarp();
    }
    if (leader) mma_commit(done_bar);   // fires once the MMAs above (if any) have completed
  }

  // ---- drain: row 32 warp + lane of the tile ---------------------------------
  int ok = 1;
  if (lane == 0) ok = mbar_wait(done_bar, 0, p.limit_ns);
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  if (!ok && lane == 0) fail();
  tc_fence_after();
  float v[16];
  {
    uint32_t r[NP];
    if constexpr (NP == 16) tmem_ld16(tmem + (uint32_t(warp * 32) << 16), r);
    else tmem_ld32(tmem + (uint32_t(warp * 32) << 16), r);
    #pragma unroll
    for (int m = 0; m < NP / 2; ++m) v[m] = __uint_as_float(r[2 * m]) + __uint_as_float(r[2 * m + 1]);
  }
  const int row = tid;
  auto store = [&](int m, int n, float val) {
    if (p.out_f32) static_cast<float*>(p.out)[int64_t(m) * p.N + n] = val;
    else static_cast<__nv_bfloat16*>(p.out)[int64_t(m) * p.N + n] = __float2bfloat16_rn(val);
  };
  if (S == 1) {
    if (ok && *abort_flag == 0u && n0 + row < p.N) {
      #pragma unroll
      for (int m = 0; m < NP / 2; ++m)
        if (m < p.M) store(m, n0 + row, v[m]);
    }
  } else {
    #pragma unroll
    for (int m = 0; m < NP / 2; ++m) part[row * 17 + m] = v[m];
    cluster_sync();
    uint32_t any_abort = 0u;
    for (int q = 0; q < S; ++q) any_abort |= ld_cluster_u32(smem_u32((const void*)abort_flag), uint32_t(q));
    // this CTA sums rows [split * 128 / S, (split + 1) * 128 / S) over the cluster's partials, in rank order
    const int r0 = split * GV_ROWS / S, r1 = (split + 1) * GV_ROWS / S;
    if (!any_abort) {
      for (int e = tid; e < (r1 - r0) * p.M; e += GV_THREADS) {   // consecutive threads: consecutive outputs
        const int m = e / (r1 - r0), rr = r0 + e - m * (r1 - r0);
        if (n0 + rr >= p.N) continue;
        float sum = 0.0f;
        for (int q = 0; q < S; ++q)
          sum += __uint_as_float(ld_cluster_u32(smem_u32(part + rr * 17 + m), uint32_t(q)));
        store(m, n0 + rr, sum);
      }
    }
    cluster_sync();   // no CTA leaves while the others still read its partials
  }

  // a CTA that gave up waiting for its weight tile still lets the copy land before it exits
  if (tid == 0 && *abort_flag) mbar_wait(w_bar, 0, p.limit_ns);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(GV_TMEM_COLS) : "memory");
  }
}

// K split for the decode GEMV: one CTA per 128 rows up to K = 512, a pair of
// CTAs up to K = 1024; 0 (the mma.sync decode GEMVs) beyond, except for 3 to
// 16 activation rows where a split into 512-column slabs gives a grid 1.5-2
// CTAs deep on every SM (two fit an SM).  Measured against the CUDA-core
// GEMVs (mxfp4 / mxfp8 E4M3, M = 1 and 8): 1.6-4x faster at K <= 1024.  At
// K = 4096, M = 1, an 8-way split runs 6.5 us against 3.4 us (N = 4096): 256
// CTAs of two per SM leave most of a launch unable to start, and so to
// request its weights, before the preceding launch ends, and the split's
// cluster reduction adds ~2 us; for M = 3-16 the same split at N = K = 4096
// runs 0.73-0.84x the batch GEMV (mxfp4, mxfp8 E4M3 / E5M2), while at 128 or
// 384 CTAs (N = 2048 or 6144, or K = 2048) it measured 0.91-1.26x.
inline int gemv_plan(int M, int64_t N, int K, int sms) {
  if (K <= 0 || K % BK) return 0;
  const int slabs = K / BK;
  const int fs = g_gemv_s.load();   // a forced split (measurements)
  if (fs >= 1 && fs <= 8 && slabs % fs == 0 && slabs / fs <= GV_SLABS) return fs;
  if (slabs <= GV_SLABS) return 1;
  if (slabs <= 2 * GV_SLABS && slabs % 2 == 0) return 2;
  if (M >= 3 && slabs % GV_SLABS == 0 && slabs / GV_SLABS <= 8) {
    const int S = slabs / GV_SLABS;
    const int64_t ctas = (N + GV_ROWS - 1) / GV_ROWS * S;
    if (2 * ctas >= 3 * int64_t(sms) && ctas <= 2 * int64_t(sms)) return S;
  }
  return 0;
}

template <int F, int NP>
static cudaError_t launch_gemv_np(const void* codes, const void* scales, const void* x, void* out, bool out_f32, int M,
                                  int N, int K, cudaStream_t st, int sms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  static std::atomic<int> done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !done[dev].load()) {
    e = cudaFuncSetAttribute(qgemv_mx_kernel<F, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, GV_SMEM);
    if (e != cudaSuccess) return e;
    done[dev].store(1);
  }
  const int S = gemv_plan(M, N, K, sms);
  if (S == 0) return cudaErrorInvalidValue;
  CUtensorMap mw;
  const bool ok = F == MXFP4 ? make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, codes, K, N, K / 2, GV_ROWS)
                             : make_map(enc, &mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K, N, K, GV_ROWS);
  if (!ok) return cudaErrorInvalidValue;
  GvParams prm;
  prm.wscales = static_cast<const uint8_t*>(scales);
  prm.x = static_cast<const __nv_bfloat16*>(x);
  prm.out = out;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.KC = K / S;
  prm.out_f32 = out_f32 ? 1 : 0;
  prm.limit_ns = g_limit_ns.load();
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = unsigned(S);
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = 1;
  lc.gridDim = dim3(unsigned(S), unsigned((N + GV_ROWS - 1) / GV_ROWS));
  lc.blockDim = dim3(GV_THREADS);
  lc.dynamicSmemBytes = GV_SMEM;
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, qgemv_mx_kernel<F, NP>, mw, prm);
}

template <int F>
static cudaError_t launch_gemv(const void* codes, const void* scales, const void* x, void* out, bool out_f32, int M,
                               int N, int K, cudaStream_t st, int sms) {
  if (M <= 8) return launch_gemv_np<F, 16>(codes, scales, x, out, out_f32, M, N, K, st, sms);
  return launch_gemv_np<F, 32>(codes, scales, x, out, out_f32, M, N, K, st, sms);
}

}  // namespace mx

bool qgemm_mx_supported(int fmt, int64_t M, int64_t K) {
  return (fmt == MXFP4 || fmt == MXFP8_E4M3 || fmt == MXFP8_E5M2) && M > 16 && K > 0 && K % mx::BK == 0;
}

size_t qgemm_mx_workspace_bytes(int64_t M, int64_t K) { return mx::ws_layout(M, K).total; }

cudaError_t launch_qgemm_mx(int fmt, const void* codes, const void* scales, const void* x, void* out, bool out_f32,
                            int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st, int sms) {
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return mx::launch_fmt<MXFP4>(codes, scales, x, out, out_f32, m, n, k, workspace, st, sms);
    case MXFP8_E4M3: return mx::launch_fmt<MXFP8_E4M3>(codes, scales, x, out, out_f32, m, n, k, workspace, st, sms);
    case MXFP8_E5M2: return mx::launch_fmt<MXFP8_E5M2>(codes, scales, x, out, out_f32, m, n, k, workspace, st, sms);
    default: return cudaErrorInvalidValue;
  }
}

bool qgemv_mx_supported(int fmt, int64_t M, int64_t N, int64_t K, const void* codes, int sms) {
  return !mx::g_gemv_off.load() && (fmt == MXFP4 || fmt == MXFP8_E4M3 || fmt == MXFP8_E5M2) && M >= 1 && M <= 16 &&
         N <= 65535LL * mx::GV_ROWS && K <= (int64_t(1) << 20) && mx::gemv_plan(int(M), N, int(K), sms) > 0 &&
         !(fmt == MXFP4 && (reinterpret_cast<uintptr_t>(codes) & 31u));
}

cudaError_t launch_qgemv_mx(int fmt, const void* codes, const void* scales, const void* x, void* out, bool out_f32,
                            int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms) {
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return mx::launch_gemv<MXFP4>(codes, scales, x, out, out_f32, m, n, k, st, sms);
    case MXFP8_E4M3: return mx::launch_gemv<MXFP8_E4M3>(codes, scales, x, out, out_f32, m, n, k, st, sms);
    case MXFP8_E5M2: return mx::launch_gemv<MXFP8_E5M2>(codes, scales, x, out, out_f32, m, n, k, st, sms);
    default: return cudaErrorInvalidValue;
  }
}

size_t qgemm_a8_workspace_bytes(int64_t M, int64_t K) { return mx::a8_workspace_bytes(M, K); }

cudaError_t launch_qgemm_a8(int fmt, const void* codes, const void* scales, const void* x, void* out, bool out_f32,
                            int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st, int sms) {
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return mx::launch_a8<MXFP4>(codes, scales, x, out, out_f32, m, n, k, workspace, st, sms);
    case MXFP8_E4M3: return mx::launch_a8<MXFP8_E4M3>(codes, scales, x, out, out_f32, m, n, k, workspace, st, sms);
    case MXFP8_E5M2: return mx::launch_a8<MXFP8_E5M2>(codes, scales, x, out, out_f32, m, n, k, workspace, st, sms);
    default: return cudaErrorInvalidValue;
  }
}

size_t qgemm_a4_workspace_bytes(int fmt, int64_t M, int64_t K) {
  return fmt == NVFP4 ? mx::nv_workspace_bytes(M, K) : mx::a4_workspace_bytes(M, K);
}

cudaError_t launch_qgemm_a4(int fmt, const void* codes, const void* scales, float global_scale, const void* x,
                            void* out, bool out_f32, int64_t M, int64_t N, int64_t K, void* workspace, cudaStream_t st,
                            int sms) {
  if (fmt == NVFP4)
    return mx::launch_a4_nv(codes, scales, global_scale, x, out, out_f32, int(M), int(N), int(K), workspace, st, sms);
  if (fmt != MXFP4) return cudaErrorInvalidValue;
  return mx::launch_a4(codes, scales, x, out, out_f32, int(M), int(N), int(K), workspace, st, sms);
}

size_t qgemm_grouped_workspace_bytes(int64_t M, int64_t K, int64_t E) { return mx::grouped_layout(M, K, E).total; }
int qgemm_grouped_max_experts() { return mx::ROUTE_MAX_E; }

cudaError_t launch_qgemm_grouped(int fmt, const void* codes, const void* scales, const void* x, const int32_t* idx,
                                 void* out, bool out_f32, int64_t M, int64_t N, int64_t K, int64_t E, void* workspace,
                                 cudaStream_t st, int sms) {
  const int m = int(M), n = int(N), k = int(K), e = int(E);
  switch (fmt) {
    case MXFP4: return mx::launch_grouped<MXFP4>(codes, scales, x, idx, out, out_f32, m, n, k, e, workspace, st, sms);
    case MXFP8_E4M3:
      return mx::launch_grouped<MXFP8_E4M3>(codes, scales, x, idx, out, out_f32, m, n, k, e, workspace, st, sms);
    case MXFP8_E5M2:
      return mx::launch_grouped<MXFP8_E5M2>(codes, scales, x, idx, out, out_f32, m, n, k, e, workspace, st, sms);
    default: return cudaErrorInvalidValue;
  }
}

void set_mx_wait_limit_ns(uint64_t ns) { mx::g_limit_ns.store(ns); }
void set_mx_gemv(int off, int s) {
  mx::g_gemv_off.store(off);
  mx::g_gemv_s.store(s);
}
void set_mx_plan(int bn, int s) {
  mx::g_force_bn.store(bn);
  mx::g_force_s.store(s);
}
void set_mx_drop_arrivals(int on) { mx::g_drop.store(on); }
void set_mx_tall(int v) { mx::g_force_tall.store(v); }

cudaError_t read_and_clear_mx_status(unsigned int* status) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_mx_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_mx_status, &zero, sizeof(unsigned int));
}

}  // namespace qfmt_dev
