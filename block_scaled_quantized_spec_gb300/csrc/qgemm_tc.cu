// Prefill dequantizing GEMM on the 5th-generation tensor cores, M > 16:
//   out[M, N] = X[M, K] (bf16) . dequant(W[N, K])^T, float32 accumulation.
//
// The pages' prefill kernels (metaltile-std src/mlx/fp_quantized_mma.rs,
// mt_fp4_qmm_mma / mt_fp8_e4m3_qmm_mma; the PR #250 block-scaled *_qmm_mma
// kernels) stage X and W tiles in threadgroup memory, decode W per lane into
// threadgroup memory and run 8x8 simdgroup MMAs.  The GB300 design keeps the
// idea -- decode the weights once per tile into on-chip memory, then run dense
// MMAs -- and maps it onto tcgen05:
//
//  * CTA tile 128 (M) x 256 (N), K step 64, four pipeline stages in shared
//    memory (X tile 16 KiB + decoded W tile 32 KiB per stage); nvfp8 and int4
//    affine use a 128 x 128 tile whose weights are hi + lo bf16 pairs;
//  * warp 0: one thread issues TMA loads of the X tile (128B-swizzled, K-major)
//    and owns the TMEM allocation;
//  * warp 1: one thread issues tcgen05.mma kind::f16 (bf16 x bf16 -> float32 in
//    TMEM, 128 x 256 x 16 per instruction) and commits each stage back to the
//    producers through an mbarrier;
//  * warps 2 and up: decoders (16 warps; 8 for nvfp8 and int4 affine).  Each
//    streams 16-byte pieces of codes (plus their block scales) from global
//    memory with 128-bit loads three K steps ahead,
//    decodes them in registers to bf16 with the block scale applied (exact for
//    power-of-two and E4M3 scales; nvfp8 and int4-affine weights become
//    float32 then a hi + lo bf16 pair, two MMAs per K slice) and writes the
//    canonical 128B-swizzled K-major layout the MMA reads;
//  * warps 2-5 (one per TMEM lane quadrant, per 128-row accumulator) then drain
//    the accumulator with tcgen05.ld, apply the nvfp4 global scale and store
//    bf16/float32 rows; 128-row tiles may split K over a cluster (when the
//    tiles alone leave SMs idle), the partial tiles then summed through
//    distributed shared memory;
//  * the launch is programmatic-dependent: weight codes stream in while the
//    preceding kernel finishes, X is read and `out` written only after
//    griddepcontrol.wait.
//
// Every mbarrier wait is bounded by a time limit; on expiry the kernel records
// an error in a device status word, lets in-flight copies and MMAs finish,
// frees its TMEM and exits (qfmt_device_status reports it).
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <type_traits>
#include <mutex>

#include "decode.cuh"
#include "kernels.h"
#include "tcgen05.cuh"

namespace qfmt_dev {

__device__ unsigned int g_device_status;

namespace tc {

constexpr int BM = 128, BK = 64;          // one MMA covers 128 rows of X
constexpr int B_BYTES = 256 * BK * 2;     // 32 KiB: 256 bf16 rows, or 128 hi rows + 128 lo rows
// Decoder warps per CTA: 16 (two pieces or one per thread and K step) for the
// formats exact in bf16; 8 for nvfp8 and int4 affine, whose hi + lo tiles were
// measured faster with eight.
template <int F> struct Dec {
  static constexpr int WARPS = (is_i4<F>() || is_fs8<F>() || is_fp4f<F>()) ? 8 : 16;
  static constexpr int THREADS = WARPS * 32;
  static constexpr int CTA_THREADS = (2 + WARPS) * 32;
};

// MT 128-row sub-tiles of X share each decoded weight tile: MT = 2 halves the
// decode work per FLOP (two accumulators, all 512 TMEM columns at BN = 256).
template <int MT> struct Pipe {
  static constexpr int A_BYTES = MT * BM * BK * 2;            // 16 or 32 KiB
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;       // 48 or 64 KiB
  static constexpr int STAGES = MT == 2 ? 3 : 4;
  static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 256;
};

// Formats whose weights are exact in bf16 use a 128 x 256 tile; nvfp8 and int4
// affine carry each weight as a hi + lo bf16 pair (two MMAs per K slice into
// one accumulator) on a 128 x 128 tile, so a stage holds the same bytes.
template <int F> struct Tile {
  static constexpr bool split = is_fs8<F>() || is_i4<F>() || is_fp4f<F>();
  static constexpr int BN = split ? 128 : 256;
};

struct Params {
  const uint8_t* codes;
  const uint8_t* scales;
  void* out;
  float glob;
  int M, N, K;
  int out_f32;
  int kb_per;          // K steps per split (grid z = the splits of one cluster)
  uint64_t limit_ns;   // bound on every wait
  int drop_arrivals;   // test hook: decoders never signal a stage (the waits must expire)
  int mfast;           // tile order: blockIdx.x the M tile, y the N tile (else x = N tile, y = M tile)
};

// The codes a decoder thread holds for one piece: 16 bytes of one row, or for
// mxfp4x2 the 16 bytes of each residual plane of one output row.
struct PiecePair {
  uint4 a, b;
};
template <int F>
using PieceCodes = std::conditional_t<F == MXFP4X2, PiecePair, uint4>;

template <int F, int MT, int BN = Tile<F>::BN>
__global__ void __launch_bounds__(Dec<F>::CTA_THREADS, 1) qgemm_tc_kernel(const __grid_constant__ CUtensorMap xmap,
                                                                          const Params p) {
  constexpr int DEC_WARPS = Dec<F>::WARPS, DEC_THREADS = Dec<F>::THREADS, THREADS = Dec<F>::CTA_THREADS;
  using T = FmtTraits<F>;
  constexpr bool SPLIT = Tile<F>::split;
  // accumulator columns: BN rounded up to a power of two (BN = 224 fills a
  // 152-SM wave where 256 leaves SMs idle), the allocation a power of two
  constexpr int ACC = BN > 128 ? 256 : BN;
  constexpr int TMEM_COLS = ACC * MT;
  constexpr int STAGES = Pipe<MT>::STAGES, STAGE_BYTES = Pipe<MT>::STAGE_BYTES, A_BYTES = Pipe<MT>::A_BYTES;
  constexpr uint32_t IDESC = idesc_bf16<BN>();
  constexpr int PIECE = T::four ? 32 : 16;                 // codes per 16-byte piece
  constexpr int PIECES_PER_ROW = BK / PIECE;               // 2 or 4 per K step
  constexpr int PIECES_PER_THREAD = (BN * PIECES_PER_ROW + DEC_THREADS - 1) / DEC_THREADS;   // 1, 2 or 4
  constexpr int ROWS_PER_PASS = DEC_THREADS / PIECES_PER_ROW;            // 128 or 64
  constexpr int NREG = T::four ? 16 : 8;
  constexpr uint32_t LO_OFF = uint32_t(BN) * BK * 2;       // lo rows follow the hi rows
  constexpr int PSTRIDE = BN + 4;                          // floats per partial-tile row (K split)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  // bars[0..S): A full (TMA), [S..2S): B full (decoders), [2S..3S): stage empty (MMA), [3S]: accumulator done
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(bars + 3 * STAGES + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // consecutive CTAs walk the N tiles of an M tile (its X tile shared, the
  // whole W streamed per M tile) or, mfast, the M tiles of an N tile (its W
  // tile shared, the whole X streamed per N tile): the host picks the order
  // that streams the smaller operand again, the larger one once
  const int n0 = (p.mfast ? blockIdx.y : blockIdx.x) * BN, m0 = (p.mfast ? blockIdx.x : blockIdx.y) * BM * MT;
  const int mtiles = p.mfast ? gridDim.x : gridDim.y;
  const int nkb = (p.K + BK - 1) / BK;
  // K split: this CTA accumulates K steps [kb0, kb1) (one split per cluster rank along z)
  const int kb0 = blockIdx.z * p.kb_per;
  const int kb1 = min(nkb, kb0 + p.kb_per);
  const int nloc = kb1 - kb0;
  const bool split_k = gridDim.z > 1;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto a_full = [&](int s) { return bar0 + 8u * s; };
  auto b_full = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  const uint32_t done_bar = bar0 + 8u * (3 * STAGES);
  auto stage_a = [&](int s) { return sbase + uint32_t(s * STAGE_BYTES); };
  auto stage_b = [&](int s) { return sbase + uint32_t(s * STAGE_BYTES + A_BYTES); };
  auto fail = [&]() {
    *abort_flag = 1u;
    atomicOr(&g_device_status, 1u);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(a_full(s), 1);
      mbar_init(b_full(s), DEC_WARPS);
      mbar_init(empty(s), 1);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&xmap)) : "memory");
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
  // The next kernel in the stream may launch now; X (and `out`) are touched only
  // after griddepcontrol.wait, the weights (not produced by the preceding kernel)
  // stream in right away.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int issued = 0;
      for (int j = 0; j < nloc; ++j) {
        const int s = j % STAGES;
        const uint32_t ph = (j / STAGES) & 1;
        if (*abort_flag) break;
        if (!mbar_wait(empty(s), ph ^ 1u, p.limit_ns)) { fail(); break; }
        mbar_arrive_expect_tx(a_full(s), A_BYTES);
        tma_load_2d(stage_a(s), &xmap, (kb0 + j) * BK, m0, a_full(s));
        issued = j + 1;
      }
      // every issued copy must land before the CTA may exit
      for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
        if (!mbar_wait(a_full(j % STAGES), (j / STAGES) & 1, p.limit_ns)) fail();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The warp walks the stages together (lane 0 waits, the outcome is
    // broadcast), so the stage addresses are warp-uniform; one elected lane
    // issues the MMAs (from one lane's branch each cost that thread ~67 cycles).
    const bool leader = elect_one();
    for (int j = 0; j < nloc; ++j) {
      const int s = j % STAGES;
      const uint32_t ph = (j / STAGES) & 1;
      int go = 1;
      if (lane == 0) {
        go = *abort_flag == 0u;
        if (go && !(mbar_wait(a_full(s), ph, p.limit_ns) && mbar_wait(b_full(s), ph, p.limit_ns))) {
          fail();
          go = 0;
        }
      }
      if (!__shfl_sync(0xFFFFFFFFu, go, 0)) break;
      tc_fence_after();
      const uint64_t bd = desc_sw128(stage_b(s)), ld = desc_sw128(stage_b(s) + LO_OFF);
      if (leader) {
        #pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {  // +32 bytes along K per instruction
          #pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint64_t ad = desc_sw128(stage_a(s) + uint32_t(mt * BM * BK * 2));
            const uint32_t d = tmem + uint32_t(mt * ACC);
            mma_f16(d, ad + uint64_t(2 * kk), bd + uint64_t(2 * kk), IDESC, (j | kk) != 0);
            if constexpr (SPLIT) mma_f16(d, ad + uint64_t(2 * kk), ld + uint64_t(2 * kk), IDESC, 1u);
          }
        }
        mma_commit(empty(s));
      }
      __syncwarp();
    }
    if (leader) mma_commit(done_bar);   // fires once every MMA issued above has completed
  } else {
    // -------------------------------------------------------------- decoders
    const int dt = threadIdx.x - 64;                       // 0 .. DEC_THREADS-1
    const int64_t row_bytes = T::four ? p.K / 2 : p.K;
    const int64_t nblk = (p.K + T::block - 1) / T::block;   // int4 affine: a ragged last group
    const int sub = dt % PIECES_PER_ROW;                   // piece index within the row's K step
    const int rbase = dt / PIECES_PER_ROW;
    using PC = PieceCodes<F>;
    PC cur[PIECES_PER_THREAD], nxt[PIECES_PER_THREAD];
    PieceScale cs[PIECES_PER_THREAD], ns[PIECES_PER_THREAD];
    auto load = [&](int kb, PC (&v)[PIECES_PER_THREAD], PieceScale (&sc)[PIECES_PER_THREAD]) {
      #pragma unroll
      for (int i = 0; i < PIECES_PER_THREAD; ++i) {
        const int r = rbase + i * ROWS_PER_PASS;
        const int n = n0 + r;
        const int64_t k0 = int64_t(kb) * BK + sub * PIECE;
        const bool ok = kb < kb1 && r < BN && n < p.N && k0 < p.K;   // rows past BN (224): zero, unused
        if constexpr (F == MXFP4X2) {   // output row n: plane 0, then plane 1, K/2 bytes each
          const uint8_t* pa = p.codes + int64_t(n) * p.K + k0 / 2;
          v[i].a = ok ? ldg_stream(pa) : make_uint4(0, 0, 0, 0);
          v[i].b = ok ? ldg_stream(pa + p.K / 2) : make_uint4(0, 0, 0, 0);
          const float* sr = reinterpret_cast<const float*>(p.scales) + int64_t(n) * 2 * nblk + k0 / 32;
          sc[i].a = ok ? __float_as_uint(__ldg(sr)) : 0u;
          sc[i].b = ok ? __float_as_uint(__ldg(sr + nblk)) : 0u;
        } else {
          v[i] = ok ? ldg_stream(p.codes + int64_t(n) * row_bytes + (T::four ? k0 / 2 : k0)) : make_uint4(0, 0, 0, 0);
          sc[i] = load_piece_scale<F>(p.scales, n, nblk, k0, ok);
        }
      }
    };
    // one M tile: this CTA's weight slab [kb0, kb1) towards L2 now (one row
    // per thread); with more M tiles the other tiles' CTAs share it
    if (mtiles == 1 && dt < BN && n0 + dt < p.N && nloc > 0) {
      const int64_t kbeg = int64_t(kb0) * BK, kend = min(int64_t(kb1) * BK, int64_t(p.K));
      if constexpr (F == MXFP4X2) {   // both planes of the row
        const uint8_t* src = p.codes + int64_t(n0 + dt) * p.K + kbeg / 2;
        prefetch_l2(src, uint64_t((kend - kbeg) / 2));
        prefetch_l2(src + p.K / 2, uint64_t((kend - kbeg) / 2));
      } else {
        const uint8_t* src = p.codes + int64_t(n0 + dt) * row_bytes + (T::four ? kbeg / 2 : kbeg);
        prefetch_l2(src, uint64_t(T::four ? (kend - kbeg) / 2 : (kend - kbeg)));
      }
    }
    // codes three K steps ahead in flight (cur, nxt, nx2 loaded; nx3 issued per step)
    PC nx2[PIECES_PER_THREAD];
    PieceScale ns2[PIECES_PER_THREAD];
    load(kb0, cur, cs);
    load(kb0 + 1, nxt, ns);
    load(kb0 + 2, nx2, ns2);
    bool aborted = false;
    for (int j = 0; j < nloc; ++j) {
      const int kb = kb0 + j;
      const int s = j % STAGES;
      const uint32_t ph = (j / STAGES) & 1;
      int ok = 1;
      if (lane == 0) ok = (*abort_flag == 0u) && mbar_wait(empty(s), ph ^ 1u, p.limit_ns);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0 && *abort_flag == 0u) fail();
        aborted = true;
        break;
      }
      PC nx3[PIECES_PER_THREAD];
      PieceScale ns3[PIECES_PER_THREAD];
      load(kb + 3, nx3, ns3);
      const uint32_t bs = stage_b(s);
      #pragma unroll
      for (int i = 0; i < PIECES_PER_THREAD; ++i) {
        const int r = rbase + i * ROWS_PER_PASS;
        if constexpr (SPLIT) {
          uint32_t hi[NREG], lo[NREG];
          if constexpr (F == MXFP4X2) decode_x2_hilo(cur[i].a, cur[i].b, cs[i], hi, lo);
          else decode_piece_hilo<F>(cur[i], cs[i], hi, lo);
          #pragma unroll
          for (int c = 0; c < NREG / 4; ++c) {
            const uint32_t off = sw128_off(r, sub * (NREG / 4) + c);
            sts128(bs + off, hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
            sts128(bs + LO_OFF + off, lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
          }
        } else {
          uint32_t w[NREG];
          decode_piece_natural<F>(cur[i], cs[i], w);
          #pragma unroll
          for (int c = 0; c < NREG / 4; ++c)
            sts128(bs + sw128_off(r, sub * (NREG / 4) + c), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
        cur[i] = nxt[i];
        cs[i] = ns[i];
        nxt[i] = nx2[i];
        ns[i] = ns2[i];
        nx2[i] = nx3[i];
        ns2[i] = ns3[i];
      }
      fence_proxy_async();                                 // generic-proxy stores -> tensor core reads
      __syncwarp();
      if (lane == 0 && !p.drop_arrivals) mbar_arrive(b_full(s));
    }
    (void)aborted;
    // --------------------------------------------------------------- epilogue
    if (warp < 2 + 4 * MT) {
      int ok = 1;
      if (lane == 0) ok = mbar_wait(done_bar, 0, p.limit_ns);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok && lane == 0) fail();
      tc_fence_after();
      const int q = warp & 3;                              // TMEM lane quadrant of this warp
      const int mt = (warp - 2) >> 2;                      // accumulator (128-row sub-tile)
      const int m = m0 + mt * BM + q * 32 + lane;
      const bool live = ok && *abort_flag == 0u;
      asm volatile("griddepcontrol.wait;" ::: "memory");
      #pragma unroll 1
      for (int cb = 0; cb < BN / 32; ++cb) {
        uint32_t r[32];
        tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(mt * ACC + cb * 32), r);
        if (split_k) {   // this split's partial tile into the (drained) stage memory
          float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(smem) + (q * 32 + lane) * PSTRIDE + cb * 32);
          #pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                                 __uint_as_float(r[4 * j + 3]));
          continue;
        }
        const int nb = n0 + cb * 32;
        if (!live || m >= p.M || nb >= p.N) continue;
        float v[32];
        #pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] = __uint_as_float(r[j]);
          if constexpr (F == NVFP4) v[j] *= p.glob;
        }
        const int ncols = p.N - nb < 32 ? p.N - nb : 32;
        if (p.out_f32) {
          float* o = static_cast<float*>(p.out) + int64_t(m) * p.N + nb;
          if (ncols == 32 && (p.N & 3) == 0) {
            #pragma unroll
            for (int j = 0; j < 8; ++j)
              reinterpret_cast<float4*>(o)[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          } else {
            #pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < ncols) o[j] = v[j];
          }
        } else {
          __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + int64_t(m) * p.N + nb;
          if (ncols == 32 && (p.N & 7) == 0) {
            #pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t h[4];
              #pragma unroll
              for (int t = 0; t < 4; ++t)
                h[t] = f32_to_bf16bits(v[8 * j + 2 * t]) | (f32_to_bf16bits(v[8 * j + 2 * t + 1]) << 16);
              reinterpret_cast<uint4*>(o)[j] = make_uint4(h[0], h[1], h[2], h[3]);
            }
          } else {
            #pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < ncols) o[j] = __float2bfloat16_rn(v[j]);
          }
        }
      }
    }
  }

  if (split_k) {
    // The splits of one tile form a cluster: each CTA sums a slice of the
    // tile over the cluster's partial tiles (rank order) and stores it.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    cluster_sync();
    uint32_t rank, csize;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(rank));
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
    // a CTA whose wait expired holds no valid partial tile: then no CTA of the
    // cluster writes its slice
    uint32_t any_abort = 0u;
    for (uint32_t q = 0; q < csize; ++q) any_abort |= ld_cluster_u32(smem_u32((const void*)abort_flag), q);
    constexpr int E = BM * (BN / 4);                       // float4 elements of the tile
    const int e0 = int(rank) * E / int(csize), e1 = any_abort ? e0 : (int(rank) + 1) * E / int(csize);
    for (int e = e0 + int(threadIdx.x); e < e1; e += THREADS) {
      const int row = e / (BN / 4), c4 = e - row * (BN / 4);
      const int m = m0 + row, n = n0 + 4 * c4;
      if (m >= p.M || n >= p.N) continue;
      const uint32_t sa = sbase + uint32_t((row * PSTRIDE + 4 * c4) * 4);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      for (uint32_t q = 0; q < csize; ++q) {
        const float4 w = ld_cluster_f32x4(sa, q);
        v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
      }
      if constexpr (F == NVFP4) { v.x *= p.glob; v.y *= p.glob; v.z *= p.glob; v.w *= p.glob; }
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

static std::atomic<uint64_t> g_limit_ns{2000000000ull};
static std::atomic<int> g_drop{0};
static std::atomic<int> g_order{0};   // tile order override for measurements: 0 the host's choice, 1 N tiles first, 2 M tiles first

template <int F, int MT, int BN = Tile<F>::BN>
static cudaError_t launch_mt(EncodeTiledFn enc, const void* codes, const void* scales, float glob, const void* x,
                             void* out, bool out_f32, int M, int N, int K, cudaStream_t st, int S) {
  static std::atomic<int> attr_done[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !attr_done[dev].load()) {
    e = cudaFuncSetAttribute(qgemm_tc_kernel<F, MT, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Pipe<MT>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_done[dev].store(1);
  }
  CUtensorMap map;
  const cuuint64_t gdim[2] = {cuuint64_t(K), cuuint64_t(M)};
  const cuuint64_t gstride[1] = {cuuint64_t(K) * 2};
  const cuuint32_t box[2] = {BK, cuuint32_t(BM * MT)};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(x), gdim, gstride, box, estride,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  Params prm;
  prm.codes = static_cast<const uint8_t*>(codes);
  prm.scales = static_cast<const uint8_t*>(scales);
  prm.out = out;
  prm.glob = glob;
  prm.M = M;
  prm.N = N;
  prm.K = K;
  prm.out_f32 = out_f32 ? 1 : 0;
  prm.limit_ns = g_limit_ns.load();
  prm.drop_arrivals = g_drop.load();
  // K split: the S splits of every tile form a cluster (MT = 1 only, whose
  // float32 partial tile fits the drained stage memory)
  const int nkb = (K + BK - 1) / BK;
  prm.kb_per = (nkb + S - 1) / S;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  at[1].id = cudaLaunchAttributeClusterDimension;
  at[1].val.clusterDim.x = 1;
  at[1].val.clusterDim.y = 1;
  at[1].val.clusterDim.z = unsigned(S);
  // Tile order (no K split): M tiles first when the activations are the
  // smaller operand, so that each wave streams a band of W once and every CTA
  // of the band re-reads X from L2 (nvfp8 M = 4096, N = 11008: X 34 MB, W 45 MB
  // read once per M tile in the N-first order)
  const int64_t ntl = (N + BN - 1) / BN, mtl = (M + BM * MT - 1) / (BM * MT);
  const double xbytes = 2.0 * double(M) * double(K);
  const double wbytes = double(N) * double(K) * (FmtTraits<F>::four && F != MXFP4X2 ? 0.5 : 1.0);
  prm.mfast = S == 1 && mtl > 1 && ntl <= 65535 && xbytes < wbytes ? 1 : 0;
  if (S == 1 && g_order.load() == 1) prm.mfast = 0;
  if (S == 1 && g_order.load() == 2 && ntl <= 65535) prm.mfast = 1;
  lc.gridDim = prm.mfast ? dim3(unsigned(mtl), unsigned(ntl), 1) : dim3(unsigned(ntl), unsigned(mtl), S);
  lc.blockDim = dim3(Dec<F>::CTA_THREADS);
  lc.dynamicSmemBytes = Pipe<MT>::SMEM_BYTES;
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, qgemm_tc_kernel<F, MT, BN>, map, prm);
}

// Tile shape (MT 128-row accumulators per CTA) and K split S, by the estimated
// time in K steps of one CTA: the decoders set the pace, so a K step costs
// about the same with one accumulator or two (two measured ~10 % longer), times
// the waves of one-CTA-per-SM work, plus ~8 K steps for a split's partial-tile
// reduction.  No split may be left empty.
struct GemmPlan {
  int MT, S, BN;
};
inline GemmPlan plan_gemm(bool split, int M, int N, int K, int sms) {
  const int nkb = (K + BK - 1) / BK;
  GemmPlan best{1, 1, split ? 128 : 256};
  double best_cost = 1e300;
  // the formats exact in bf16 may also take 224-wide tiles without a K split
  // (152 SMs hold 19 x 8 tiles of 224 x 256 in one wave where 16 x 8 tiles of
  // 256 leave 24 idle; a K step then costs about 224/256 of a 256-wide one)
  for (int bn : {256, 224, 128}) {
    if (split ? bn != 128 : bn == 128) continue;
    const int ntiles = (N + bn - 1) / bn;
    for (int mt = 1; mt <= 2; ++mt) {
      if (mt == 2 && M <= BM) continue;
      const int64_t mtiles = (M + int64_t(BM) * mt - 1) / (int64_t(BM) * mt);
      for (int s = 1; s <= (mt == 1 ? 4 : 1); ++s) {
        const int per = (nkb + s - 1) / s;
        if (s > 1 && (s - 1) * per >= nkb) continue;
        // a K split runs as clusters of s CTAs, packed per GPC: 224-wide tiles
        // would overflow the co-resident clusters of a wave (measured slower)
        if (bn == 224 && s > 1) continue;
        const int64_t ctas = int64_t(ntiles) * mtiles * s;
        const int64_t waves = (ctas + sms - 1) / sms;
        const double width = split ? 1.0 : bn / 256.0;
        const double cost = double(waves) * per * (mt == 2 ? 1.1 : 1.0) * width + (s > 1 ? 8.0 : 0.0);
        if (cost < best_cost - 1e-9) {
          best_cost = cost;
          best = {mt, s, bn};
        }
      }
    }
  }
  return best;
}

template <int F>
static cudaError_t launch_fmt(const void* codes, const void* scales, float glob, const void* x, void* out,
                              bool out_f32, int M, int N, int K, cudaStream_t st, int sms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const GemmPlan pl = plan_gemm(Tile<F>::split, M, N, K, sms > 0 ? sms : 1);
  if constexpr (!Tile<F>::split) {
    if (pl.BN == 224) {
      if (pl.MT == 2) return launch_mt<F, 2, 224>(enc, codes, scales, glob, x, out, out_f32, M, N, K, st, 1);
      return launch_mt<F, 1, 224>(enc, codes, scales, glob, x, out, out_f32, M, N, K, st, pl.S);
    }
  }
  if (pl.MT == 2) return launch_mt<F, 2>(enc, codes, scales, glob, x, out, out_f32, M, N, K, st, 1);
  return launch_mt<F, 1>(enc, codes, scales, glob, x, out, out_f32, M, N, K, st, pl.S);
}

}  // namespace tc

cudaError_t launch_qgemm_tc(int fmt, const void* codes, const void* scales, float glob, const void* x, void* out,
                            bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st, int sms) {
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return tc::launch_fmt<MXFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case NVFP4: return tc::launch_fmt<NVFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXFP8_E4M3: return tc::launch_fmt<MXFP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXFP8_E5M2: return tc::launch_fmt<MXFP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case NVFP8: return tc::launch_fmt<NVFP8>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case NVFP8_F16: return tc::launch_fmt<NVFP8_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXINT8: return tc::launch_fmt<MXINT8>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case INT8: return tc::launch_fmt<INT8>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case INT8_F16: return tc::launch_fmt<INT8_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case INT4: return tc::launch_fmt<INT4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case INT4_F16: return tc::launch_fmt<INT4_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXFP4X2: return tc::launch_fmt<MXFP4X2>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case MXINT4: return tc::launch_fmt<MXINT4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP4: return tc::launch_fmt<FP4>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP4_F16: return tc::launch_fmt<FP4_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP8_E4M3: return tc::launch_fmt<FP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP8_E4M3_F16: return tc::launch_fmt<FP8_E4M3_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP8_E5M2: return tc::launch_fmt<FP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    case FP8_E5M2_F16: return tc::launch_fmt<FP8_E5M2_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
    default: return tc::launch_fmt<INT4_AFFINE>(codes, scales, glob, x, out, out_f32, m, n, k, st, sms);
  }
}

// Test hooks for the bounded waits (see qfmt_debug_set in the C ABI).
void set_wait_limit_ns(uint64_t ns) { tc::g_limit_ns.store(ns); }
uint64_t wait_limit_ns() { return tc::g_limit_ns.load(); }
void set_drop_arrivals(int on) { tc::g_drop.store(on); }
void set_tc_order(int v) { tc::g_order.store(v); }
int drop_arrivals() { return tc::g_drop.load(); }

cudaError_t read_and_clear_device_status(unsigned int* status) {
  cudaError_t e = cudaMemcpyFromSymbol(status, g_device_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
}

}  // namespace qfmt_dev
