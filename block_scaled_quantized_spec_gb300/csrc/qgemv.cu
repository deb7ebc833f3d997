// Decode-phase dequantizing GEMV, 1 <= M <= 16:
//   out[m, n] = sum_k x[m, k] * dequant(W)[n, k]
// (metaltile PR #250 qgemv commits: output[row] = sum_k dequant(weight[row,k])
// * input[k], and the multi-row qmm; rlx-cpu thunk/ops/quant.rs
// dequant_matmul_nvfp4, whose m == 1 loop streams the packed codes once).
//
// The pages' Metal kernels give each row one threadgroup and reduce with a
// scalar loop; they note it reads at a low fraction of bandwidth.  Here the
// work is shaped for GB300 instead:
//  * a CTA owns 16 weight rows and 8 warps split K between them; every lane
//    streams 16-byte pieces (32 four-bit / 16 eight-bit codes) of two rows with
//    128-bit loads, four pieces per row per warp in flight;
//  * codes are decoded in registers straight into bf16 tensor-core fragments
//    with the block scale applied (exact for the power-of-two and E4M3 scales;
//    nvfp8/int4-affine weights round once to bf16), and warp-level
//    mma.sync m16n8k16 (bf16 in, float32 accumulate) multiplies them by the
//    activations: weights are the 16-row A operand, activations the 8-column B
//    operand (a second B block covers 9 <= M <= 16);
//  * the per-warp partial tiles are summed through shared memory and the
//    nvfp4 global scale is applied once to each output.
#include <cuda_runtime.h>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {

constexpr int GEMV_WARPS = 8;
constexpr int GEMV_UNROLL = 4;

__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Activation B-fragment halves for one column (batch row) over the same k
// slots as decode_piece: xs points at the piece's first activation.
template <bool FOUR>
__device__ __forceinline__ void load_x_piece(const __nv_bfloat16* xs, bool ok, uint32_t B[FOUR ? 8 : 4][2]) {
  if constexpr (FOUR) {
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(xs) + j) : make_uint4(0, 0, 0, 0);
      B[2 * j][0] = prmt(v.x, v.z, 0x5410u);      // (x0, x4)
      B[2 * j][1] = prmt(v.x, v.z, 0x7632u);      // (x1, x5)
      B[2 * j + 1][0] = prmt(v.y, v.w, 0x5410u);  // (x2, x6)
      B[2 * j + 1][1] = prmt(v.y, v.w, 0x7632u);  // (x3, x7)
    }
  } else {
    #pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(xs) + h) : make_uint4(0, 0, 0, 0);
      B[2 * h][0] = prmt(v.x, v.y, 0x5410u);      // (x0, x2)
      B[2 * h][1] = prmt(v.x, v.y, 0x7632u);      // (x1, x3)
      B[2 * h + 1][0] = prmt(v.z, v.w, 0x5410u);
      B[2 * h + 1][1] = prmt(v.z, v.w, 0x7632u);
    }
  }
}

template <int F, int NB>
__global__ void __launch_bounds__(GEMV_WARPS * 32) qgemv_kernel(
    const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, float glob,
    const __nv_bfloat16* __restrict__ x, void* __restrict__ out, int out_f32, int M, int N, int K) {
  using T = FmtTraits<F>;
  constexpr int PIECE = T::four ? 32 : 16;  // codes per lane per row per chunk
  constexpr int CHUNK = PIECE * 4;          // codes per row per chunk (one quad)
  constexpr int STEPS = T::four ? 8 : 4;    // mma k16 steps per piece
  __shared__ float red[GEMV_WARPS][16][8 * NB];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * 16;
  const int rA = row0 + g, rB = row0 + g + 8;
  const bool okA = rA < N, okB = rB < N;
  const int64_t row_bytes = T::four ? K / 2 : K;
  const int64_t nblk = K / T::block;
  const int nchunks = (K + CHUNK - 1) / CHUNK;
  const uint8_t* pA = codes + int64_t(okA ? rA : 0) * row_bytes;
  const uint8_t* pB = codes + int64_t(okB ? rB : 0) * row_bytes;

  float acc[NB][4];
  #pragma unroll
  for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;

  for (int c0 = warp; c0 < nchunks; c0 += GEMV_WARPS * GEMV_UNROLL) {
    uint4 wa[GEMV_UNROLL], wb[GEMV_UNROLL];
    PieceScale sa[GEMV_UNROLL], sb[GEMV_UNROLL];
    bool kin[GEMV_UNROLL];
    #pragma unroll
    for (int u = 0; u < GEMV_UNROLL; ++u) {
      const int c = c0 + u * GEMV_WARPS;
      const int64_t k0 = int64_t(c) * CHUNK + t * PIECE;
      kin[u] = c < nchunks && k0 < K;
      const int64_t off = T::four ? k0 / 2 : k0;
      wa[u] = kin[u] && okA ? ldg_stream(pA + off) : make_uint4(0, 0, 0, 0);
      wb[u] = kin[u] && okB ? ldg_stream(pB + off) : make_uint4(0, 0, 0, 0);
      sa[u] = load_piece_scale<F>(scales, rA, nblk, k0, kin[u] && okA);
      sb[u] = load_piece_scale<F>(scales, rB, nblk, k0, kin[u] && okB);
    }
    #pragma unroll
    for (int u = 0; u < GEMV_UNROLL; ++u) {
      const int c = c0 + u * GEMV_WARPS;
      if (c >= nchunks) break;
      const int64_t k0 = int64_t(c) * CHUNK + t * PIECE;
      uint32_t A0[STEPS][2], A1[STEPS][2];
      decode_piece<F>(wa[u], sa[u], A0);
      decode_piece<F>(wb[u], sb[u], A1);
      #pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int m = nb * 8 + g;
        uint32_t B[STEPS][2];
        load_x_piece<T::four>(x + int64_t(m < M ? m : 0) * K + k0, kin[u] && m < M, B);
        #pragma unroll
        for (int s = 0; s < STEPS; ++s)
          mma_bf16(acc[nb], A0[s][0], A1[s][0], A0[s][1], A1[s][1], B[s][0], B[s][1]);
      }
    }
  }

  // acc[nb]: c0 = (row g, col 2t), c1 = (g, 2t+1), c2 = (g+8, 2t), c3 = (g+8, 2t+1).
  #pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    red[warp][g][nb * 8 + 2 * t] = acc[nb][0];
    red[warp][g][nb * 8 + 2 * t + 1] = acc[nb][1];
    red[warp][g + 8][nb * 8 + 2 * t] = acc[nb][2];
    red[warp][g + 8][nb * 8 + 2 * t + 1] = acc[nb][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * M; i += blockDim.x) {
    const int r = i & 15, m = i >> 4;
    if (row0 + r >= N) continue;
    float sum = 0.0f;
    #pragma unroll
    for (int w = 0; w < GEMV_WARPS; ++w) sum += red[w][r][m];
    if constexpr (F == NVFP4) sum *= glob;
    const int64_t o = int64_t(m) * N + row0 + r;
    if (out_f32) static_cast<float*>(out)[o] = sum;
    else static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(sum);
  }
}

// ---------------------------------------------------------------------------
// nvfp8 and int4 affine: the weights stay exact in bf16 (E4M3 codes, or the
// integers 128 + q) and the block scale is applied to float32 partial sums.
// That needs every mma.sync to draw its 16 k values from one block, so the
// four lanes of a quad share each block: nvfp8 lanes take word t of each of
// four consecutive 16-byte blocks (32-bit loads), int4 affine lanes take bytes
// 8t..8t+7 of each of two 32-byte groups (64-bit loads).  int4 affine adds
// one mma per step against a matrix of ones to get the activation sums the
// affine bias multiplies: sum_k x (s q + b) = s sum_k x (128 + q) + (b - 128 s) sum_k x.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mma_bf16_zero(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint32_t ldg32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ldg64(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

template <int F, int NB>
__global__ void __launch_bounds__(GEMV_WARPS * 32) qgemv_blockacc_kernel(
    const uint8_t* __restrict__ codes, const uint8_t* __restrict__ scales, const __nv_bfloat16* __restrict__ x,
    void* __restrict__ out, int out_f32, int M, int N, int K) {
  constexpr bool I4 = F == INT4_AFFINE;
  constexpr int CHUNK = I4 ? 128 : 64;         // codes per row per chunk: 2 groups / 4 blocks
  constexpr int NSUB = I4 ? 2 : 4;             // scale blocks per chunk
  __shared__ float red[GEMV_WARPS][16][8 * NB];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int row0 = blockIdx.x * 16;
  const int rA = row0 + g, rB = row0 + g + 8;
  const bool okA = rA < N, okB = rB < N;
  const int64_t row_bytes = I4 ? K / 2 : K;
  const int64_t nblk = K / (I4 ? 64 : 16);
  const int nchunks = (K + CHUNK - 1) / CHUNK;
  const uint8_t* pA = codes + int64_t(okA ? rA : 0) * row_bytes;
  const uint8_t* pB = codes + int64_t(okB ? rB : 0) * row_bytes;
  const int64_t sA0 = int64_t(okA ? rA : 0) * nblk, sB0 = int64_t(okB ? rB : 0) * nblk;

  float acc[NB][4];
  #pragma unroll
  for (int nb = 0; nb < NB; ++nb) acc[nb][0] = acc[nb][1] = acc[nb][2] = acc[nb][3] = 0.0f;

  for (int c0 = warp; c0 < nchunks; c0 += GEMV_WARPS * GEMV_UNROLL) {
    // words[u][j]: nvfp8: word t of block j (4 codes); int4: word j of the lane's 8 bytes in group j/2
    uint32_t wa[GEMV_UNROLL][4], wb[GEMV_UNROLL][4];
    uint32_t sa[GEMV_UNROLL][NSUB], sb[GEMV_UNROLL][NSUB];
    #pragma unroll
    for (int u = 0; u < GEMV_UNROLL; ++u) {
      const int c = c0 + u * GEMV_WARPS;
      #pragma unroll
      for (int j = 0; j < NSUB; ++j) {
        const int64_t kb = int64_t(c) * CHUNK + j * (I4 ? 64 : 16);   // first k of the block
        const bool ok = c < nchunks && kb < K;
        const int64_t blk = kb / (I4 ? 64 : 16);
        if constexpr (I4) {
          const int64_t off = kb / 2 + 8 * t;
          uint2 va = ok && okA ? ldg64(pA + off) : make_uint2(0, 0);
          uint2 vb = ok && okB ? ldg64(pB + off) : make_uint2(0, 0);
          wa[u][2 * j] = va.x; wa[u][2 * j + 1] = va.y;
          wb[u][2 * j] = vb.x; wb[u][2 * j + 1] = vb.y;
          sa[u][j] = ok && okA ? __ldg(reinterpret_cast<const uint32_t*>(scales) + sA0 + blk) : 0u;
          sb[u][j] = ok && okB ? __ldg(reinterpret_cast<const uint32_t*>(scales) + sB0 + blk) : 0u;
        } else {
          const int64_t off = kb + 4 * t;
          wa[u][j] = ok && okA ? ldg32(pA + off) : 0u;
          wb[u][j] = ok && okB ? ldg32(pB + off) : 0u;
          sa[u][j] = ok && okA ? __ldg(reinterpret_cast<const uint32_t*>(scales) + sA0 + blk) : 0u;
          sb[u][j] = ok && okB ? __ldg(reinterpret_cast<const uint32_t*>(scales) + sB0 + blk) : 0u;
        }
      }
    }
    #pragma unroll
    for (int u = 0; u < GEMV_UNROLL; ++u) {
      const int c = c0 + u * GEMV_WARPS;
      if (c >= nchunks) break;
      #pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        const int m = nb * 8 + g;
        const bool mok = m < M;
        const __nv_bfloat16* xr = x + int64_t(mok ? m : 0) * K;
        #pragma unroll
        for (int j = 0; j < NSUB; ++j) {
          const int64_t kb = int64_t(c) * CHUNK + j * (I4 ? 64 : 16);
          const bool ok = kb < K && mok;
          if constexpr (I4) {
            // lane's 16 activations of group j: k = kb + 16t .. +15 (two words of 8)
            const uint4 v0 = ok ? __ldg(reinterpret_cast<const uint4*>(xr + kb + 16 * t)) : make_uint4(0, 0, 0, 0);
            const uint4 v1 = ok ? __ldg(reinterpret_cast<const uint4*>(xr + kb + 16 * t + 8)) : make_uint4(0, 0, 0, 0);
            float d[4] = {0.f, 0.f, 0.f, 0.f}, xs[4] = {0.f, 0.f, 0.f, 0.f};
            #pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint4 v = h ? v1 : v0;
              uint32_t ra[4], rb[4];
              int4x8_biased_bf16(wa[u][2 * j + h], ra);
              int4x8_biased_bf16(wb[u][2 * j + h], rb);
              const uint32_t b00 = prmt(v.x, v.z, 0x5410u), b01 = prmt(v.x, v.z, 0x7632u);
              const uint32_t b10 = prmt(v.y, v.w, 0x5410u), b11 = prmt(v.y, v.w, 0x7632u);
              mma_bf16(d, ra[0], rb[0], ra[1], rb[1], b00, b01);
              mma_bf16(d, ra[2], rb[2], ra[3], rb[3], b10, b11);
              const uint32_t one = 0x3F803F80u;
              mma_bf16(xs, one, one, one, one, b00, b01);
              mma_bf16(xs, one, one, one, one, b10, b11);
            }
            const float sA = bf16bits_f32(sa[u][j] & 0xFFFFu), bA = bf16bits_f32(sa[u][j] >> 16);
            const float sB = bf16bits_f32(sb[u][j] & 0xFFFFu), bB = bf16bits_f32(sb[u][j] >> 16);
            const float cA = __fmaf_rn(-128.0f, sA, bA), cB = __fmaf_rn(-128.0f, sB, bB);
            acc[nb][0] = __fmaf_rn(sA, d[0], __fmaf_rn(cA, xs[0], acc[nb][0]));
            acc[nb][1] = __fmaf_rn(sA, d[1], __fmaf_rn(cA, xs[1], acc[nb][1]));
            acc[nb][2] = __fmaf_rn(sB, d[2], __fmaf_rn(cB, xs[2], acc[nb][2]));
            acc[nb][3] = __fmaf_rn(sB, d[3], __fmaf_rn(cB, xs[3], acc[nb][3]));
          } else {
            // lane's 4 activations of block j: k = kb + 4t .. +3
            const uint2 v = ok ? ldg64(xr + kb + 4 * t) : make_uint2(0, 0);
            const uint32_t b0 = prmt(v.x, v.y, 0x5410u), b1 = prmt(v.x, v.y, 0x7632u);   // (x0,x2) (x1,x3)
            uint32_t ra[2], rb[2];
            e4m3x4_bf16_raw(wa[u][j], ra);
            e4m3x4_bf16_raw(wb[u][j], rb);
            const uint32_t k120 = 0x7B807B80u;                     // 2^120: exact E4M3 values
            float d[4];
            mma_bf16_zero(d, hmul2(ra[0], k120), hmul2(rb[0], k120), hmul2(ra[1], k120), hmul2(rb[1], k120), b0, b1);
            const float sA = __uint_as_float(sa[u][j]), sB = __uint_as_float(sb[u][j]);
            acc[nb][0] = __fmaf_rn(sA, d[0], acc[nb][0]);
            acc[nb][1] = __fmaf_rn(sA, d[1], acc[nb][1]);
            acc[nb][2] = __fmaf_rn(sB, d[2], acc[nb][2]);
            acc[nb][3] = __fmaf_rn(sB, d[3], acc[nb][3]);
          }
        }
      }
    }
  }

  #pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    red[warp][g][nb * 8 + 2 * t] = acc[nb][0];
    red[warp][g][nb * 8 + 2 * t + 1] = acc[nb][1];
    red[warp][g + 8][nb * 8 + 2 * t] = acc[nb][2];
    red[warp][g + 8][nb * 8 + 2 * t + 1] = acc[nb][3];
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 16 * M; i += blockDim.x) {
    const int r = i & 15, m = i >> 4;
    if (row0 + r >= N) continue;
    float sum = 0.0f;
    #pragma unroll
    for (int w = 0; w < GEMV_WARPS; ++w) sum += red[w][r][m];
    const int64_t o = int64_t(m) * N + row0 + r;
    if (out_f32) static_cast<float*>(out)[o] = sum;
    else static_cast<__nv_bfloat16*>(out)[o] = __float2bfloat16_rn(sum);
  }
}

template <int F>
static cudaError_t launch_qgemv_fmt(const void* codes, const void* scales, float glob, const void* x,
                                    void* out, bool out_f32, int M, int N, int K, cudaStream_t st) {
  dim3 grid((N + 15) / 16), block(GEMV_WARPS * 32);
  auto c = static_cast<const uint8_t*>(codes);
  auto s = static_cast<const uint8_t*>(scales);
  auto xx = static_cast<const __nv_bfloat16*>(x);
  if constexpr (F == NVFP8 || F == INT4_AFFINE) {
    if (M <= 8) qgemv_blockacc_kernel<F, 1><<<grid, block, 0, st>>>(c, s, xx, out, out_f32, M, N, K);
    else qgemv_blockacc_kernel<F, 2><<<grid, block, 0, st>>>(c, s, xx, out, out_f32, M, N, K);
  } else {
    if (M <= 8) qgemv_kernel<F, 1><<<grid, block, 0, st>>>(c, s, glob, xx, out, out_f32, M, N, K);
    else qgemv_kernel<F, 2><<<grid, block, 0, st>>>(c, s, glob, xx, out, out_f32, M, N, K);
  }
  return cudaGetLastError();
}

cudaError_t launch_qgemv(int fmt, const void* codes, const void* scales, float glob, const void* x,
                         void* out, bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st,
                         int sms) {
  (void)sms;
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return launch_qgemv_fmt<MXFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP4: return launch_qgemv_fmt<NVFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP8_E4M3: return launch_qgemv_fmt<MXFP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP8_E5M2: return launch_qgemv_fmt<MXFP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP8: return launch_qgemv_fmt<NVFP8>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    default: return launch_qgemv_fmt<INT4_AFFINE>(codes, scales, glob, x, out, out_f32, m, n, k, st);
  }
}

// ---------------------------------------------------------------------------
// Float32 activations: CUDA-core path with exact float32 weights.
// One warp per (row n, group of up to 8 batch rows); lanes stride K by pieces.
// ---------------------------------------------------------------------------

template <int F>
__device__ __forceinline__ float exact_weight(uint32_t code, float s, float b) {
  if constexpr (F == MXFP4 || F == NVFP4) return __fmul_rn(e2m1_f32(code), s);
  if constexpr (F == MXFP8_E4M3 || F == NVFP8) return __fmul_rn(e4m3_f32(code), s);
  if constexpr (F == MXFP8_E5M2) return __fmul_rn(e5m2_f32(code), s);
  return __fmaf_rn(s, float(code), b);
}

template <int F>
__global__ void __launch_bounds__(256) qmm_f32x_kernel(const uint8_t* __restrict__ codes,
                                                       const uint8_t* __restrict__ scales, float glob,
                                                       const float* __restrict__ x, void* __restrict__ out,
                                                       int out_f32, int M, int N, int K) {
  using T = FmtTraits<F>;
  constexpr int PIECE = T::four ? 32 : 16;
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int mgroups = (M + 7) / 8;
  if (wid >= int64_t(N) * mgroups) return;
  const int n = int(wid / mgroups), m0 = int(wid % mgroups) * 8;
  const int64_t row_bytes = T::four ? K / 2 : K;
  const int64_t nblk = K / T::block;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int k0 = lane * PIECE; k0 < K; k0 += 32 * PIECE) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(codes + n * row_bytes + (T::four ? k0 / 2 : k0)));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    #pragma unroll
    for (int i = 0; i < PIECE; ++i) {
      const int k = k0 + i;
      const int64_t bi = n * nblk + k / T::block;
      float s, b = 0.0f;
      if constexpr (F == MXFP4 || F == MXFP8_E4M3 || F == MXFP8_E5M2) s = e8m0_f32(scales[bi]);
      else if constexpr (F == NVFP4) s = e4m3_f32(scales[bi]);
      else if constexpr (F == NVFP8) s = reinterpret_cast<const float*>(scales)[bi];
      else {
        const uint32_t p = reinterpret_cast<const uint32_t*>(scales)[bi];
        s = bf16bits_f32(p & 0xFFFFu);
        b = bf16bits_f32(p >> 16);
      }
      const uint32_t code = T::four ? (wv[i >> 3] >> (4 * (i & 7))) & 0xFu : (wv[i >> 2] >> (8 * (i & 3))) & 0xFFu;
      const float w = exact_weight<F>(code, s, b);
      #pragma unroll
      for (int j = 0; j < 8; ++j)
        if (m0 + j < M) acc[j] = __fmaf_rn(x[int64_t(m0 + j) * K + k], w, acc[j]);
    }
  }
  #pragma unroll
  for (int j = 0; j < 8; ++j) {
    float v = acc[j];
    #pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if (lane == 0 && m0 + j < M) {
      if constexpr (F == NVFP4) v *= glob;
      const int64_t oi = int64_t(m0 + j) * N + n;
      if (out_f32) static_cast<float*>(out)[oi] = v;
      else static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(v);
    }
  }
}

template <int F>
static cudaError_t launch_f32x_fmt(const void* codes, const void* scales, float glob, const float* x,
                                   void* out, bool out_f32, int M, int N, int K, cudaStream_t st) {
  const int64_t warps = int64_t(N) * ((M + 7) / 8);
  const int64_t blocks = (warps * 32 + 255) / 256;
  qmm_f32x_kernel<F><<<dim3(unsigned(blocks)), 256, 0, st>>>(
      static_cast<const uint8_t*>(codes), static_cast<const uint8_t*>(scales), glob, x, out, out_f32, M, N, K);
  return cudaGetLastError();
}

cudaError_t launch_qmm_f32x(int fmt, const void* codes, const void* scales, float glob, const float* x,
                            void* out, bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st,
                            int sms) {
  (void)sms;
  const int m = int(M), n = int(N), k = int(K);
  switch (fmt) {
    case MXFP4: return launch_f32x_fmt<MXFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP4: return launch_f32x_fmt<NVFP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP8_E4M3: return launch_f32x_fmt<MXFP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP8_E5M2: return launch_f32x_fmt<MXFP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case NVFP8: return launch_f32x_fmt<NVFP8>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    default: return launch_f32x_fmt<INT4_AFFINE>(codes, scales, glob, x, out, out_f32, m, n, k, st);
  }
}

}  // namespace qfmt_dev
