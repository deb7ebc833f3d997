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

// Per-piece scale state, loaded with the codes.
struct PieceScale {
  uint32_t a, b;  // format-specific raw scale words
};

template <int F>
__device__ __forceinline__ PieceScale load_piece_scale(const uint8_t* scales, int64_t row, int64_t nblk,
                                                       int64_t k0, bool ok) {
  PieceScale s{0u, 0u};
  if (!ok) return s;
  const int64_t base = row * nblk;
  if constexpr (F == MXFP4 || F == MXFP8_E4M3 || F == MXFP8_E5M2) {
    s.a = __ldg(scales + base + k0 / 32);
  } else if constexpr (F == NVFP4) {
    s.a = __ldg(reinterpret_cast<const unsigned short*>(scales + base + k0 / 16));
  } else if constexpr (F == NVFP8) {
    s.a = __ldg(reinterpret_cast<const uint32_t*>(scales) + base + k0 / 16);
  } else {
    s.a = __ldg(reinterpret_cast<const uint32_t*>(scales) + base + k0 / 64);
  }
  return s;
}

// Decode one 16-byte piece of one row into the A-fragment halves of each mma
// step: A[s][0] feeds k slots (2t, 2t+1), A[s][1] slots (2t+8, 2t+9).
// 4-bit: 8 steps (word j gives steps 2j, 2j+1); 8-bit: 4 steps (word j -> step j).
template <int F>
__device__ __forceinline__ void decode_piece(const uint4& v, const PieceScale& ps,
                                             uint32_t A[FmtTraits<F>::four ? 8 : 4][2]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (F == MXFP4 || F == NVFP4) {
    uint32_t sc0, sc1;
    if constexpr (F == MXFP4) {
      sc0 = sc1 = bf16x2_splat(e8m0_bf16(ps.a));
    } else {
      sc0 = bf16x2_splat(f32_to_bf16bits(e4m3_f32(ps.a & 0xFFu)));
      sc1 = bf16x2_splat(f32_to_bf16bits(e4m3_f32(ps.a >> 8)));
    }
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t r[4];
      e2m1x8_bf16(w[j], r);
      const uint32_t sc = j < 2 ? sc0 : sc1;
      A[2 * j][0] = hmul2(r[0], sc);
      A[2 * j][1] = hmul2(r[1], sc);
      A[2 * j + 1][0] = hmul2(r[2], sc);
      A[2 * j + 1][1] = hmul2(r[3], sc);
    }
  } else if constexpr (F == INT4_AFFINE) {
    const uint32_t s2 = bf16x2_splat(ps.a & 0xFFFFu), b2 = bf16x2_splat(ps.a >> 16);
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t r[4];
      int4x8_affine_bf16(w[j], s2, b2, r);
      A[2 * j][0] = r[0];
      A[2 * j][1] = r[1];
      A[2 * j + 1][0] = r[2];
      A[2 * j + 1][1] = r[3];
    }
  } else {
    // 8-bit: raw bf16 = value * 2^-bias_gap; one multiply restores the bias and
    // applies the block scale when the combined factor fits bf16, else two.
    uint32_t m1, m2 = 0x3F803F80u;
    bool two = false;
    if constexpr (F == MXFP8_E4M3 || F == MXFP8_E5M2) {
      constexpr int gap = F == MXFP8_E4M3 ? 120 : 112;
      const int b = int(ps.a);
      if (b == 255) {
        m1 = 0x7FC07FC0u;
      } else if (b - 127 + gap <= 127) {
        m1 = bf16x2_splat(pow2_bf16(b - 127 + gap));
      } else {
        m1 = bf16x2_splat(pow2_bf16(gap));
        m2 = bf16x2_splat(pow2_bf16(b - 127));
        two = true;
      }
    } else {  // NVFP8: float32 scale rounded once to bf16
      const float s = __uint_as_float(ps.a);
      if (fabsf(s) < 128.0f) {
        m1 = bf16x2_splat(f32_to_bf16bits(s * 0x1p120f));
      } else {
        m1 = bf16x2_splat(pow2_bf16(120));
        m2 = bf16x2_splat(f32_to_bf16bits(s));
        two = true;
      }
    }
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t r[2];
      if constexpr (F == MXFP8_E5M2) e5m2x4_bf16_raw(w[j], r);
      else e4m3x4_bf16_raw(w[j], r);
      A[j][0] = hmul2(r[0], m1);
      A[j][1] = hmul2(r[1], m1);
      if (two) {
        A[j][0] = hmul2(A[j][0], m2);
        A[j][1] = hmul2(A[j][1], m2);
      }
    }
  }
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

template <int F>
static cudaError_t launch_qgemv_fmt(const void* codes, const void* scales, float glob, const void* x,
                                    void* out, bool out_f32, int M, int N, int K, cudaStream_t st) {
  dim3 grid((N + 15) / 16), block(GEMV_WARPS * 32);
  auto c = static_cast<const uint8_t*>(codes);
  auto s = static_cast<const uint8_t*>(scales);
  auto xx = static_cast<const __nv_bfloat16*>(x);
  if (M <= 8) qgemv_kernel<F, 1><<<grid, block, 0, st>>>(c, s, glob, xx, out, out_f32, M, N, K);
  else qgemv_kernel<F, 2><<<grid, block, 0, st>>>(c, s, glob, xx, out, out_f32, M, N, K);
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
