// Float32-activation dequantizing matmul on CUDA cores (any M): exact float32
// weights (the dequant values of the standalone dequant kernel) times float32
// activations, float32 accumulation.  Used for float32 X, e.g. the tiny
// correctness workload (M = 8, N = 16, K = 512).
#include <cuda_runtime.h>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {

// One warp per (row n, group of up to 8 batch rows); lanes stride K by 16-byte pieces.

template <int F>
__device__ __forceinline__ float exact_weight(uint32_t code, float s, float b) {
  if constexpr (F == MXFP4 || F == NVFP4 || F == FP4 || F == FP4_F16) return __fmul_rn(e2m1_f32(code), s);
  if constexpr (is_int8<F>()) return __fmul_rn(float(int8_t(uint8_t(code))), s);
  if constexpr (is_e5m2<F>()) return __fmul_rn(e5m2_f32(code), s);
  if constexpr (F == MXFP8_E4M3 || is_fs8<F>()) return __fmul_rn(e4m3_f32(code), s);
  if constexpr (is_i4sym<F>() || F == MXINT4) return __fmul_rn(float(int(code ^ 8u) - 8), s);
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
  const int64_t nblk = (K + T::block - 1) / T::block;   // int4 affine: a ragged last group
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if constexpr (F == MXFP4X2) {   // rows 2n and 2n + 1: the residual planes of output row n
    for (int k0 = lane * PIECE; k0 < K; k0 += 32 * PIECE) {
      const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(codes + (2 * int64_t(n)) * row_bytes + k0 / 2));
      const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(codes + (2 * int64_t(n) + 1) * row_bytes + k0 / 2));
      const float* sr = reinterpret_cast<const float*>(scales) + 2 * int64_t(n) * nblk;
      const float s0 = sr[k0 / 32], s1 = sr[nblk + k0 / 32];
      const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
      #pragma unroll
      for (int i = 0; i < PIECE; ++i) {
        const float w = __fmaf_rn(e2m1_f32((w1[i >> 3] >> (4 * (i & 7))) & 0xFu), s1,
                                  __fmul_rn(e2m1_f32((w0[i >> 3] >> (4 * (i & 7))) & 0xFu), s0));
        #pragma unroll
        for (int j = 0; j < 8; ++j)
          if (m0 + j < M) acc[j] = __fmaf_rn(x[int64_t(m0 + j) * K + k0 + i], w, acc[j]);
      }
    }
  } else {
  for (int k0 = lane * PIECE; k0 < K; k0 += 32 * PIECE) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(codes + n * row_bytes + (T::four ? k0 / 2 : k0)));
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    #pragma unroll
    for (int i = 0; i < PIECE; ++i) {
      const int k = k0 + i;
      const int64_t bi = n * nblk + k / T::block;
      float s, b = 0.0f;
      if constexpr (is_e8m0<F>()) s = e8m0_f32(scales[bi]);
      else if constexpr (F == NVFP4) s = e4m3_f32(scales[bi]);
      else if constexpr (is_fs8<F>() || is_i4sym<F>() || is_fp4f<F>()) s = float_scale<F>(scales, bi);
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
    case NVFP8_F16: return launch_f32x_fmt<NVFP8_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXINT8: return launch_f32x_fmt<MXINT8>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case INT8: return launch_f32x_fmt<INT8>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case INT8_F16: return launch_f32x_fmt<INT8_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case INT4: return launch_f32x_fmt<INT4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case INT4_F16: return launch_f32x_fmt<INT4_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXFP4X2: return launch_f32x_fmt<MXFP4X2>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case MXINT4: return launch_f32x_fmt<MXINT4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP4: return launch_f32x_fmt<FP4>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP4_F16: return launch_f32x_fmt<FP4_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP8_E4M3: return launch_f32x_fmt<FP8_E4M3>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP8_E4M3_F16: return launch_f32x_fmt<FP8_E4M3_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP8_E5M2: return launch_f32x_fmt<FP8_E5M2>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    case FP8_E5M2_F16: return launch_f32x_fmt<FP8_E5M2_F16>(codes, scales, glob, x, out, out_f32, m, n, k, st);
    default: return launch_f32x_fmt<INT4_AFFINE>(codes, scales, glob, x, out, out_f32, m, n, k, st);
  }
}

}  // namespace qfmt_dev
