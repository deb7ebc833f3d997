// Standalone block-scaled dequant: out[n, k] = elem(code) * scale(block).
//
// metaltile PR #250, "First spec-conformant block-scaled dequant kernel" and
// the commit completing the five dequant kernels: out[i] = e2m1(code) *
// 2^(scale_bits - 127) (mxfp4), E2M1 x E4M3 micro-scale x FP32 global (nvfp4),
// 8-bit elements with E8M0 (mxfp8) or FP32 (nvfp8) block scales; the int4
// affine value scale * q + bias of metaltile-std tests/qmm_gpu_correctness.rs.
//
// GB300 layout: one thread owns one 16-byte piece of codes (32 four-bit or 16
// eight-bit codes, always inside one row since K is a multiple of 32), loads it
// with one 128-bit load and writes its 32 (16) outputs with 128-bit stores, so
// a warp streams 512 contiguous code bytes in and 4 KiB (2 KiB) out.  The
// kernel is bound by the output write; the grid is a multiple of the SM count
// and strides over the pieces.  Every product rounds once in float32 (no
// flush-to-zero), which is the bit-exact contract.
#include <cuda_runtime.h>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {

template <int F>
__device__ __forceinline__ float dq_value(uint32_t code, float s, float b, float glob) {
  if constexpr (F == MXFP4 || F == FP4 || F == FP4_F16) return __fmul_rn(e2m1_f32(code), s);
  if constexpr (F == NVFP4) return __fmul_rn(__fmul_rn(e2m1_f32(code), s), glob);   // (e2m1 * e4m3) exact
  if constexpr (F == MXFP8_E4M3) return __fmul_rn(e4m3_f32(code), s);
  if constexpr (is_e5m2<F>()) return __fmul_rn(e5m2_f32(code), s);
  if constexpr (is_int8<F>()) return __fmul_rn(float(int8_t(uint8_t(code))), s);
  if constexpr (is_fs8<F>()) return __fmul_rn(e4m3_f32(code), s);
  if constexpr (is_i4sym<F>() || F == MXINT4) return __fmul_rn(float(int(code ^ 8u) - 8), s);   // the sign-extended nibble
  return __fmaf_rn(s, float(code), b);                                               // INT4_AFFINE
}

// Scale (and bias) of block `blk` of row `row`, decoded to float32.
template <int F>
__device__ __forceinline__ void dq_scale(const uint8_t* scales, int64_t idx, float& s, float& b) {
  b = 0.0f;
  if constexpr (is_e8m0<F>()) s = e8m0_f32(scales[idx]);
  else if constexpr (F == NVFP4) s = e4m3_f32(scales[idx]);
  else if constexpr (is_fs8<F>() || is_i4sym<F>() || is_fp4f<F>()) s = float_scale<F>(scales, idx);
  else {
    const uint32_t p = reinterpret_cast<const uint32_t*>(scales)[idx];
    s = bf16bits_f32(p & 0xFFFFu);
    b = bf16bits_f32(p >> 16);
  }
}

template <int F, bool OUT_BF16>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ codes,
                                                      const uint8_t* __restrict__ scales, float glob,
                                                      void* __restrict__ out, int64_t N, int64_t K) {
  using T = FmtTraits<F>;
  constexpr int PIECE = T::four ? 32 : 16;     // codes per 16-byte piece
  const int64_t pieces_per_row = K / PIECE;
  const int64_t total = N * pieces_per_row;
  const int64_t nblk = (K + T::block - 1) / T::block;   // int4 affine: a ragged last group
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int64_t p = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; p < total;
       p += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = p / pieces_per_row;
    const int64_t k0 = (p - row * pieces_per_row) * PIECE;
    float o[PIECE];
    if constexpr (F == MXFP4X2) {
      // the two residual planes of row `row` (plane 0, then plane 1, K/2 bytes
      // each) under their float32 block scales: s0 e0 + s1 e1, the products
      // exact in double, the sum rounded in double and then to float32
      const int64_t j = p - row * pieces_per_row;
      const uint4 v0 = __ldg(reinterpret_cast<const uint4*>(codes) + 2 * row * pieces_per_row + j);
      const uint4 v1 = __ldg(reinterpret_cast<const uint4*>(codes) + (2 * row + 1) * pieces_per_row + j);
      const float* sr = reinterpret_cast<const float*>(scales) + 2 * row * nblk;
      const double s0 = __ldg(sr + k0 / 32), s1 = __ldg(sr + nblk + k0 / 32);
      const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
      #pragma unroll
      for (int i = 0; i < PIECE; ++i) {
        const double e0 = e2m1_f32((w0[i >> 3] >> (4 * (i & 7))) & 0xFu);
        const double e1 = e2m1_f32((w1[i >> 3] >> (4 * (i & 7))) & 0xFu);
        o[i] = __double2float_rn(__dadd_rn(__dmul_rn(e0, s0), __dmul_rn(e1, s1)));
      }
    } else {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(codes) + p);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    float s = 0.0f, b = 0.0f;
    // blocks inside the piece: 4-bit: 32 codes = 1 (mx), 2 (nvfp4), 1/2 (int4) blocks;
    // 8-bit: 16 codes = 1/2 (mx) or 1 (nvfp8) block.
    #pragma unroll
    for (int i = 0; i < PIECE; ++i) {
      const int64_t blk = row * nblk + (k0 + i) / T::block;
      if (i == 0 || ((k0 + i) % T::block) == 0) dq_scale<F>(scales, blk, s, b);
      uint32_t code = T::four ? (wv[i >> 3] >> (4 * (i & 7))) & 0xFu : (wv[i >> 2] >> (8 * (i & 3))) & 0xFFu;
      o[i] = dq_value<F>(code, s, b, glob);
    }
    }
    if constexpr (OUT_BF16) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row * K + k0);
      #pragma unroll
      for (int q = 0; q < PIECE / 8; ++q) {
        uint32_t h[4];
        #pragma unroll
        for (int j = 0; j < 4; ++j)
          h[j] = f32_to_bf16bits(o[8 * q + 2 * j]) | (f32_to_bf16bits(o[8 * q + 2 * j + 1]) << 16);
        dst[q] = make_uint4(h[0], h[1], h[2], h[3]);
      }
    } else {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(out) + row * K + k0);
      #pragma unroll
      for (int q = 0; q < PIECE / 4; ++q) dst[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
    }
  }
}

template <int F>
static cudaError_t launch_dequant_fmt(const void* codes, const void* scales, float glob, void* out,
                                      bool bf16, int64_t N, int64_t K, cudaStream_t st, int sms) {
  constexpr int PIECE = FmtTraits<F>::four ? 32 : 16;
  const int64_t total = N * (K / PIECE);
  const int threads = 256;
  int64_t want = (total + threads - 1) / threads;
  int64_t cap = int64_t(sms) * 8;
  int grid = int(want < cap ? want : cap);
  if (grid < 1) grid = 1;
  auto c = static_cast<const uint8_t*>(codes);
  auto s = static_cast<const uint8_t*>(scales);
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(grid);
  lc.blockDim = dim3(threads);
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 1;
  return bf16 ? cudaLaunchKernelEx(&lc, dequant_kernel<F, true>, c, s, glob, out, N, K)
              : cudaLaunchKernelEx(&lc, dequant_kernel<F, false>, c, s, glob, out, N, K);
}

cudaError_t launch_dequant(int fmt, const void* codes, const void* scales, float glob, void* out,
                           bool out_bf16, int64_t N, int64_t K, cudaStream_t st, int sms) {
  switch (fmt) {
    case MXFP4: return launch_dequant_fmt<MXFP4>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case NVFP4: return launch_dequant_fmt<NVFP4>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case MXFP8_E4M3: return launch_dequant_fmt<MXFP8_E4M3>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case MXFP8_E5M2: return launch_dequant_fmt<MXFP8_E5M2>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case NVFP8: return launch_dequant_fmt<NVFP8>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case NVFP8_F16: return launch_dequant_fmt<NVFP8_F16>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case MXINT8: return launch_dequant_fmt<MXINT8>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case INT8: return launch_dequant_fmt<INT8>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case INT8_F16: return launch_dequant_fmt<INT8_F16>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case INT4: return launch_dequant_fmt<INT4>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case INT4_F16: return launch_dequant_fmt<INT4_F16>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case MXFP4X2: return launch_dequant_fmt<MXFP4X2>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case MXINT4: return launch_dequant_fmt<MXINT4>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case FP4: return launch_dequant_fmt<FP4>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case FP4_F16: return launch_dequant_fmt<FP4_F16>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case FP8_E4M3: return launch_dequant_fmt<FP8_E4M3>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case FP8_E4M3_F16: return launch_dequant_fmt<FP8_E4M3_F16>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case FP8_E5M2: return launch_dequant_fmt<FP8_E5M2>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    case FP8_E5M2_F16: return launch_dequant_fmt<FP8_E5M2_F16>(codes, scales, glob, out, out_bf16, N, K, st, sms);
    default: return launch_dequant_fmt<INT4_AFFINE>(codes, scales, glob, out, out_bf16, N, K, st, sms);
  }
}

}  // namespace qfmt_dev
