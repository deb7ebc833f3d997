// Standalone block-scaled dequant: out[n, k] = elem(code) * scale(block).
//
// metaltile PR #250, "First spec-conformant block-scaled dequant kernel" and
// the commit completing the five dequant kernels: out[i] = e2m1(code) *
// 2^(scale_bits - 127) (mxfp4), E2M1 x E4M3 micro-scale x FP32 global (nvfp4),
// 8-bit elements with E8M0 (mxfp8) or FP32 (nvfp8) block scales; the int4
// affine value scale * q + bias of metaltile-std tests/qmm_gpu_correctness.rs.
//
// GB300 layout: a thread writes 16 bytes of output per step (4 float32 or 8
// bf16 values of one row, inside one block since every block size is a
// multiple of 8), reading their 2-8 code bytes and one scale; consecutive
// lanes take consecutive steps, so each warp instruction stores 512
// contiguous bytes.  The kernel is bound by the output write; the grid fills
// every SM and strides over the steps.  Every product rounds once in float32
// (no flush-to-zero), which is the bit-exact contract.
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

// A warp takes 32 consecutive 16-byte code pieces (pieces run in row-major
// order over [N, K], so their outputs are one contiguous run of out): each
// lane loads one piece with a 128-bit load into shared memory, then the warp
// writes the run 512 bytes per instruction, lane l taking the V (4 float32 or
// 8 bf16) outputs at l V of each 32 V.
template <int F, bool OUT_BF16>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ codes,
                                                      const uint8_t* __restrict__ scales, float glob,
                                                      void* __restrict__ out, int64_t N, int64_t K) {
  using T = FmtTraits<F>;
  constexpr int PIECE = T::four ? 32 : 16;            // codes per 16-byte piece
  constexpr int V = OUT_BF16 ? 8 : 4;                 // outputs per lane and store: 16 bytes
  constexpr int BITS = T::four ? 4 : 8;
  constexpr int STEPS = 32 * PIECE / (32 * V);        // store instructions per warp run
  __shared__ uint4 stage[8][32];
  __shared__ uint4 stage1[F == MXFP4X2 ? 8 : 1][32];   // mxfp4x2: the plane-1 pieces
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t pieces = N * (K / PIECE);             // mxfp4x2: pieces of plane 0, one per 32 outputs
  const int64_t nblk = (K + T::block - 1) / T::block; // int4 affine: a ragged last group
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t wstride = int64_t(gridDim.x) * (blockDim.x >> 5) * 32;
  for (int64_t base = (int64_t(blockIdx.x) * (blockDim.x >> 5) + warp) * 32; base < pieces; base += wstride) {
    const int64_t p = base + lane;
    const int64_t e0 = base * PIECE;                  // first output element of the run
    const int64_t row0 = e0 / K;
    if constexpr (F == MXFP4X2) {
      // the residual planes of a row sit side by side: plane q of row r is
      // code row 2r + q; both planes' pieces are staged
      uint4 v0 = make_uint4(0, 0, 0, 0), v1 = v0;
      if (p < pieces) {
        const int64_t r = p / (K / PIECE), j = p - r * (K / PIECE);
        v0 = __ldg(reinterpret_cast<const uint4*>(codes) + (2 * r) * (K / PIECE) + j);
        v1 = __ldg(reinterpret_cast<const uint4*>(codes) + (2 * r + 1) * (K / PIECE) + j);
      }
      stage[warp][lane] = v0;
      stage1[warp][lane] = v1;
      __syncwarp();
      const uint32_t* sw0 = reinterpret_cast<const uint32_t*>(&stage[warp][0]);
      const uint32_t* sw1 = reinterpret_cast<const uint32_t*>(&stage1[warp][0]);
      #pragma unroll
      for (int q = 0; q < STEPS; ++q) {
        const int off = q * 32 * V + lane * V;          // element offset in the run
        const int64_t e = e0 + off;
        if (e >= N * K) break;
        const int sh = 4 * (off % 8);
        const uint32_t w0 = sw0[off / 8], w1 = sw1[off / 8];
        const int64_t r = row0 + int64_t(uint32_t(e - row0 * K) / uint32_t(K)), k = e - r * K;
        const float* sr = reinterpret_cast<const float*>(scales) + 2 * r * nblk;
        const double s0 = __ldg(sr + k / 32), s1 = __ldg(sr + nblk + k / 32);
        float o[V];
        #pragma unroll
        for (int i = 0; i < V; ++i) {
          const double a = e2m1_f32((w0 >> (sh + 4 * i)) & 0xFu);
          const double b = e2m1_f32((w1 >> (sh + 4 * i)) & 0xFu);
          o[i] = __double2float_rn(__dadd_rn(__dmul_rn(a, s0), __dmul_rn(b, s1)));
        }
        if constexpr (OUT_BF16) {
          uint32_t h[4];
          #pragma unroll
          for (int t = 0; t < 4; ++t) h[t] = f32_to_bf16bits(o[2 * t]) | (f32_to_bf16bits(o[2 * t + 1]) << 16);
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + e) = make_uint4(h[0], h[1], h[2], h[3]);
        } else {
          *reinterpret_cast<float4*>(static_cast<float*>(out) + e) = make_float4(o[0], o[1], o[2], o[3]);
        }
      }
      __syncwarp();
    } else {
      stage[warp][lane] = p < pieces ? __ldg(reinterpret_cast<const uint4*>(codes) + p) : make_uint4(0, 0, 0, 0);
      __syncwarp();
      const uint8_t* sb = reinterpret_cast<const uint8_t*>(&stage[warp][0]);
      #pragma unroll
      for (int q = 0; q < STEPS; ++q) {
        const int off = q * 32 * V + lane * V;          // element offset in the run
        const int64_t e = e0 + off;
        if (e >= N * K) break;
        const int64_t r = row0 + int64_t(uint32_t(e - row0 * K) / uint32_t(K)), k = e - r * K;
        float s, b;
        dq_scale<F>(scales, r * nblk + k / T::block, s, b);
        uint64_t w;
        if constexpr (BITS * V == 16) w = *reinterpret_cast<const unsigned short*>(sb + off / 2);
        else if constexpr (BITS * V == 32) w = *reinterpret_cast<const unsigned int*>(sb + off * BITS / 8);
        else w = *reinterpret_cast<const unsigned long long*>(sb + off);
        float o[V];
        #pragma unroll
        for (int i = 0; i < V; ++i) o[i] = dq_value<F>(uint32_t(w >> (BITS * i)) & ((1u << BITS) - 1u), s, b, glob);
        if constexpr (OUT_BF16) {
          uint32_t h[4];
          #pragma unroll
          for (int t = 0; t < 4; ++t) h[t] = f32_to_bf16bits(o[2 * t]) | (f32_to_bf16bits(o[2 * t + 1]) << 16);
          *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + e) = make_uint4(h[0], h[1], h[2], h[3]);
        } else {
          *reinterpret_cast<float4*>(static_cast<float*>(out) + e) = make_float4(o[0], o[1], o[2], o[3]);
        }
      }
      __syncwarp();
    }
  }
}

template <int F>
static cudaError_t launch_dequant_fmt(const void* codes, const void* scales, float glob, void* out,
                                      bool bf16, int64_t N, int64_t K, cudaStream_t st, int sms) {
  const int64_t total = N * (K / (FmtTraits<F>::four ? 32 : 16));   // 16-byte pieces, one a lane
  const int threads = 256;
  int64_t want = (total + threads - 1) / threads;
  // as many CTAs as the SMs hold at once (the loop strides over the rest)
  static int per_sm[2] = {0, 0};
  int& ps = per_sm[bf16 ? 1 : 0];
  if (ps == 0) {
    int v = 0;
    const cudaError_t e = bf16 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, dequant_kernel<F, true>, threads, 0)
                               : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, dequant_kernel<F, false>, threads, 0);
    ps = (e == cudaSuccess && v > 0) ? v : 4;
  }
  int64_t cap = int64_t(sms) * ps;
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
