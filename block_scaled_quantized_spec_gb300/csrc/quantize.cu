// Activation quantizer on the GPU: X [M, K] (bf16 or float32) -> an MX
// format's codes and E8M0 scales, the same bytes the host packer gives for a
// weight of that format (rlx-cpu thunk/ops/quant.rs lowp_compute_scales /
// lowp_snap_scale / lowp_quantize; metaltile PR #250's packer commit):
//   per block of 32 along K: amax = max |x|; s = amax / max_finite in float32
//   (1.0 for an all-zero block); the stored scale is the smallest power of two
//   >= s (E8M0, read exactly off s's float32 bits); codes = the element
//   format's nearest-even, saturating encoding of x / 2^e (cvt.rn.satfinite).
// One thread per block (a warp takes a row's 32 consecutive blocks).  Two
// output layouts: the library's weight layout (codes [M, K] or [M, K/2]
// bytes, scales [M, K/32]), and for the quantized-activation GEMMs the
// workspace layout (codes as in the weight layout, scales in 512-byte atoms
// of 128 rows x 4 blocks, the source layout of tcgen05.cp).
#include <cuda_runtime.h>

#include "decode.cuh"
#include "kernels.h"
#include "umma_desc.h"

namespace qfmt_dev {
namespace quant {

// E8M0 code (biased by 127) of the smallest power of two >= s, for finite
// float32 s > 0: a normal s = 1.m 2^E gives E, +1 when m != 0; a subnormal s =
// m 2^-149 gives ceil(log2 m) - 149; clamped to [-127, 127].
__device__ __forceinline__ uint32_t e8m0_ceil_code(float s) {
  const uint32_t b = __float_as_uint(s);
  const int E = int(b >> 23), m = int(b & 0x7FFFFFu);
  int e;
  if (E > 0) e = E - 127 + (m != 0 ? 1 : 0);
  else e = (m <= 1 ? 0 : 32 - __clz(m - 1)) - 149;
  return uint32_t(min(max(e, -127), 127) + 127);
}

// 2^-(code - 127) as a float32 (code <= 254): exact, subnormal at code 254.
__device__ __forceinline__ float e8m0_inv(uint32_t code) {
  const int e = 127 - int(code);
  return e >= -126 ? __uint_as_float(uint32_t(e + 127) << 23) : __uint_as_float(0x00400000u);
}

template <int F> struct Elem;
template <> struct Elem<MXFP4> {
  static constexpr float MAXF = 6.0f;
  // two float32 -> one byte, `a` in the low nibble
  static __device__ __forceinline__ uint32_t pair(float a, float b) {
    uint32_t r;
    asm("{.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;}" : "=r"(r) : "f"(b), "f"(a));
    return r;
  }
};
template <> struct Elem<MXFP8_E4M3> {
  static constexpr float MAXF = 448.0f;
  static __device__ __forceinline__ uint32_t pair(float a, float b) {   // two bytes, `a` in the low byte
    uint16_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h) : "f"(b), "f"(a));
    return h;
  }
};
template <> struct Elem<MXFP8_E5M2> {
  static constexpr float MAXF = 57344.0f;
  static __device__ __forceinline__ uint32_t pair(float a, float b) {
    uint16_t h;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(h) : "f"(b), "f"(a));
    return h;
  }
};

// The 32 values of block b of row m as float32.
template <bool IN_F32>
__device__ __forceinline__ void load32(const void* x, int64_t m, int64_t K, int b, float (&v)[32]) {
  if constexpr (IN_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + m * K + 32 * int64_t(b));
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 f = __ldg(p + i);
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + m * K + 32 * int64_t(b));
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = __ldg(p + i);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      #pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * i + 2 * j] = __uint_as_float(ws[j] << 16);
        v[8 * i + 2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
      }
    }
  }
}

// ATOMS: the workspace layout of the quantized-activation GEMMs (E4M3 codes
// [M, K], or mxfp4 codes [M, K/2]); rows past M up to the 128-row tile then
// get neutral scale words.
template <int F, bool IN_F32, bool ATOMS>
__global__ void __launch_bounds__(256) quantize_kernel(const void* __restrict__ x, uint8_t* __restrict__ codes,
                                                       uint8_t* __restrict__ scales, int M, int K) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nblk = K / 32, chunks = (nblk + 31) / 32;
  const int rows = ATOMS ? (M + 127) / 128 * 128 : M;
  const int m = warp / chunks, b = (warp - m * chunks) * 32 + lane;
  if (m >= rows) return;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const bool live = b < nblk;
  uint32_t sc = 127u;
  if (live && m < M) {
    float v[32];
    load32<IN_F32>(x, m, K, b, v);
    float amax = 0.0f;
    bool finite = true;
    #pragma unroll
    for (int i = 0; i < 32; ++i) {
      finite &= fabsf(v[i]) <= 3.4028235e38f;                 // false for an infinity or a NaN
      amax = fmaxf(amax, fabsf(v[i]));
    }
    const float s = amax > 0.0f ? __fdiv_rn(amax, Elem<F>::MAXF) : 1.0f;
    sc = finite ? e8m0_ceil_code(s) : 255u;                   // a non-finite block: the NaN scale
    const float inv = finite ? e8m0_inv(sc) : 1.0f;
    if constexpr (F == MXFP4) {
      uint32_t w[4];
      #pragma unroll
      for (int i = 0; i < 4; ++i) {
        w[i] = 0u;
        #pragma unroll
        for (int j = 0; j < 4; ++j)
          w[i] |= Elem<F>::pair(__fmul_rn(v[8 * i + 2 * j], inv), __fmul_rn(v[8 * i + 2 * j + 1], inv)) << (8 * j);
      }
      *reinterpret_cast<uint4*>(codes + int64_t(m) * (K / 2) + 16 * int64_t(b)) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      uint32_t w[8];
      #pragma unroll
      for (int i = 0; i < 8; ++i)
        w[i] = Elem<F>::pair(__fmul_rn(v[4 * i], inv), __fmul_rn(v[4 * i + 1], inv)) |
               (Elem<F>::pair(__fmul_rn(v[4 * i + 2], inv), __fmul_rn(v[4 * i + 3], inv)) << 16);
      uint4* d = reinterpret_cast<uint4*>(codes + int64_t(m) * K + 32 * int64_t(b));
      d[0] = make_uint4(w[0], w[1], w[2], w[3]);
      d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
  if constexpr (ATOMS) {
    // four blocks of one row share a 32-bit scale cell of the atom
    uint32_t word = sc;
    #pragma unroll
    for (int d = 1; d < 4; ++d) word |= __shfl_down_sync(0xFFFFFFFFu, sc, d) << (8 * d);
    if (live && (lane & 3) == 0) {
      const size_t atom = size_t(m / 128) * size_t(K / 128) + size_t(b / 4);
      *reinterpret_cast<uint32_t*>(scales + atom * 512 + umma::sf_atom_offset(uint32_t(m % 128), 0)) = word;
    }
  } else {
    if (live && m < M) scales[int64_t(m) * nblk + b] = uint8_t(sc);
  }
}

// ---- NVFP4 activations (the all-FP4 product over nvfp4 weights) ----------
//
// The packer's nvfp4 rule over the whole X as one tensor: global g =
// amax(X) / (6 * 448) (1.0 for a zero X); per block of 16, t = (amax / 6) / g
// in float32, its E4M3 code by nearest-even saturating conversion (a zero
// block: 0x38 = 1.0), eff = E4M3(code) * g, codes = E2M1(x / eff) (eff = 0:
// code 0).  Two kernels: per-CTA maxima of |x|, then (every CTA reducing the
// maxima) the codes and the scale atoms; CTA 0 stores g.  A non-finite X
// makes g, hence every output, NaN.

constexpr int NV_PARTIALS = 1024;

// CTA c's largest |x| over the 16-byte chunks of X taken grid-stride (X is
// [M, K] contiguous), four independent loads in flight a thread.
__global__ void __launch_bounds__(256) amax_partial_kernel(const __nv_bfloat16* __restrict__ x, int M, int K,
                                                           float* __restrict__ partial) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float red[8];
  float a = 0.0f;
  bool finite = true;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t chunks = int64_t(M) * (K / 8), stride = int64_t(gridDim.x) * blockDim.x;
  auto take = [&](const uint4 v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = fabsf(__uint_as_float(w[j] << 16)), hi = fabsf(__uint_as_float(w[j] & 0xFFFF0000u));
      finite &= lo <= 3.4028235e38f && hi <= 3.4028235e38f;   // false for an infinity or a NaN
      a = fmaxf(a, fmaxf(lo, hi));
    }
  };
  int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; c + 3 * stride < chunks; c += 4 * stride) {
    const uint4 v0 = __ldg(xv + c), v1 = __ldg(xv + c + stride), v2 = __ldg(xv + c + 2 * stride),
                v3 = __ldg(xv + c + 3 * stride);
    take(v0);
    take(v1);
    take(v2);
    take(v3);
  }
  for (; c < chunks; c += stride) take(__ldg(xv + c));
  if (!finite) a = __uint_as_float(0x7FC00000u);
  #pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, a, d);
    a = (a != a || o != o) ? __uint_as_float(0x7FC00000u) : fmaxf(a, o);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = red[0];
    for (int i = 1; i < int(blockDim.x >> 5); ++i) r = (r != r || red[i] != red[i]) ? __uint_as_float(0x7FC00000u) : fmaxf(r, red[i]);
    partial[blockIdx.x] = r;
  }
}

// Codes [M, K/2] and E4M3 scales in 512-byte atoms (128 rows x 4 blocks of
// 16: a 32-bit cell covers 64 K); one thread per 32 values (two blocks), a
// warp per row and 1,024 columns; rows past M up to the 128-row tile get
// neutral scales (1.0).  `nparts` maxima from amax_partial_kernel.
__global__ void __launch_bounds__(256) quantize_nv_atoms_kernel(const __nv_bfloat16* __restrict__ x,
                                                                uint8_t* __restrict__ codes,
                                                                uint8_t* __restrict__ atoms,
                                                                const float* __restrict__ partial, int nparts,
                                                                float* __restrict__ g_out, int M, int K) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float red[8];
  __shared__ float gsh;
  float a = 0.0f;
  for (int i = threadIdx.x; i < nparts; i += blockDim.x) {
    const float v = __ldg(partial + i);
    a = (a != a || v != v) ? __uint_as_float(0x7FC00000u) : fmaxf(a, v);
  }
  #pragma unroll
  for (int d = 16; d > 0; d >>= 1) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, a, d);
    a = (a != a || o != o) ? __uint_as_float(0x7FC00000u) : fmaxf(a, o);
  }
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = red[0];
    for (int i = 1; i < int(blockDim.x >> 5); ++i) r = (r != r || red[i] != red[i]) ? __uint_as_float(0x7FC00000u) : fmaxf(r, red[i]);
    const float g = r != r ? r : (r > 0.0f ? __fdiv_rn(r, 2688.0f) : 1.0f);
    gsh = g;
    if (blockIdx.x == 0) *g_out = g;
  }
  __syncthreads();
  const float g = gsh;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int nchunk = K / 32, chunks = (nchunk + 31) / 32;
  const int rows = (M + 127) / 128 * 128;
  const int m = warp / chunks, b = (warp - m * chunks) * 32 + lane;   // b: 32-value chunk of the row
  if (m >= rows || b >= nchunk) return;
  uint32_t sc[2] = {0x38u, 0x38u};
  if (m < M) {
    float v[32];
    load32<false>(x, m, K, b, v);
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    #pragma unroll
    for (int h = 0; h < 2; ++h) {                               // the two blocks of 16
      float amax = 0.0f;
      #pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[16 * h + i]));
      uint32_t code = 0x38u;
      if (amax > 0.0f) {
        const float t = __fdiv_rn(__fdiv_rn(amax, 6.0f), g);
        uint16_t two;
        asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(two) : "f"(0.0f), "f"(t));
        code = two & 0xFFu;
      }
      if (h) sc[1] = code;
      else sc[0] = code;
      const float eff = __fmul_rn(e4m3_f32(code), g);
      // The code of float32(x / eff) without a division per value: q = x * r
      // (r the rounded reciprocal) is within 3 * 2^-24 of float32(x / eff),
      // relative; the E2M1 rounding is monotone, so where q (1 - 2^-20) and
      // q (1 + 2^-20) take the same code, that is the code (a tie, i.e. a
      // quotient on a midpoint, always falls between them).  Otherwise, and
      // for a non-finite q, the pair is divided.
      const float r = __frcp_rn(eff);
      #pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float a = v[16 * h + 2 * i], b = v[16 * h + 2 * i + 1];
        uint32_t byte = 0u;
        if (eff != 0.0f) {
          const float qa = __fmul_rn(a, r), qb = __fmul_rn(b, r);
          const uint32_t lo = Elem<MXFP4>::pair(__fmul_rn(qa, 1.0f - 0x1p-20f), __fmul_rn(qb, 1.0f - 0x1p-20f));
          const uint32_t hi = Elem<MXFP4>::pair(__fmul_rn(qa, 1.0f + 0x1p-20f), __fmul_rn(qb, 1.0f + 0x1p-20f));
          const bool fin = fabsf(qa) <= 3.4028235e38f && fabsf(qb) <= 3.4028235e38f;
          byte = (lo == hi && fin) ? lo : Elem<MXFP4>::pair(__fdiv_rn(a, eff), __fdiv_rn(b, eff));
        }
        w[2 * h + i / 4] |= byte << (8 * (i % 4));
      }
    }
    *reinterpret_cast<uint4*>(codes + int64_t(m) * (K / 2) + 16 * int64_t(b)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  // blocks 2b, 2b + 1: bytes (2b) % 4, (2b + 1) % 4 of cell (2b) / 4
  const size_t atom = size_t(m / 128) * size_t(K / 64) + size_t(b / 2);
  uint8_t* cell = atoms + atom * 512 + umma::sf_atom_offset(uint32_t(m % 128), uint32_t((2 * b) & 3));
  cell[0] = uint8_t(sc[0]);
  cell[1] = uint8_t(sc[1]);
}

template <int F, bool IN_F32, bool ATOMS>
static cudaError_t launch(const void* x, void* codes, void* scales, int M, int K, cudaStream_t st) {
  const int rows = ATOMS ? (M + 127) / 128 * 128 : M;
  const int64_t warps = int64_t(rows) * ((K / 32 + 31) / 32);
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(unsigned((warps + 7) / 8));
  lc.blockDim = dim3(256);
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, quantize_kernel<F, IN_F32, ATOMS>, x, static_cast<uint8_t*>(codes),
                            static_cast<uint8_t*>(scales), M, K);
}

}  // namespace quant

cudaError_t launch_quantize(int fmt, const void* x, bool x_f32, void* codes, void* scales, int64_t M, int64_t K,
                            cudaStream_t st) {
  const int m = int(M), k = int(K);
  switch (fmt) {
    case MXFP4:
      return x_f32 ? quant::launch<MXFP4, true, false>(x, codes, scales, m, k, st)
                   : quant::launch<MXFP4, false, false>(x, codes, scales, m, k, st);
    case MXFP8_E4M3:
      return x_f32 ? quant::launch<MXFP8_E4M3, true, false>(x, codes, scales, m, k, st)
                   : quant::launch<MXFP8_E4M3, false, false>(x, codes, scales, m, k, st);
    case MXFP8_E5M2:
      return x_f32 ? quant::launch<MXFP8_E5M2, true, false>(x, codes, scales, m, k, st)
                   : quant::launch<MXFP8_E5M2, false, false>(x, codes, scales, m, k, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quantize_e4m3_atoms(const void* x, void* codes, void* atoms, int64_t M, int64_t K,
                                       cudaStream_t st) {
  return quant::launch<MXFP8_E4M3, false, true>(x, codes, atoms, int(M), int(K), st);
}

cudaError_t launch_quantize_mxfp4_atoms(const void* x, void* codes, void* atoms, int64_t M, int64_t K,
                                        cudaStream_t st) {
  return quant::launch<MXFP4, false, true>(x, codes, atoms, int(M), int(K), st);
}

// CTAs of the maxima pass: ~16 KiB of X each, at most NV_PARTIALS
int quantize_nvfp4_partials(int64_t M, int64_t K) {
  const int64_t c = (M * K * 2 + 16383) / 16384;
  return int(c < quant::NV_PARTIALS ? (c > 0 ? c : 1) : quant::NV_PARTIALS);
}

cudaError_t launch_quantize_nvfp4_atoms(const void* x, void* codes, void* atoms, float* partials, float* g_out,
                                        int64_t M, int64_t K, cudaStream_t st) {
  const int m = int(M), k = int(K), np = quantize_nvfp4_partials(M, K);
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(unsigned(np));
  lc.blockDim = dim3(256);
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&lc, quant::amax_partial_kernel, static_cast<const __nv_bfloat16*>(x), m, k,
                                     partials);
  if (e != cudaSuccess) return e;
  const int rows = (m + 127) / 128 * 128;
  const int64_t warps = int64_t(rows) * ((k / 32 + 31) / 32);
  lc.gridDim = dim3(unsigned((warps + 7) / 8));
  return cudaLaunchKernelEx(&lc, quant::quantize_nv_atoms_kernel, static_cast<const __nv_bfloat16*>(x),
                            static_cast<uint8_t*>(codes), static_cast<uint8_t*>(atoms),
                            static_cast<const float*>(partials), np, g_out, m, k);
}

}  // namespace qfmt_dev
