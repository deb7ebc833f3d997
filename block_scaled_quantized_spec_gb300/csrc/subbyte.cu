// The 2/3/5/6-bit symmetric integer formats (int2/3/5/6, their fp16-scale
// twins, mxint2/3/5/6): dequant and the dequantizing matmul.
//
// A row's codes are one LSB-first bit stream (metaltile PR #250, the
// sub-byte packing commit: a tight bit stream with reads straddling word
// boundaries for widths 3, 5 and 6): code k at bits [k N, k N + N), sign-
// extended from bit N - 1; the value is q * scale, the scale a float32 or
// IEEE half per 64 (the intN path) or an E8M0 byte per 32 (the MXINT axis).
// Since K is a multiple of 32, every 32 codes of a row fill N whole 32-bit
// words: both kernels work in these 32-code units (one thread per unit),
// loading N words and extracting each code with at most one word straddle.
// These formats run on CUDA cores: exact float32 weights (dequant: one
// rounding of q * scale) and, in the matmul, per unit the exact float32 sum
// of q x over 32 codes (q at most 6 bits, x bf16) times the scale.
#include <cuda_runtime.h>

#include "decode.cuh"
#include "kernels.h"

namespace qfmt_dev {
namespace sub {

enum ScaleKind { SK_F32 = 0, SK_F16 = 1, SK_E8M0 = 2 };

template <int SK>
__device__ __forceinline__ float scale_at(const uint8_t* scales, int64_t idx) {
  if constexpr (SK == SK_F32) return __ldg(reinterpret_cast<const float*>(scales) + idx);
  else if constexpr (SK == SK_F16) return __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(scales) + idx)));
  else return e8m0_f32(__ldg(scales + idx));
}

// The 32 codes of one unit (B words), sign-extended.
template <int B>
__device__ __forceinline__ void decode32(const uint32_t (&w)[B], int (&q)[32]) {
  #pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int p = j * B, wi = p >> 5, off = p & 31;
    uint32_t v = w[wi] >> off;
    if (off + B > 32) v |= w[wi + 1] << (32 - off);
    q[j] = int(v << (32 - B)) >> (32 - B);
  }
}

template <int B>
__device__ __forceinline__ void load_unit(const uint8_t* codes, int64_t row, int64_t K, int64_t c, uint32_t (&w)[B]) {
  const uint32_t* p = reinterpret_cast<const uint32_t*>(codes + row * (K * B / 8)) + c * B;
  #pragma unroll
  for (int i = 0; i < B; ++i) w[i] = __ldg(p + i);
}

template <int B, int SK, bool OUT_BF16>
__global__ void __launch_bounds__(256) dequant_bits_kernel(const uint8_t* __restrict__ codes,
                                                           const uint8_t* __restrict__ scales,
                                                           void* __restrict__ out, int64_t N, int64_t K) {
  constexpr int BLK = SK == SK_E8M0 ? 32 : 64;
  const int64_t units = K / 32, total = N * units, nblk = (K + BLK - 1) / BLK;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int64_t u = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; u < total; u += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = u / units, c = u - row * units;
    uint32_t w[B];
    load_unit<B>(codes, row, K, c, w);
    int q[32];
    decode32<B>(w, q);
    const float s = scale_at<SK>(scales, row * nblk + (c * 32) / BLK);
    float o[32];
    #pragma unroll
    for (int j = 0; j < 32; ++j) o[j] = __fmul_rn(float(q[j]), s);
    if constexpr (OUT_BF16) {
      uint4* d = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) + row * K + c * 32);
      #pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t h[4];
        #pragma unroll
        for (int t = 0; t < 4; ++t) h[t] = f32_to_bf16bits(o[8 * i + 2 * t]) | (f32_to_bf16bits(o[8 * i + 2 * t + 1]) << 16);
        d[i] = make_uint4(h[0], h[1], h[2], h[3]);
      }
    } else {
      float4* d = reinterpret_cast<float4*>(static_cast<float*>(out) + row * K + c * 32);
      #pragma unroll
      for (int i = 0; i < 8; ++i) d[i] = make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    }
  }
}

// 32 activations of row m from k0, as float32 (bf16 or float32 storage).
template <bool X_F32>
__device__ __forceinline__ void load_x32(const void* x, int64_t m, int64_t K, int64_t k0, float (&v)[32]) {
  if constexpr (X_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) + m * K + k0);
    #pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 f = __ldg(p + i);
      v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + m * K + k0);
    #pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = __ldg(p + i);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
      #pragma unroll
      for (int t = 0; t < 4; ++t) {
        v[8 * i + 2 * t] = __uint_as_float(ws[t] << 16);
        v[8 * i + 2 * t + 1] = __uint_as_float(ws[t] & 0xFFFF0000u);
      }
    }
  }
}

constexpr int MT = 8;   // activation rows per CTA

// A warp per weight row (4 a CTA), MT activation rows per CTA; lanes stride
// over the row's 32-code units.
template <int B, int SK, bool X_F32>
__global__ void __launch_bounds__(128) qmm_bits_kernel(const uint8_t* __restrict__ codes,
                                                       const uint8_t* __restrict__ scales, const void* __restrict__ x,
                                                       void* __restrict__ out, int out_f32, int M, int N, int K) {
  constexpr int BLK = SK == SK_E8M0 ? 32 : 64;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = blockIdx.x * 4 + warp, m0 = blockIdx.y * MT;
  const int mr = min(MT, M - m0);
  const int64_t units = K / 32, nblk = (K + BLK - 1) / BLK;
  float acc[MT];
  #pragma unroll
  for (int r = 0; r < MT; ++r) acc[r] = 0.0f;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (n < N) {
    for (int64_t c = lane; c < units; c += 32) {
      uint32_t w[B];
      load_unit<B>(codes, n, K, c, w);
      int q[32];
      decode32<B>(w, q);
      const float s = scale_at<SK>(scales, int64_t(n) * nblk + (c * 32) / BLK);
      #pragma unroll
      for (int r = 0; r < MT; ++r) {
        if (r >= mr) break;
        float v[32];
        load_x32<X_F32>(x, m0 + r, K, c * 32, v);
        float d = 0.0f;
        #pragma unroll
        for (int j = 0; j < 32; ++j) d = __fmaf_rn(float(q[j]), v[j], d);
        acc[r] = __fmaf_rn(s, d, acc[r]);
      }
    }
  }
  #pragma unroll
  for (int r = 0; r < MT; ++r) {
    float a = acc[r];
    #pragma unroll
    for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xFFFFFFFFu, a, o);
    if (lane == 0 && n < N && r < mr) {
      const int64_t idx = int64_t(m0 + r) * N + n;
      if (out_f32) static_cast<float*>(out)[idx] = a;
      else static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(a);
    }
  }
}

// M > 4: a CTA (128 threads) takes 32 weight rows (16 pairs) and up to 8
// activation rows and walks K in chunks of 256 (8 units).  Each chunk of X is
// staged once in shared memory as float32 (double-buffered; 36 floats a unit
// so the 8 units a warp reads at once fall in distinct banks) and serves all
// 32 rows.
// Thread t takes row pair t / 8 and unit t % 8 of every chunk: it decodes the
// unit's 32 codes of both rows once and forms, for each activation row, the
// 32-term sums of q x (two partial sums a row) times the unit's scale.  The
// next chunk's codes, scales and activations are loaded while this one is
// computed.  The 8 threads of a row pair meet by shuffles at the end.
constexpr int TM = 8, TROWS = 32, TCK = 256, TUNITS = TCK / 32, TSTRIDE = 36, TTHREADS = 128;

template <int B, int SK, bool X_F32>
__global__ void __launch_bounds__(TTHREADS) qmm_bits_tile_kernel(const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ scales,
                                                            const void* __restrict__ x, void* __restrict__ out,
                                                            int out_f32, int M, int N, int K) {
  constexpr int BLK = SK == SK_E8M0 ? 32 : 64;
  __shared__ __align__(16) float xs[2][TM][TUNITS * TSTRIDE];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int t = threadIdx.x, g = t & 7, pr = t >> 3;
  const int n0 = blockIdx.x * TROWS + 2 * pr, m0 = blockIdx.y * TM;
  const int mr = min(TM, M - m0);
  const int64_t units = K / 32, nblk = (K + BLK - 1) / BLK;
  const int nchunks = int((units + TUNITS - 1) / TUNITS);
  const bool r0ok = n0 < N, r1ok = n0 + 1 < N;
  // activation staging: thread t carries row t / 16, columns (t % 16) * 16 .. + 16 of a chunk
  static_assert(TTHREADS / 16 == TM && TTHREADS / 8 == TROWS / 2, "the thread maps");
  const int xr = t >> 4, xc = (t & 15) * 16;
  float xv[16];
  auto load_x = [&](int c) {
    const int64_t k = int64_t(c) * TCK + xc;
    const bool ok = xr < mr && k < K;                      // K is a multiple of 32: 16 columns all in or all out
    if constexpr (X_F32) {
      const float4* p4 = reinterpret_cast<const float4*>(static_cast<const float*>(x) + int64_t(m0 + xr) * K + k);
      #pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float4 f = ok ? __ldg(p4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        xv[4 * i] = f.x; xv[4 * i + 1] = f.y; xv[4 * i + 2] = f.z; xv[4 * i + 3] = f.w;
      }
    } else {
      const uint4* p4 = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(x) + int64_t(m0 + xr) * K + k);
      #pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 w = ok ? __ldg(p4 + i) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
          xv[8 * i + 2 * j] = __uint_as_float(ws[j] << 16);
          xv[8 * i + 2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
        }
      }
    }
  };
  auto store_x = [&](int buf) {
    if (xr < TM) {
      float* d = &xs[buf][xr][(xc / 32) * TSTRIDE + (xc % 32)];
      #pragma unroll
      for (int i = 0; i < 4; ++i) reinterpret_cast<float4*>(d)[i] = make_float4(xv[4 * i], xv[4 * i + 1], xv[4 * i + 2], xv[4 * i + 3]);
    }
  };
  // this thread's unit of a chunk: codes and scales of both rows
  uint32_t w0[B], w1[B];
  float s0 = 0.f, s1 = 0.f;
  auto load_w = [&](int c, uint32_t (&a)[B], uint32_t (&b)[B], float& sa, float& sb) {
    const int64_t u = int64_t(c) * TUNITS + g;
    const bool in = c < nchunks && u < units;
    #pragma unroll
    for (int i = 0; i < B; ++i) { a[i] = 0u; b[i] = 0u; }
    sa = 0.f;
    sb = 0.f;
    if (in && r0ok) { load_unit<B>(codes, n0, K, u, a); sa = scale_at<SK>(scales, int64_t(n0) * nblk + (u * 32) / BLK); }
    if (in && r1ok) { load_unit<B>(codes, n0 + 1, K, u, b); sb = scale_at<SK>(scales, int64_t(n0 + 1) * nblk + (u * 32) / BLK); }
  };
  float acc0[TM], acc1[TM];
  #pragma unroll
  for (int m = 0; m < TM; ++m) { acc0[m] = 0.f; acc1[m] = 0.f; }
  load_w(0, w0, w1, s0, s1);                               // the weights: before the dependent wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  load_x(0);
  store_x(0);
  __syncthreads();
  for (int c = 0; c < nchunks; ++c) {
    uint32_t nw0[B], nw1[B];
    float ns0, ns1;
    load_w(c + 1, nw0, nw1, ns0, ns1);
    if (c + 1 < nchunks) load_x(c + 1);
    {
      int q0[32], q1[32];
      decode32<B>(w0, q0);
      decode32<B>(w1, q1);
      float f0[32], f1[32];
      #pragma unroll
      for (int j = 0; j < 32; ++j) { f0[j] = float(q0[j]); f1[j] = float(q1[j]); }
      const float* xb = &xs[c & 1][0][g * TSTRIDE];
      #pragma unroll
      for (int m = 0; m < TM; ++m) {
        if (m >= mr) break;
        const float4* xp = reinterpret_cast<const float4*>(xb + m * (TUNITS * TSTRIDE));
        float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 v = xp[i];
          a0 = __fmaf_rn(f0[4 * i], v.x, a0); a1 = __fmaf_rn(f0[4 * i + 1], v.y, a1);
          a0 = __fmaf_rn(f0[4 * i + 2], v.z, a0); a1 = __fmaf_rn(f0[4 * i + 3], v.w, a1);
          b0 = __fmaf_rn(f1[4 * i], v.x, b0); b1 = __fmaf_rn(f1[4 * i + 1], v.y, b1);
          b0 = __fmaf_rn(f1[4 * i + 2], v.z, b0); b1 = __fmaf_rn(f1[4 * i + 3], v.w, b1);
        }
        acc0[m] = __fmaf_rn(s0, a0 + a1, acc0[m]);
        acc1[m] = __fmaf_rn(s1, b0 + b1, acc1[m]);
      }
    }
    if (c + 1 < nchunks) store_x((c + 1) & 1);
    __syncthreads();
    #pragma unroll
    for (int i = 0; i < B; ++i) { w0[i] = nw0[i]; w1[i] = nw1[i]; }
    s0 = ns0;
    s1 = ns1;
  }
  // the 8 threads of a row pair (consecutive lanes) sum their units
  #pragma unroll
  for (int m = 0; m < TM; ++m) {
    #pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      acc0[m] += __shfl_xor_sync(0xFFFFFFFFu, acc0[m], o);
      acc1[m] += __shfl_xor_sync(0xFFFFFFFFu, acc1[m], o);
    }
  }
  if (g == 0) {
    #pragma unroll
    for (int m = 0; m < TM; ++m) {
      if (m >= mr) break;
      const int64_t base = int64_t(m0 + m) * N;
      if (r0ok) {
        if (out_f32) static_cast<float*>(out)[base + n0] = acc0[m];
        else static_cast<__nv_bfloat16*>(out)[base + n0] = __float2bfloat16_rn(acc0[m]);
      }
      if (r1ok) {
        if (out_f32) static_cast<float*>(out)[base + n0 + 1] = acc1[m];
        else static_cast<__nv_bfloat16*>(out)[base + n0 + 1] = __float2bfloat16_rn(acc1[m]);
      }
    }
  }
}

template <int B, int SK>
static cudaError_t dequant_fmt(const void* codes, const void* scales, void* out, bool bf16, int64_t N, int64_t K,
                               cudaStream_t st, int sms) {
  const int64_t total = N * (K / 32);
  int64_t grid = (total + 255) / 256;
  if (grid > int64_t(sms) * 8) grid = int64_t(sms) * 8;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.gridDim = dim3(unsigned(grid));
  lc.blockDim = dim3(256);
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 1;
  auto c = static_cast<const uint8_t*>(codes);
  auto s = static_cast<const uint8_t*>(scales);
  return bf16 ? cudaLaunchKernelEx(&lc, dequant_bits_kernel<B, SK, true>, c, s, out, N, K)
              : cudaLaunchKernelEx(&lc, dequant_bits_kernel<B, SK, false>, c, s, out, N, K);
}

template <int B, int SK>
static cudaError_t qmm_fmt(const void* codes, const void* scales, const void* x, bool x_f32, void* out, bool out_f32,
                           int64_t M, int64_t N, int64_t K, cudaStream_t st) {
  cudaLaunchConfig_t lc = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  auto c = static_cast<const uint8_t*>(codes);
  auto s = static_cast<const uint8_t*>(scales);
  lc.stream = st;
  lc.attrs = at;
  lc.numAttrs = 1;
  if (M > 4) {   // tiles of 32 weight rows x 8 activation rows, X staged in shared memory
    lc.gridDim = dim3(unsigned((N + TROWS - 1) / TROWS), unsigned((M + TM - 1) / TM));
    lc.blockDim = dim3(TTHREADS);
    return x_f32 ? cudaLaunchKernelEx(&lc, qmm_bits_tile_kernel<B, SK, true>, c, s, x, out, int(out_f32), int(M),
                                      int(N), int(K))
                 : cudaLaunchKernelEx(&lc, qmm_bits_tile_kernel<B, SK, false>, c, s, x, out, int(out_f32), int(M),
                                      int(N), int(K));
  }
  lc.gridDim = dim3(unsigned((N + 3) / 4), unsigned((M + MT - 1) / MT));
  lc.blockDim = dim3(128);
  return x_f32 ? cudaLaunchKernelEx(&lc, qmm_bits_kernel<B, SK, true>, c, s, x, out, int(out_f32), int(M), int(N), int(K))
               : cudaLaunchKernelEx(&lc, qmm_bits_kernel<B, SK, false>, c, s, x, out, int(out_f32), int(M), int(N),
                                    int(K));
}

// format id -> (bits, scale kind): ids 21-24 int2/3/5/6 (float32 scale per
// 64), 25-28 their fp16-scale twins, 29-32 mxint2/3/5/6 (E8M0 per 32)
constexpr int FIRST = 21;

}  // namespace sub

bool is_sub_byte(int fmt) { return fmt >= sub::FIRST && fmt < sub::FIRST + 12; }

#define QFMT_SUB_DISPATCH(CALL)                                                      \
  switch (fmt - sub::FIRST) {                                                        \
    case 0: return CALL(2, sub::SK_F32);  case 1: return CALL(3, sub::SK_F32);        \
    case 2: return CALL(5, sub::SK_F32);  case 3: return CALL(6, sub::SK_F32);        \
    case 4: return CALL(2, sub::SK_F16);  case 5: return CALL(3, sub::SK_F16);        \
    case 6: return CALL(5, sub::SK_F16);  case 7: return CALL(6, sub::SK_F16);        \
    case 8: return CALL(2, sub::SK_E8M0); case 9: return CALL(3, sub::SK_E8M0);       \
    case 10: return CALL(5, sub::SK_E8M0); case 11: return CALL(6, sub::SK_E8M0);     \
    default: return cudaErrorInvalidValue;                                           \
  }

cudaError_t launch_dequant_sub(int fmt, const void* codes, const void* scales, void* out, bool out_bf16, int64_t N,
                               int64_t K, cudaStream_t st, int sms) {
#define QFMT_DQ(B, SK) sub::dequant_fmt<B, SK>(codes, scales, out, out_bf16, N, K, st, sms)
  QFMT_SUB_DISPATCH(QFMT_DQ)
#undef QFMT_DQ
}

cudaError_t launch_qmm_sub(int fmt, const void* codes, const void* scales, const void* x, bool x_f32, void* out,
                           bool out_f32, int64_t M, int64_t N, int64_t K, cudaStream_t st) {
#define QFMT_QM(B, SK) sub::qmm_fmt<B, SK>(codes, scales, x, x_f32, out, out_f32, M, N, K, st)
  QFMT_SUB_DISPATCH(QFMT_QM)
#undef QFMT_QM
}

}  // namespace qfmt_dev
