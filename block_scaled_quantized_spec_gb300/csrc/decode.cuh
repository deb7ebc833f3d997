// Device-side element and scale decoders for the block-scaled formats.
//
// Two families:
//  * exact float32 decoders (dequant kernel, float32-activation path): each
//    code becomes its exact value; products with the block scale round once.
//  * bf16-pair decoders feeding tensor-core fragments: a 32-bit word of codes
//    becomes bf16x2 registers holding the *scaled* weights.  Which two codes
//    share a register is chosen to keep the decode short; callers pair the
//    activations the same way (any permutation of k that is applied to both
//    operands leaves a dot product unchanged).
//
// Element formats: metaltile-std src/mlx/fp_quantized_mma.rs header ("fp4 E2M1
// codebook", "fp8 E4M3 dequant"); metaltile PR #250 codec commit (E4M3 with
// +-448 saturation and no infinity, E5M2 = high byte of an IEEE half, E8M0 =
// 2^(bits-127)); int4 affine w = scale * q + bias (metaltile-std
// tests/qmm_gpu_correctness.rs, cpu_qmm_reference).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qfmt_dev {

enum Fmt {
  MXFP4 = 1, NVFP4 = 2, MXFP8_E4M3 = 3, MXFP8_E5M2 = 4, NVFP8 = 5, INT4_AFFINE = 6, NVFP8_F16 = 7, MXINT8 = 8,
  INT8 = 9, INT8_F16 = 10, INT4 = 11, INT4_F16 = 12, MXFP4X2 = 13, MXINT4 = 14,
  FP4 = 15, FP4_F16 = 16, FP8_E4M3 = 17, FP8_E4M3_F16 = 18, FP8_E5M2 = 19, FP8_E5M2_F16 = 20
};

template <int F> struct FmtTraits;
template <> struct FmtTraits<MXFP4> { static constexpr bool four = true; static constexpr int block = 32; static constexpr int sbytes = 1; };
template <> struct FmtTraits<NVFP4> { static constexpr bool four = true; static constexpr int block = 16; static constexpr int sbytes = 1; };
template <> struct FmtTraits<MXFP8_E4M3> { static constexpr bool four = false; static constexpr int block = 32; static constexpr int sbytes = 1; };
template <> struct FmtTraits<MXFP8_E5M2> { static constexpr bool four = false; static constexpr int block = 32; static constexpr int sbytes = 1; };
template <> struct FmtTraits<NVFP8> { static constexpr bool four = false; static constexpr int block = 16; static constexpr int sbytes = 4; };
template <> struct FmtTraits<INT4_AFFINE> { static constexpr bool four = true; static constexpr int block = 64; static constexpr int sbytes = 4; };
template <> struct FmtTraits<NVFP8_F16> { static constexpr bool four = false; static constexpr int block = 16; static constexpr int sbytes = 2; };
template <> struct FmtTraits<MXINT8> { static constexpr bool four = false; static constexpr int block = 32; static constexpr int sbytes = 1; };
template <> struct FmtTraits<INT8> { static constexpr bool four = false; static constexpr int block = 64; static constexpr int sbytes = 4; };
template <> struct FmtTraits<INT8_F16> { static constexpr bool four = false; static constexpr int block = 64; static constexpr int sbytes = 2; };
template <> struct FmtTraits<INT4> { static constexpr bool four = true; static constexpr int block = 64; static constexpr int sbytes = 4; };
template <> struct FmtTraits<INT4_F16> { static constexpr bool four = true; static constexpr int block = 64; static constexpr int sbytes = 2; };
// mxfp4x2 as the GEMVs see it: 2N rows of E2M1 codes (row 2n the residual
// plane 0 of output row n, row 2n + 1 its plane 1) with a float32 scale per
// 32, an output the sum of its two rows' products; the GEMM decodes both
// planes of an output row into one weight (decode_x2_hilo).
template <> struct FmtTraits<MXFP4X2> { static constexpr bool four = true; static constexpr int block = 32; static constexpr int sbytes = 4; };
template <> struct FmtTraits<MXINT4> { static constexpr bool four = true; static constexpr int block = 32; static constexpr int sbytes = 1; };
// the legacy float formats: an E2M1 / E4M3 / E5M2 element under a float32 (or
// IEEE half) scale per 32
template <> struct FmtTraits<FP4> { static constexpr bool four = true; static constexpr int block = 32; static constexpr int sbytes = 4; };
template <> struct FmtTraits<FP4_F16> { static constexpr bool four = true; static constexpr int block = 32; static constexpr int sbytes = 2; };
template <> struct FmtTraits<FP8_E4M3> { static constexpr bool four = false; static constexpr int block = 32; static constexpr int sbytes = 4; };
template <> struct FmtTraits<FP8_E4M3_F16> { static constexpr bool four = false; static constexpr int block = 32; static constexpr int sbytes = 2; };
template <> struct FmtTraits<FP8_E5M2> { static constexpr bool four = false; static constexpr int block = 32; static constexpr int sbytes = 4; };
template <> struct FmtTraits<FP8_E5M2_F16> { static constexpr bool four = false; static constexpr int block = 32; static constexpr int sbytes = 2; };

// 8-bit elements under an E8M0 scale per 32 (mxfp8 E4M3/E5M2, mxint8), and
// every E8M0-scaled format (those and mxfp4)
template <int F>
constexpr bool is_mx8() { return F == MXFP8_E4M3 || F == MXFP8_E5M2 || F == MXINT8; }
// 4-bit elements under an E8M0 scale per 32 (mxfp4's E2M1, mxint4's signed nibble)
template <int F>
constexpr bool is_mx4() { return F == MXFP4 || F == MXINT4; }
template <int F>
constexpr bool is_e8m0() { return is_mx4<F>() || is_mx8<F>(); }

// 8-bit elements under a float block scale (float32 or IEEE half): nvfp8 and
// its twin (E4M3, per 16), symmetric int8 and its twin (per 64)
template <int F>
constexpr bool is_fs8() {
  return F == NVFP8 || F == NVFP8_F16 || F == INT8 || F == INT8_F16 || F == FP8_E4M3 || F == FP8_E4M3_F16 ||
         F == FP8_E5M2 || F == FP8_E5M2_F16;
}

// E5M2 elements (under any scale)
template <int F>
constexpr bool is_e5m2() { return F == MXFP8_E5M2 || F == FP8_E5M2 || F == FP8_E5M2_F16; }

// E2M1 elements under a float scale per 32: the legacy fp4 (float32 or half
// scale) and the residual planes of mxfp4x2
template <int F>
constexpr bool is_fp4f() { return F == FP4 || F == FP4_F16 || F == MXFP4X2; }

// signed-int8 elements (under an E8M0 or a float scale)
template <int F>
constexpr bool is_int8() { return F == MXINT8 || F == INT8 || F == INT8_F16; }

// 4-bit integer elements with one (scale, bias) per group of 64: int4 affine
// (stored bf16 pair), and the symmetric int4 / int4_f16 (float32 / half
// scale, bias -8 s on the code with its sign bit flipped, see i4_u)
template <int F>
constexpr bool is_i4() { return F == INT4_AFFINE || F == INT4 || F == INT4_F16; }
template <int F>
constexpr bool is_i4sym() { return F == INT4 || F == INT4_F16; }
inline constexpr bool fmt_is_i4(int f) { return f == INT4_AFFINE || f == INT4 || f == INT4_F16; }
inline constexpr bool fmt_is_four(int f) {
  return f == MXFP4 || f == NVFP4 || f == MXFP4X2 || f == MXINT4 || f == FP4 || f == FP4_F16 || fmt_is_i4(f);
}

// A read-only value from global memory (G) or any state space (a copy in
// shared memory).
template <bool G, typename T>
__device__ __forceinline__ T ld_ro(const T* p) {
  if constexpr (G) return __ldg(p);
  else return *p;
}

// Block scale idx of a float-scaled array as float32: the stored float32, or
// the (exact) float32 of the stored IEEE half.
template <int F, bool G = true>
__device__ __forceinline__ float float_scale(const uint8_t* scales, int64_t idx) {
  if constexpr (FmtTraits<F>::sbytes == 4) return ld_ro<G>(reinterpret_cast<const float*>(scales) + idx);
  else return __half2float(__ushort_as_half(ld_ro<G>(reinterpret_cast<const unsigned short*>(scales) + idx)));
}

// Raw scale word of group idx of a 4-bit integer format: int4 affine's
// (scale, bias) bf16 pair, the float32 bits, or the half bits (zero-extended).
template <int F, bool G = true>
__device__ __forceinline__ uint32_t i4_word(const uint8_t* scales, int64_t idx) {
  if constexpr (FmtTraits<F>::sbytes == 2) return ld_ro<G>(reinterpret_cast<const unsigned short*>(scales) + idx);
  else return ld_ro<G>(reinterpret_cast<const uint32_t*>(scales) + idx);
}

// (scale, bias) of a group from its raw word, for the unsigned u of i4_u:
// w = s * u + b.  Symmetric: u = q + 8, so b = -8 s.
template <int F>
__device__ __forceinline__ void i4_scale_bias(uint32_t wd, float& s, float& b) {
  if constexpr (F == INT4_AFFINE) {
    s = __uint_as_float(wd << 16);
    b = __uint_as_float(wd & 0xFFFF0000u);
  } else {
    s = FmtTraits<F>::sbytes == 4 ? __uint_as_float(wd) : __half2float(__ushort_as_half((unsigned short)wd));
    b = -8.0f * s;
  }
}

// 8 nibble codes as the unsigned u the affine decode works on: a symmetric
// two's-complement nibble q becomes u = q + 8 by flipping its sign bit.
template <int F>
__device__ __forceinline__ uint32_t i4_u(uint32_t w) {
  if constexpr (is_i4sym<F>() || F == MXINT4) return w ^ 0x88888888u;
  else return w;
}

// ------------------------------------------------------------------ exact ---

__device__ __forceinline__ float e2m1_f32(uint32_t c) {
  // magnitude index i = [e1 e0 m]: i = 1 is 0.5 (subnormal), i >= 2 is
  // 2^(e-1) * (1 + m/2): float32 exponent 126 + e, mantissa msb m.
  const uint32_t i = c & 7u;
  const uint32_t mag = i < 2u ? (i ? 0x3F000000u : 0u) : (((126u + (i >> 1)) << 23) | ((i & 1u) << 22));
  return __uint_as_float(mag | ((c & 8u) << 28));
}

__device__ __forceinline__ float e4m3_f32(uint32_t c) {
  const uint32_t e = (c >> 3) & 15u, m = c & 7u;
  float mag;
  if ((c & 0x7Fu) == 0x7Fu) mag = __uint_as_float(0x7FC00000u);           // the only NaN
  else if (e == 0u) mag = __fmul_rn(float(m), 0.001953125f);              // m * 2^-9
  else mag = __uint_as_float(((e + 120u) << 23) | (m << 20));             // 2^(e-7) (1 + m/8)
  return (c & 0x80u) ? -mag : mag;
}

__device__ __forceinline__ float e5m2_f32(uint32_t c) {
  return __half2float(__ushort_as_half((unsigned short)(c << 8)));        // IEEE half high byte
}

__device__ __forceinline__ float e8m0_f32(uint32_t b) {
  if (b == 255u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float(b ? (b << 23) : 0x00400000u);                    // 2^(b-127); b=0 subnormal
}

__device__ __forceinline__ float bf16bits_f32(uint32_t h) { return __uint_as_float(h << 16); }

// ------------------------------------------------------------ bf16 pairs ---

// Start [p, p + bytes) towards L2, trimmed to the whole 16-byte units inside
// the range: the bulk prefetch takes 16-byte aligned addresses and sizes (code
// rows always are; a row of block scales need not be).
__device__ __forceinline__ void prefetch_l2(const void* p, uint64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uintptr_t s = (a + 15) & ~uintptr_t(15), e = (a + bytes) & ~uintptr_t(15);
  if (e > s) asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(s), "r"(uint32_t(e - s)) : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t bf16x2_splat(uint32_t h) { return (h & 0xFFFFu) * 0x00010001u; }

// bf16 bits of 2^(b-127) for an E8M0 byte (bf16 shares float32's exponent
// field): b << 7, with b = 0 the subnormal 2^-127 and b = 255 a NaN.
__device__ __forceinline__ uint32_t e8m0_bf16(uint32_t b) {
  return b == 255u ? 0x7FC0u : (b ? (b << 7) : 0x0040u);
}

// 8 E2M1 codes (code i at bits 4i) -> bf16x2 {c0,c4} {c1,c5} {c2,c6} {c3,c7}.
// Magnitudes come from two 8-entry byte tables (low and high byte of the bf16
// value of {0,.5,1,1.5,2,3,4,6}) indexed by prmt; the sign bit of each code is
// moved to bit 15 / 31 of its half.
__device__ __forceinline__ void e2m1x8_bf16(uint32_t w, uint32_t r[4]) {
  const uint32_t LO0 = 0xC0800000u, LO1 = 0xC0804000u;   // low bytes, entries 0-3 and 4-7
  const uint32_t HI0 = 0x3F3F3F00u, HI1 = 0x40404040u;   // high bytes
  const uint32_t m = w & 0x77777777u;
  const uint32_t s1 = prmt(m, 0u, 0x0020u);  // nibbles c0 c1 c4 c5
  const uint32_t s2 = prmt(m, 0u, 0x0031u);  // nibbles c2 c3 c6 c7
  const uint32_t l1 = prmt(LO0, LO1, s1), h1 = prmt(HI0, HI1, s1);
  const uint32_t l2 = prmt(LO0, LO1, s2), h2 = prmt(HI0, HI1, s2);
  r[0] = prmt(l1, h1, 0x6240u) | ((w << 12) & 0x80008000u);
  r[1] = prmt(l1, h1, 0x7351u) | ((w << 8) & 0x80008000u);
  r[2] = prmt(l2, h2, 0x6240u) | ((w << 4) & 0x80008000u);
  r[3] = prmt(l2, h2, 0x7351u) | (w & 0x80008000u);
}

// 8 signed two's-complement nibbles -> bf16x2 {q0,q4} {q1,q5} {q2,q6} {q3,q7}
// (the pairing of e2m1x8_bf16), exact: the nibble with its sign bit flipped
// is u = q + 8, 0x4300 | u the bf16 of 128 + u, less 136.
__device__ __forceinline__ void sint4x8_bf16(uint32_t w, uint32_t r[4]) {
  const uint32_t t = w ^ 0x88888888u;
  #pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t u = ((t >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r[j]) : "r"(u), "r"(0x43084308u));
  }
}

// 8 signed two's-complement nibbles (code i at bits 4i) -> f16x2 (q0,q1)
// (q2,q3) (q4,q5) (q6,q7), exact: byte i spread to both halves, the low half
// keeps its low nibble under the exponent of 1024 (1024 + u), the high half
// its high nibble four bits up (1024 + 16 u); one fma by (1, 1/16) and
// (-1032, -72) leaves u - 8 = q in each half (u: the nibble, sign bit flipped).
__device__ __forceinline__ void sint4x8_f16(uint32_t w, uint32_t r[4]) {
  const uint32_t t = w ^ 0x88888888u;
  #pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t b = prmt(t, 0u, 0x4040u | (uint32_t(i) * 0x0101u));   // byte i in bytes 0 and 2
    const uint32_t y = (b & 0x00F0000Fu) | 0x64006400u;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r[i]) : "r"(y), "r"(0x2C003C00u), "r"(0xD480E408u));
  }
}

// 8 unsigned 4-bit q (int4 affine) -> bf16x2 {q0,q4} {q1,q5} {q2,q6} {q3,q7},
// each finished as fma(q, scale, bias) in bf16 (one rounding).  0x4300 | q is
// the bf16 of 128 + q, from which 128 is subtracted exactly.
__device__ __forceinline__ void int4x8_affine_bf16(uint32_t w, uint32_t s2, uint32_t b2, uint32_t r[4]) {
  const uint32_t k128 = 0x43004300u;
  #pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t t = ((w >> (4 * j)) & 0x000F000Fu) | k128;
    uint32_t q;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(q) : "r"(t), "r"(k128));
    r[j] = hfma2(q, s2, b2);
  }
}

// 4 E4M3 codes (code i in byte i) -> bf16x2 {c0,c2} {c1,c3} holding the
// value times 2^-120: the 7 magnitude bits land in the low exponent and the
// top mantissa bits of a bf16, which represents every E4M3 value (subnormals
// included) scaled by 2^(7-127).
__device__ __forceinline__ void e4m3x4_bf16_raw(uint32_t w, uint32_t r[2]) {
  r[0] = ((w << 4) & 0x07F007F0u) | ((w << 8) & 0x80008000u);
  r[1] = ((w >> 4) & 0x07F007F0u) | (w & 0x80008000u);
}

// 4 E5M2 codes -> bf16x2 {c0,c2} {c1,c3} holding value times 2^-112.
__device__ __forceinline__ void e5m2x4_bf16_raw(uint32_t w, uint32_t r[2]) {
  r[0] = ((w << 5) & 0x0FE00FE0u) | ((w << 8) & 0x80008000u);
  r[1] = ((w >> 3) & 0x0FE00FE0u) | (w & 0x80008000u);
}

// The codes these bit placements do not map to their value: the E4M3 NaNs
// (S.1111.111) and the E5M2 infinities and NaNs (S.11111.mm).  Bit 7 of byte i
// of the result is set when code i of `w` is one (no carry crosses a byte).
template <int F>
__device__ __forceinline__ uint32_t special8_mask(uint32_t w) {
  if constexpr (is_e5m2<F>()) return ((w & 0x7C7C7C7Cu) + 0x04040404u) & 0x80808080u;
  else return ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
}

// 4 signed-int8 codes -> bf16x2 {c0,c2} {c1,c3}, exact: each byte with its
// sign bit flipped is 128 + q, placed under the float32 exponent of 2^23 and
// rebased by 2^23 + 128 in float32, then packed (|q| <= 128 is exact in bf16).
__device__ __forceinline__ void int8x4_bf16(uint32_t w, uint32_t r[2]) {
  const uint32_t t = w ^ 0x80808080u;
  float f[4];
  #pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = __fsub_rn(__uint_as_float(0x4B000000u | ((t >> (8 * i)) & 0xFFu)), 8388736.0f);
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r[0]) : "f"(f[2]), "f"(f[0]));
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r[1]) : "f"(f[3]), "f"(f[1]));
}

// 4 8-bit codes (code i in byte i) -> f16x2 (c0,c1) (c2,c3), exact: E4M3 and
// E5M2 by the hardware conversions; a signed int8 as the f16 1152 + q (its
// byte with the sign bit flipped, under the exponent of 1024) less 1152.
template <int F>
__device__ __forceinline__ void elem8x4_f16(uint32_t w, uint32_t* r) {
  if constexpr (is_int8<F>()) {
    const uint32_t t = w ^ 0x80808080u;
    const uint32_t a = prmt(t, 0x64u, 0x4140u), b = prmt(t, 0x64u, 0x4342u);
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r[0]) : "r"(a), "r"(0x64806480u));
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r[1]) : "r"(b), "r"(0x64806480u));
  } else if constexpr (is_e5m2<F>()) {
    asm("{.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, h0;\n\tcvt.rn.f16x2.e5m2x2 %1, h1;}"
        : "=r"(r[0]), "=r"(r[1]) : "r"(w));
  } else {
    asm("{.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;}"
        : "=r"(r[0]), "=r"(r[1]) : "r"(w));
  }
}

// bf16 bits of 2^e for -133 <= e <= 127.
__device__ __forceinline__ uint32_t pow2_bf16(int e) {
  return e >= -126 ? uint32_t(e + 127) << 7 : (0x40u >> (-127 - e));
}

// Two floats -> f16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float f16x2_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFFu))); }
__device__ __forceinline__ float f16x2_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

__device__ __forceinline__ uint32_t f32_to_bf16bits(float f) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// ------------------------------------------------------ 16-byte pieces ---
// A piece is 16 bytes of one row's codes: 32 four-bit or 16 eight-bit codes,
// always inside one scale block (mx: 1 block / half a block, nvfp4: 2 blocks,
// int4 affine: half a group, nvfp8: 1 block).

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
  if constexpr (is_e8m0<F>()) {
    s.a = __ldg(scales + base + k0 / 32);
  } else if constexpr (F == NVFP4) {
    s.a = __ldg(reinterpret_cast<const unsigned short*>(scales + base + k0 / 16));
  } else if constexpr (is_fs8<F>() || is_fp4f<F>()) {
    s.a = __float_as_uint(float_scale<F>(scales, base + k0 / FmtTraits<F>::block));
  } else {
    s.a = i4_word<F>(scales, base + k0 / 64);
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
  if constexpr (F == MXFP4 || F == NVFP4 || F == MXINT4) {
    uint32_t sc0, sc1;
    if constexpr (is_mx4<F>()) {
      sc0 = sc1 = bf16x2_splat(e8m0_bf16(ps.a));
    } else {
      sc0 = bf16x2_splat(f32_to_bf16bits(e4m3_f32(ps.a & 0xFFu)));
      sc1 = bf16x2_splat(f32_to_bf16bits(e4m3_f32(ps.a >> 8)));
    }
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t r[4];
      if constexpr (F == MXINT4) sint4x8_bf16(w[j], r);
      else e2m1x8_bf16(w[j], r);
      const uint32_t sc = j < 2 ? sc0 : sc1;
      A[2 * j][0] = hmul2(r[0], sc);
      A[2 * j][1] = hmul2(r[1], sc);
      A[2 * j + 1][0] = hmul2(r[2], sc);
      A[2 * j + 1][1] = hmul2(r[3], sc);
    }
  } else if constexpr (is_i4<F>()) {
    static_assert(F == INT4_AFFINE, "the symmetric int4 formats decode through decode_piece_hilo");
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
    if constexpr (is_mx8<F>()) {
      constexpr int gap = F == MXFP8_E4M3 ? 120 : (F == MXFP8_E5M2 ? 112 : 0);   // int8: the exact value
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
    } else {  // nvfp8 (either scale storage): the float32 scale rounded once to bf16
      static_assert(!is_int8<F>(), "float-scaled int8 decodes through decode_piece_hilo");
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
      else if constexpr (F == MXINT8) int8x4_bf16(w[j], r);
      else e4m3x4_bf16_raw(w[j], r);
      A[j][0] = hmul2(r[0], m1);
      A[j][1] = hmul2(r[1], m1);
      if (two) {
        A[j][0] = hmul2(A[j][0], m2);
        A[j][1] = hmul2(A[j][1], m2);
      }
    }
    if constexpr (!is_int8<F>()) {
      // a NaN / Inf code (outside the packer's range; one test per piece):
      // its value times the block scale in float32, rounded to bf16
      if (special8_mask<F>(w[0]) | special8_mask<F>(w[1]) | special8_mask<F>(w[2]) | special8_mask<F>(w[3])) {
        const float s = is_mx8<F>() ? e8m0_f32(ps.a) : __uint_as_float(ps.a);
        #pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t sm = special8_mask<F>(w[j]);
          #pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (!(sm & (0x80u << (8 * i)))) continue;
            const uint32_t c = (w[j] >> (8 * i)) & 0xFFu;
            const uint32_t h = f32_to_bf16bits(__fmul_rn(is_e5m2<F>() ? e5m2_f32(c) : e4m3_f32(c), s));
            uint32_t& dst = A[j][i & 1];
            dst = (i & 2) ? ((dst & 0x0000FFFFu) | (h << 16)) : ((dst & 0xFFFF0000u) | h);
          }
        }
      }
    }
  }
}

// The same piece as bf16 pairs in natural k order: 4-bit -> 16 registers
// (word j gives registers 4j..4j+3 = codes 8j..8j+7), 8-bit -> 8 registers.
template <int F>
__device__ __forceinline__ void decode_piece_natural(const uint4& v, const PieceScale& ps,
                                                     uint32_t out[FmtTraits<F>::four ? 16 : 8]) {
  uint32_t A[FmtTraits<F>::four ? 8 : 4][2];
  decode_piece<F>(v, ps, A);
  if constexpr (FmtTraits<F>::four) {
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[4 * j + 0] = prmt(A[2 * j][0], A[2 * j][1], 0x5410u);          // (c0, c1)
      out[4 * j + 1] = prmt(A[2 * j + 1][0], A[2 * j + 1][1], 0x5410u);  // (c2, c3)
      out[4 * j + 2] = prmt(A[2 * j][0], A[2 * j][1], 0x7632u);          // (c4, c5)
      out[4 * j + 3] = prmt(A[2 * j + 1][0], A[2 * j + 1][1], 0x7632u);  // (c6, c7)
    }
  } else {
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[2 * j + 0] = prmt(A[j][0], A[j][1], 0x5410u);                  // (c0, c1)
      out[2 * j + 1] = prmt(A[j][0], A[j][1], 0x7632u);                  // (c2, c3)
    }
  }
}

// ----------------------------------------------------- hi/lo bf16 splits ---
// nvfp8 (E4M3 x float32 scale) and int4 affine (scale * q + bias) weights are
// not exact in bf16.  Where a kernel cannot apply the block scale to float32
// partial sums, the float32 weight v is carried as hi + lo with hi = bf16(v)
// and lo = bf16(v - hi) (the subtraction is exact): |v - hi - lo| <= 2^-17 |v|.

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

__device__ __forceinline__ void split_bf16x2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16x2(a, b);
  lo = pack_bf16x2(__fsub_rn(a, __uint_as_float(hi << 16)), __fsub_rn(b, __uint_as_float(hi & 0xFFFF0000u)));
}

// One piece of 32 k of an mxfp4x2 row, both residual planes (a: plane 0, b:
// plane 1, 16 bytes each) and their float32 block scales (ps.a, ps.b): the
// weight s0 e2m1(q0) + s1 e2m1(q1) (one fma, one rounding) as hi/lo bf16 pairs
// in natural k order (16 registers each).
__device__ __forceinline__ void decode_x2_hilo(const uint4& va, const uint4& vb, const PieceScale& ps, uint32_t* hi,
                                               uint32_t* lo) {
  const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
  const float s0 = __uint_as_float(ps.a), s1 = __uint_as_float(ps.b);
  #pragma unroll
  for (int j = 0; j < 4; ++j) {
    #pragma unroll
    for (int p = 0; p < 4; ++p) {
      const uint32_t ba = (wa[j] >> (8 * p)) & 0xFFu, bb = (wb[j] >> (8 * p)) & 0xFFu;
      const float w0 = __fmaf_rn(e2m1_f32(bb & 0xFu), s1, __fmul_rn(e2m1_f32(ba & 0xFu), s0));
      const float w1 = __fmaf_rn(e2m1_f32(bb >> 4), s1, __fmul_rn(e2m1_f32(ba >> 4), s0));
      split_bf16x2(w0, w1, hi[4 * j + p], lo[4 * j + p]);
    }
  }
}

// One 16-byte piece of a float-scaled 8-bit (16 codes) or int4-affine (32
// codes) row as hi/lo bf16 pairs in natural k order (8 or 16 registers each).
template <int F>
__device__ __forceinline__ void decode_piece_hilo(const uint4& v, const PieceScale& ps, uint32_t* hi, uint32_t* lo) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (is_fp4f<F>()) {   // 32 E2M1 codes (a residual plane of mxfp4x2) times their float block scale
    const float s = __uint_as_float(ps.a);
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      #pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t byte = (w[j] >> (8 * p)) & 0xFFu;
        split_bf16x2(__fmul_rn(e2m1_f32(byte & 0xFu), s), __fmul_rn(e2m1_f32(byte >> 4), s), hi[4 * j + p], lo[4 * j + p]);
      }
    }
  } else if constexpr (is_fs8<F>()) {
    const float s = __uint_as_float(ps.a);
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t r[2], e02, e13;
      if constexpr (is_int8<F>()) {
        int8x4_bf16(w[j], r);                                                       // exact values
        e02 = r[0];
        e13 = r[1];
      } else if constexpr (is_e5m2<F>()) {
        e5m2x4_bf16_raw(w[j], r);
        e02 = hmul2(r[0], 0x77807780u);                                             // x 2^112: exact values
        e13 = hmul2(r[1], 0x77807780u);
      } else {
        e4m3x4_bf16_raw(w[j], r);
        e02 = hmul2(r[0], 0x7B807B80u);                                             // x 2^120: exact values
        e13 = hmul2(r[1], 0x7B807B80u);
      }
      float v0 = __fmul_rn(__uint_as_float(e02 << 16), s), v2 = __fmul_rn(__uint_as_float(e02 & 0xFFFF0000u), s);
      float v1 = __fmul_rn(__uint_as_float(e13 << 16), s), v3 = __fmul_rn(__uint_as_float(e13 & 0xFFFF0000u), s);
      if constexpr (!is_int8<F>()) {
        if (special8_mask<F>(w[j])) {   // NaN / Inf codes: their value times the scale
          auto fix = [&](float& v, uint32_t c) {
            if (special8_mask<F>(c)) v = __fmul_rn(is_e5m2<F>() ? e5m2_f32(c) : e4m3_f32(c), s);
          };
          fix(v0, w[j] & 0xFFu);
          fix(v1, (w[j] >> 8) & 0xFFu);
          fix(v2, (w[j] >> 16) & 0xFFu);
          fix(v3, w[j] >> 24);
        }
      }
      split_bf16x2(v0, v1, hi[2 * j], lo[2 * j]);
      split_bf16x2(v2, v3, hi[2 * j + 1], lo[2 * j + 1]);
    }
  } else {   // int4 affine: fma(s, q, b); symmetric int4: s * q (one rounding either way)
    float s, b;
    i4_scale_bias<F>(ps.a, s, b);
    #pragma unroll
    for (int j = 0; j < 4; ++j) {
      #pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t byte = (w[j] >> (8 * p)) & 0xFFu;
        float q0 = __fsub_rn(__uint_as_float(0x4B000000u | (byte & 0xFu)), 8388608.0f);
        float q1 = __fsub_rn(__uint_as_float(0x4B000000u | (byte >> 4)), 8388608.0f);
        if constexpr (is_i4sym<F>()) {   // the sign-extended nibble
          q0 = q0 >= 8.0f ? q0 - 16.0f : q0;
          q1 = q1 >= 8.0f ? q1 - 16.0f : q1;
          split_bf16x2(__fmul_rn(s, q0), __fmul_rn(s, q1), hi[4 * j + p], lo[4 * j + p]);
        } else {
          split_bf16x2(__fmaf_rn(s, q0, b), __fmaf_rn(s, q1, b), hi[4 * j + p], lo[4 * j + p]);
        }
      }
    }
  }
}

}  // namespace qfmt_dev
