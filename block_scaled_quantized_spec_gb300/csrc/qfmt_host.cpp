// Host side of libqfmt: element/scale encoders, the weight packer, byte-size
// queries and the per-thread error message.
//
// Built with -ffp-contract=off: every float operation rounds once, so the
// packer gives the same bytes on x86-64 and aarch64.
//
// The packer follows metaltile PR #250 (commit "Foundation for the
// spec-conformant nvfp4/mxfp4/mxfp8/nvfp8 formats": per-block amax scaling
// along K, a two-level FP32 global for nvfp4, codes quantized against the
// effective post-encode scale) and rlx-cpu thunk/ops/quant.rs
// (lowp_compute_scales: scale = amax / max_finite, 1.0 for an all-zero
// block; lowp_snap_scale; lowp_quantize: code = encode(x / s), 0 if s == 0).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "qfmt_internal.h"

namespace qfmt {

static thread_local char g_err[512];

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return status;
}

void clear_error() { g_err[0] = '\0'; }

bool valid_format(int fmt) { return fmt >= QFMT_MXFP4 && fmt <= QFMT_MXINT6; }

// Bits per code of the sub-byte integer formats (2, 3, 5, 6); 0 for the rest.
int sub_bits(int fmt) {
  switch (fmt) {
    case QFMT_INT2: case QFMT_INT2_F16: case QFMT_MXINT2: return 2;
    case QFMT_INT3: case QFMT_INT3_F16: case QFMT_MXINT3: return 3;
    case QFMT_INT5: case QFMT_INT5_F16: case QFMT_MXINT5: return 5;
    case QFMT_INT6: case QFMT_INT6_F16: case QFMT_MXINT6: return 6;
    default: return 0;
  }
}

static bool is_mxint_sub(int fmt) { return fmt >= QFMT_MXINT2 && fmt <= QFMT_MXINT6; }
static bool is_f16_sub(int fmt) { return fmt >= QFMT_INT2_F16 && fmt <= QFMT_INT6_F16; }

int block_of(int fmt) {
  switch (fmt) {
    case QFMT_MXFP4: case QFMT_MXFP8_E4M3: case QFMT_MXFP8_E5M2: case QFMT_MXINT8: case QFMT_MXFP4X2:
    case QFMT_MXINT4: case QFMT_FP4: case QFMT_FP4_F16: case QFMT_FP8_E4M3: case QFMT_FP8_E4M3_F16: case QFMT_FP8_E5M2:
    case QFMT_FP8_E5M2_F16: return 32;
    case QFMT_NVFP4: case QFMT_NVFP8: case QFMT_NVFP8_F16: return 16;
    case QFMT_INT4_AFFINE: case QFMT_INT8: case QFMT_INT8_F16: case QFMT_INT4: case QFMT_INT4_F16: return 64;
    default:
      if (sub_bits(fmt)) return is_mxint_sub(fmt) ? 32 : 64;
      return 0;
  }
}

bool is_4bit(int fmt) {
  return fmt == QFMT_MXFP4 || fmt == QFMT_NVFP4 || fmt == QFMT_INT4_AFFINE || fmt == QFMT_INT4 || fmt == QFMT_INT4_F16 ||
         fmt == QFMT_MXINT4 || fmt == QFMT_FP4 || fmt == QFMT_FP4_F16;
}

bool is_sym_int(int fmt) {
  return fmt == QFMT_MXINT8 || fmt == QFMT_INT8 || fmt == QFMT_INT8_F16 || fmt == QFMT_INT4 || fmt == QFMT_INT4_F16 ||
         fmt == QFMT_MXINT4 || sub_bits(fmt) != 0;
}

// Bits per code: 4, 8, or a sub-byte width (mxfp4x2: its two planes, 8 a weight).
int code_bits(int fmt) { return sub_bits(fmt) ? sub_bits(fmt) : (is_4bit(fmt) ? 4 : 8); }

// Largest finite element magnitude: amax / elem_max is the raw block scale.
float elem_max(int fmt) {
  switch (fmt) {
    case QFMT_MXFP4: case QFMT_NVFP4: case QFMT_MXFP4X2: case QFMT_FP4: case QFMT_FP4_F16: return 6.0f;
    case QFMT_MXFP8_E5M2: case QFMT_FP8_E5M2: case QFMT_FP8_E5M2_F16: return 57344.0f;
    case QFMT_MXINT8: case QFMT_INT8: case QFMT_INT8_F16: return 127.0f;
    case QFMT_INT4: case QFMT_INT4_F16: case QFMT_MXINT4: return 7.0f;
    default:
      if (sub_bits(fmt)) return float((1 << (sub_bits(fmt) - 1)) - 1);
      return 448.0f;   // E4M3
  }
}

int scale_entry_bytes(int fmt) {
  if (fmt == QFMT_MXFP4X2) return 8;   // s0 and s1, float32 each (stored as two [nb] runs per row)
  if (fmt == QFMT_NVFP8 || fmt == QFMT_INT4_AFFINE || fmt == QFMT_INT8 || fmt == QFMT_INT4 || fmt == QFMT_FP4 ||
      fmt == QFMT_FP8_E4M3 || fmt == QFMT_FP8_E5M2 || (fmt >= QFMT_INT2 && fmt <= QFMT_INT6))
    return 4;
  if (is_f16_sub(fmt)) return 2;
  return (fmt == QFMT_NVFP8_F16 || fmt == QFMT_INT8_F16 || fmt == QFMT_INT4_F16 || fmt == QFMT_FP4_F16 ||
          fmt == QFMT_FP8_E4M3_F16 || fmt == QFMT_FP8_E5M2_F16)
             ? 2
             : 1;
}

int check_group(int fmt, int group) {
  if (!valid_format(fmt)) return fail(QFMT_EINVAL, "unknown format %d", fmt);
  if (group != 0 && group != block_of(fmt))
    return fail(QFMT_EUNSUPPORTED, "group %d not supported for format %d (block %d)", group, fmt,
                block_of(fmt));
  return QFMT_OK;
}

int check_shape(int fmt, int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return fail(QFMT_ESHAPE, "negative size M=%lld N=%lld K=%lld",
                                           (long long)M, (long long)N, (long long)K);
  // int4 affine (group 64) may end in a ragged group of 32 (ceil(K/64) groups)
  if (K % 32) return fail(QFMT_ESHAPE, "K=%lld must be a multiple of 32", (long long)K);
  // the kernels index rows and columns with 32-bit ints; mxfp4x2 streams 2N code rows
  const int64_t lim = int64_t(1) << 31;
  const int64_t rows = fmt == QFMT_MXFP4X2 ? 2 * N : N;
  if (rows >= lim || M >= lim || K >= lim) return fail(QFMT_ESHAPE, "size of 2^31 or more");
  return QFMT_OK;
}

int check_ptr(const void* p, int align, const char* what) {
  if (!p) return fail(QFMT_EINVAL, "%s is NULL", what);
  if (reinterpret_cast<uintptr_t>(p) % align)
    return fail(QFMT_EALIGN, "%s not %d-byte aligned", what, align);
  return QFMT_OK;
}

// ---------------------------------------------------------------------------
// Element encoders.
// ---------------------------------------------------------------------------

// Round-to-nearest-even into a minifloat with `mbits` mantissa bits and
// exponent bias `bias`, saturating to `max_code` (magnitude code of the largest
// finite value `max_val`).  The quantum of the binade holding |v| (the
// min-normal binade for subnormals) divides |v| exactly, nearbyintf rounds
// ties to even, and the code is (biased exponent << mbits) + (n - 2^mbits):
// a mantissa carry moves into the next exponent by itself, and in the
// subnormal binade the same expression yields the subnormal code n.
static uint32_t encode_minifloat(float v, int mbits, int bias, uint32_t max_code, float max_val,
                                 uint32_t sign_bit) {
  const uint32_t sign = std::signbit(v) ? sign_bit : 0u;
  const float a = std::fabs(v);
  if (!(a < max_val)) return max_code | sign;
  const int min_exp = 1 - bias;
  int e = min_exp;
  if (a >= std::ldexp(1.0f, min_exp)) {
    int ex;
    std::frexp(a, &ex);  // a = f * 2^ex, f in [0.5, 1)
    e = ex - 1;
  }
  const float n = std::nearbyint(a / std::ldexp(1.0f, e - mbits));
  const uint32_t code = (uint32_t(e + bias) << mbits) + uint32_t(n) - (1u << mbits);
  return std::min(code, max_code) | sign;
}

static inline uint32_t enc_e2m1(float v) { return encode_minifloat(v, 1, 1, 0x7, 6.0f, 0x8); }
static inline uint32_t enc_e4m3(float v) { return encode_minifloat(v, 3, 7, 0x7E, 448.0f, 0x80); }
static inline uint32_t enc_e5m2(float v) { return encode_minifloat(v, 2, 15, 0x7B, 57344.0f, 0x80); }
// E2M1 code -> value: magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}, sign bit 3.
static float dec_e2m1(uint32_t c) {
  static const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
  return (c & 0x8u) ? -mag[c & 7u] : mag[c & 7u];
}

static inline uint32_t f32_bits(float f) { uint32_t u; std::memcpy(&u, &f, 4); return u; }
static inline float bits_f32(uint32_t u) { float f; std::memcpy(&f, &u, 4); return f; }

// E4M3 decode (exact in float32); the packer never stores the NaN code.
static float dec_e4m3(uint32_t c) {
  const uint32_t e = (c >> 3) & 15, m = c & 7;
  float mag = (e == 0) ? std::ldexp(float(m), -9) : bits_f32(((e + 120u) << 23) | (m << 20));
  return (c & 0x80) ? -mag : mag;
}

// E8M0 code of the smallest power of two >= s (finite s > 0): ceil(log2 s)
// from the float32 fields, clamped to [-127, 127], biased by 127.
static uint32_t enc_e8m0_ceil(float s) {
  const uint32_t u = f32_bits(s);
  const int E = int((u >> 23) & 0xFF);
  const uint32_t M = u & 0x7FFFFF;
  int e;
  if (E != 0) {
    e = E - 127 + (M != 0);
  } else {
    int lg = 0;                                   // ceil(log2 M), M >= 1
    while ((uint64_t(1) << lg) < M) ++lg;
    e = lg - 149;
  }
  e = std::max(-127, std::min(127, e));
  return uint32_t(e + 127);
}

static float dec_e8m0(uint32_t b) {  // b <= 254
  return b == 0 ? bits_f32(0x00400000u) : bits_f32(b << 23);
}

// float32 -> bfloat16, nearest with ties to even (finite inputs).
static uint16_t bf16_rne(float f) {
  const uint32_t u = f32_bits(f);
  return uint16_t((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}
static float bf16_f32(uint16_t h) { return bits_f32(uint32_t(h) << 16); }

// ---------------------------------------------------------------------------
// Packer.
// ---------------------------------------------------------------------------

template <class F>
static void parallel_rows(int64_t N, F&& body) {
  unsigned hw = std::max(1u, std::thread::hardware_concurrency());
  int64_t nt = std::min<int64_t>(hw, std::max<int64_t>(1, N / 64));
  if (nt <= 1) { body(0, N); return; }
  std::vector<std::thread> ts;
  int64_t per = (N + nt - 1) / nt;
  for (int64_t t = 0; t < nt; ++t) {
    int64_t r0 = t * per, r1 = std::min(N, r0 + per);
    if (r0 >= r1) break;
    ts.emplace_back([&, r0, r1] { body(r0, r1); });
  }
  for (auto& t : ts) t.join();
}

static inline void put_code(uint8_t* row, int64_t k, uint32_t code, bool four_bit) {
  if (!four_bit) { row[k] = uint8_t(code); return; }
  if (k & 1) row[k >> 1] |= uint8_t(code << 4);
  else row[k >> 1] = uint8_t(code & 0xF);
}

// Code k of a row's LSB-first bit stream of `bits`-bit codes (the row's bytes
// zeroed beforehand): bits [k bits, k bits + bits) of the little-endian bit
// sequence, which may straddle two bytes.
static inline void put_bits(uint8_t* row, int64_t k, uint32_t code, int bits) {
  const int64_t p = k * bits;
  const uint32_t v = (code & ((1u << bits) - 1u)) << (p & 7);
  row[p >> 3] |= uint8_t(v);
  if ((p & 7) + bits > 8) row[(p >> 3) + 1] |= uint8_t(v >> 8);
}

}  // namespace qfmt

using namespace qfmt;

extern "C" {

int qfmt_version(void) { return 107; }

const char* qfmt_last_error(void) { return qfmt::g_err; }

int qfmt_block_size(int fmt, int group) {
  clear_error();
  if (check_group(fmt, group) != QFMT_OK) return 0;
  return block_of(fmt);
}

size_t qfmt_codes_bytes(int fmt, int64_t N, int64_t K, int group) {
  clear_error();
  if (check_group(fmt, group) != QFMT_OK || check_shape(fmt, 0, N, K) != QFMT_OK) return SIZE_MAX;
  return size_t(N * K * code_bits(fmt) / 8);
}

size_t qfmt_scales_bytes(int fmt, int64_t N, int64_t K, int group) {
  clear_error();
  if (check_group(fmt, group) != QFMT_OK || check_shape(fmt, 0, N, K) != QFMT_OK) return SIZE_MAX;
  return size_t(N * ((K + block_of(fmt) - 1) / block_of(fmt)) * scale_entry_bytes(fmt));
}

int qfmt_pack(int fmt, const float* W, int64_t N, int64_t K, int group, void* codes,
              void* scales, float* global_scale) {
  clear_error();
  int st = check_group(fmt, group);
  if (st) return st;
  if ((st = check_shape(fmt, 0, N, K))) return st;
  if (N * K > 0 && (!W || !codes || !scales))
    return fail(QFMT_EINVAL, "NULL buffer");
  if (!global_scale) return fail(QFMT_EINVAL, "global_scale is NULL");
  *global_scale = 1.0f;
  if (N == 0 || K == 0) return QFMT_OK;

  const int blk = block_of(fmt);
  const int64_t nb = (K + blk - 1) / blk;   // int4 affine: a ragged last group of K - 64 (nb - 1) values
  const bool four = is_4bit(fmt);
  const int sbits = sub_bits(fmt);
  const int64_t row_bytes = K * code_bits(fmt) / 8;
  uint8_t* cb = static_cast<uint8_t*>(codes);
  if (sbits) std::memset(cb, 0, size_t(N * row_bytes));   // put_bits ORs into zeroed rows
  uint8_t* sb = static_cast<uint8_t*>(scales);

  // Reject NaN/Inf weights up front (the block statistics assume finite input).
  std::atomic<bool> bad{false};
  parallel_rows(N, [&](int64_t r0, int64_t r1) {
    for (int64_t i = r0 * K; i < r1 * K && !bad.load(std::memory_order_relaxed); ++i)
      if (!std::isfinite(W[i])) bad = true;
  });
  if (bad) return fail(QFMT_ENONFINITE, "weights contain NaN or Inf");

  float glob = 1.0f;
  if (fmt == QFMT_NVFP4) {
    std::vector<float> part(std::max<unsigned>(1, std::thread::hardware_concurrency()) * 4, 0.0f);
    std::atomic<int> slot{0};
    parallel_rows(N, [&](int64_t r0, int64_t r1) {
      float m = 0.0f;
      for (int64_t i = r0 * K; i < r1 * K; ++i) m = std::max(m, std::fabs(W[i]));
      part[slot++] = m;
    });
    float amax_t = 0.0f;
    for (float m : part) amax_t = std::max(amax_t, m);
    glob = amax_t > 0.0f ? amax_t / 2688.0f : 1.0f;  // 2688 = 6 * 448
  }

  parallel_rows(N, [&](int64_t r0, int64_t r1) {
    for (int64_t n = r0; n < r1; ++n) {
      const float* w = W + n * K;
      uint8_t* crow = cb + n * row_bytes;
      if (fmt == QFMT_MXFP4X2) {
        // two residual E2M1 levels per block: level 0 packs w with s0 = amax/6,
        // level 1 the float32 residual r = w - s0 e2m1(q0) with s1 = amax(r)/6;
        // plane p's codes at byte p K/2 of the row, its scales at float p nb
        float* srow = reinterpret_cast<float*>(sb) + n * 2 * nb;
        std::vector<float> r(w, w + K);
        for (int p = 0; p < 2; ++p) {
          for (int64_t b = 0; b < nb; ++b) {
            float* rb = r.data() + b * blk;
            float amax = 0.0f;
            for (int j = 0; j < blk; ++j) amax = std::max(amax, std::fabs(rb[j]));
            const float sc = amax > 0.0f ? amax / 6.0f : 1.0f;
            if (!std::isfinite(sc)) { bad = true; continue; }
            srow[p * nb + b] = sc;
            for (int j = 0; j < blk; ++j) {
              const uint32_t code = sc != 0.0f ? enc_e2m1(rb[j] / sc) : 0u;
              put_code(crow + p * (K / 2), b * blk + j, code, true);
              const float approx = sc * dec_e2m1(code);
              rb[j] = rb[j] - approx;
            }
          }
        }
        continue;
      }
      for (int64_t b = 0; b < nb; ++b) {
        const float* wb = w + b * blk;
        const int len = int(std::min<int64_t>(blk, K - b * blk));
        if (fmt == QFMT_INT4_AFFINE) {
          float mn = wb[0], mx = wb[0];
          for (int j = 1; j < len; ++j) { mn = std::min(mn, wb[j]); mx = std::max(mx, wb[j]); }
          float s = (mx - mn) / 15.0f;
          if (s == 0.0f) s = 1.0f;
          if (!std::isfinite(s)) { bad = true; continue; }
          const uint16_t sh = bf16_rne(s), bh = bf16_rne(mn);
          const float sf = bf16_f32(sh), bfv = bf16_f32(bh);
          uint16_t* pr = reinterpret_cast<uint16_t*>(sb + (n * nb + b) * 4);
          pr[0] = sh;
          pr[1] = bh;
          for (int j = 0; j < len; ++j) {
            uint32_t q = 0;
            if (sf != 0.0f) {
              float v = std::round((wb[j] - bfv) / sf);
              q = uint32_t(std::max(0.0f, std::min(15.0f, v)));
            }
            put_code(crow, b * blk + j, q, true);
          }
          continue;
        }
        float amax = 0.0f;
        for (int j = 0; j < len; ++j) amax = std::max(amax, std::fabs(wb[j]));
        float eff;
        switch (fmt) {
          case QFMT_MXFP4: case QFMT_MXFP8_E4M3: case QFMT_MXFP8_E5M2: case QFMT_MXINT8: case QFMT_MXINT4:
          case QFMT_MXINT2: case QFMT_MXINT3: case QFMT_MXINT5: case QFMT_MXINT6: {
            const float s = amax > 0.0f ? amax / elem_max(fmt) : 1.0f;
            const uint32_t code = enc_e8m0_ceil(s);
            sb[n * nb + b] = uint8_t(code);
            eff = dec_e8m0(code);
            break;
          }
          case QFMT_NVFP4: {
            const uint32_t u = amax > 0.0f ? enc_e4m3((amax / 6.0f) / glob) : 0x38u;
            sb[n * nb + b] = uint8_t(u);
            eff = dec_e4m3(u) * glob;
            break;
          }
          case QFMT_NVFP8_F16: case QFMT_INT8_F16: case QFMT_INT4_F16: case QFMT_FP4_F16: case QFMT_FP8_E4M3_F16:
          case QFMT_FP8_E5M2_F16: case QFMT_INT2_F16: case QFMT_INT3_F16: case QFMT_INT5_F16:
          case QFMT_INT6_F16: {  // an IEEE half, rounded to nearest even
            const float s = amax > 0.0f ? amax / elem_max(fmt) : 1.0f;
            const _Float16 h = static_cast<_Float16>(s);
            std::memcpy(sb + (n * nb + b) * 2, &h, 2);
            eff = static_cast<float>(h);
            break;
          }
          default: {  // QFMT_NVFP8, QFMT_INT8, QFMT_INT4 and the legacy float formats: the float32 scale raw
            const float s = amax > 0.0f ? amax / elem_max(fmt) : 1.0f;
            std::memcpy(sb + (n * nb + b) * 4, &s, 4);
            eff = s;
            break;
          }
        }
        if (!std::isfinite(eff)) { bad = true; continue; }
        for (int j = 0; j < len; ++j) {
          uint32_t code = 0;
          if (eff != 0.0f) {
            const float v = wb[j] / eff;
            if (is_sym_int(fmt)) {  // symmetric: round half away from zero, clamp to +-max, two's complement
              const float qm = elem_max(fmt);
              code = uint32_t(uint8_t(int8_t(std::max(-qm, std::min(qm, std::round(v)))))) &
                     ((1u << code_bits(fmt)) - 1u);
              if (sbits) put_bits(crow, b * blk + j, code, sbits);
              else put_code(crow, b * blk + j, code, four);
              continue;
            }
            const bool e5 = fmt == QFMT_MXFP8_E5M2 || fmt == QFMT_FP8_E5M2 || fmt == QFMT_FP8_E5M2_F16;
            const bool e2 = fmt == QFMT_MXFP4 || fmt == QFMT_NVFP4 || fmt == QFMT_FP4 || fmt == QFMT_FP4_F16;
            code = e5 ? enc_e5m2(v) : e2 ? enc_e2m1(v) : enc_e4m3(v);
          }
          // (eff == 0: a half scale that underflowed; the code is 0)
          if (sbits) put_bits(crow, b * blk + j, code, sbits);
          else put_code(crow, b * blk + j, code, four);
        }
      }
    }
  });
  if (bad) return fail(QFMT_ENONFINITE, "a block scale overflows float32");
  *global_scale = glob;
  return QFMT_OK;
}

}  // extern "C"
