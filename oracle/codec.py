"""Oracle element and scale codecs (TEST INFRASTRUCTURE ONLY).

Plain, slow-but-obvious decoders built code-by-code from the format formulas,
and nearest-value encoders written from the definition of round-to-nearest-even
with saturation.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` may import this package; the library never does.

Sources (page title, then the section it comes from):

* E2M1 (fp4): metaltile-std ``src/mlx/fp_quantized_mma.rs``, module header
  "fp4 E2M1 codebook": layout [sign:1][exp:2][mantissa:1], magnitudes
  {0, .5, 1, 1.5, 2, 3, 4, 6}.  metaltile PR #250, codec commit ("E2M1 fp4
  codebook ... + midpoint-threshold encode").
* E4M3: same module header, "fp8 E4M3 dequant": normal 2^(e-7)(1+m/8),
  subnormal 2^-6 * m/8, sign 1-2(code>>7).  PR #250 codec commit: PyTorch-style,
  saturating at +-448, no infinity.  Reading taken: S.1111.111 is the only NaN
  encoding and exponent 15 is otherwise finite (that is what "+-448 with no
  inf" requires; 0x7E = 448).
* E5M2: PR #250 codec commit: the high byte of an IEEE half; the encoder
  saturates finite inputs (maximum finite 57344).
* E8M0: PR #250 codec commit: power-of-two block scale 2^(bits-127).  Reading
  taken for the code the formula leaves open: 255 is NaN (OCP MX convention).
* bf16 (int4-affine scale and bias): IEEE-style binary16 with 8 exponent bits.

Parity pins for every function here live in ``tests/test_oracle_codec.py``.
"""
from __future__ import annotations

import math

import numpy as np

# --------------------------------------------------------------------------
# Decoders: one exact Python float per code, straight from the formulas.
# --------------------------------------------------------------------------


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code: [s:1][e:2][m:1], bias 1, subnormal at e = 0."""
    sign = -1.0 if (code >> 3) & 1 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = m * 0.5                      # subnormal: m * 2^(1-1) * 1/2
    else:
        mag = 2.0 ** (e - 1) * (1.0 + m / 2.0)
    return sign * mag                      # code 8 gives -0.0


def e4m3_value(code: int) -> float:
    """Value of an 8-bit E4M3 code (bias 7, no infinity, only S.1111.111 is NaN)."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return sign * (m / 8.0) * 2.0 ** -6     # subnormal: 2^-6 * m/8
    return sign * 2.0 ** (e - 7) * (1.0 + m / 8.0)


def e5m2_value(code: int) -> float:
    """Value of an 8-bit E5M2 code (bias 15, IEEE specials at exponent 31)."""
    sign = -1.0 if (code >> 7) & 1 else 1.0
    e = (code >> 2) & 31
    m = code & 3
    if e == 31:
        return sign * math.inf if m == 0 else math.nan
    if e == 0:
        return sign * (m / 4.0) * 2.0 ** -14    # subnormal: 2^-14 * m/4
    return sign * 2.0 ** (e - 15) * (1.0 + m / 4.0)


def e8m0_value(code: int) -> float:
    """Value of an E8M0 scale byte: 2^(code - 127); 255 is NaN."""
    if code == 255:
        return math.nan
    return 2.0 ** (code - 127)


def bf16_value(bits: int) -> float:
    """Value of a bfloat16 bit pattern (8 exponent bits, bias 127, 7 mantissa bits)."""
    sign = -1.0 if (bits >> 15) & 1 else 1.0
    e = (bits >> 7) & 255
    m = bits & 127
    if e == 255:
        return sign * math.inf if m == 0 else math.nan
    if e == 0:
        return sign * (m / 128.0) * 2.0 ** -126
    return sign * 2.0 ** (e - 127) * (1.0 + m / 128.0)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E5M2_TABLE = np.array([e5m2_value(c) for c in range(256)], dtype=np.float64)
E8M0_TABLE = np.array([e8m0_value(c) for c in range(256)], dtype=np.float64)

E2M1_MAX = 6.0
E4M3_MAX = 448.0
E5M2_MAX = 57344.0


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """Vector bf16 decode to float64 through the per-code formula (65536-entry table)."""
    return _BF16_TABLE[np.asarray(bits, dtype=np.uint16)]


_BF16_TABLE = np.array([bf16_value(b) for b in range(65536)], dtype=np.float64)

# --------------------------------------------------------------------------
# Encoders: nearest representable value, ties to the even code, saturating.
# --------------------------------------------------------------------------


def _positive_grid(table: np.ndarray, n_codes_per_sign: int):
    """(values, codes) of the finite non-negative codes, ascending."""
    vals = table[:n_codes_per_sign]
    codes = np.arange(n_codes_per_sign)
    keep = np.isfinite(vals)
    vals, codes = vals[keep], codes[keep]
    order = np.argsort(vals, kind="stable")
    return vals[order], codes[order]


_GRIDS = {
    "e2m1": (_positive_grid(E2M1_TABLE, 8), 0x8),
    "e4m3": (_positive_grid(E4M3_TABLE, 128), 0x80),
    "e5m2": (_positive_grid(E5M2_TABLE, 128), 0x80),
}


def encode_rne_sat(v: np.ndarray, fmt: str) -> np.ndarray:
    """Encode float32 values to ``fmt`` codes ("e2m1", "e4m3", "e5m2").

    Round to nearest; on an exact tie pick the even code (mantissa LSB 0);
    magnitudes above the largest finite value saturate to it; the sign code
    bit copies the sign bit of the input (so -0.0 and small negatives that
    round to zero give the sign-set zero code).  Inputs must not be NaN.
    """
    (vals, codes), sign_bit = _GRIDS[fmt]
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v.astype(np.float64))
    hi_i = np.minimum(np.searchsorted(vals, a, side="left"), len(vals) - 1)
    lo_i = np.maximum(hi_i - 1, 0)
    lo, hi = vals[lo_i], vals[hi_i]
    d_lo, d_hi = a - lo, hi - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi_i] % 2 == 0))
    pick_hi |= a >= hi                       # exact hit or saturation
    out = np.where(pick_hi, codes[hi_i], codes[lo_i]).astype(np.uint8)
    out |= np.where(np.signbit(v), sign_bit, 0).astype(np.uint8)
    return out


def e8m0_encode_ceil(s: np.ndarray) -> np.ndarray:
    """E8M0 code of the smallest power of two >= s, for finite float32 s > 0.

    ceil(log2 s) is read exactly off the float32 bits: for a normal s with
    biased exponent E and mantissa M it is E-127, plus one when M != 0; for a
    subnormal s = M * 2^-149 it is ceil(log2 M) - 149.  The exponent is clamped
    to [-127, 127] and stored with bias 127 (so 254 is the largest code used).
    """
    s = np.asarray(s, dtype=np.float32)
    bits = s.view(np.uint32).astype(np.int64)
    E = (bits >> 23) & 0xFF
    M = bits & 0x7FFFFF
    e_norm = E - 127 + (M != 0)
    frac, ex = np.frexp(np.maximum(M, 1).astype(np.float64))   # M = frac * 2^ex
    e_sub = np.where(frac == 0.5, ex - 1, ex) - 149
    e = np.where(E == 0, e_sub, e_norm)
    e = np.clip(e, -127, 127)
    return (e + 127).astype(np.uint8)


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); uint16 bits.

    Written from the definition: the two bfloat16 neighbours of v are the
    float32 pattern truncated to its top 16 bits and the next pattern up; take
    the nearer one, the one with an even last bit on a tie.  Finite inputs only.
    """
    v = np.asarray(v, dtype=np.float32)
    u = v.view(np.uint32).astype(np.uint64)
    down = (u >> 16) << 16
    up = down + (1 << 16)
    rem = u - down                                  # distance above the lower neighbour (in f32 ulps)
    half = 1 << 15
    take_up = (rem > half) | ((rem == half) & (((down >> 16) & 1) == 1))
    return (np.where(take_up, up, down) >> 16).astype(np.uint16)
