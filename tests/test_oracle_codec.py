"""Pins for the oracle's element/scale codecs against the pages, mathematics and libraries.

Every decoder is compared exhaustively over its whole code space with a source
that does not share the oracle's formula code: the codebook the pages print,
the pages' own alternative integer formula, numpy/torch reinterpretations and
casts.  Encoders are checked at every representable value and every midpoint
between neighbours, against a brute-force nearest search and library casts.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import codec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    assert rows, name
    return rows


def _same(a, b):
    """Equal as IEEE values, NaN == NaN, and the sign of zero must agree."""
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


# ---------------------------------------------------------------- E2M1 ----

def test_e2m1_codebook_matches_pages():
    rows = _golden("e2m1_codebook.txt")
    assert len(rows) == 16
    for code, val in rows:
        assert _same(codec.e2m1_value(int(code)), float(val)), code
        assert _same(codec.E2M1_TABLE[int(code)], float(val)), code


def test_e2m1_two_m_int_formula():
    # fp_quantized_mma.rs header: code3 = c & 7; exp = code3 >> 1, mant = code3 & 1;
    # subnormal two_m = mant, normal two_m = (mant + 2) * 2^(exp-1); value = sign * two_m / 2.
    for c in range(16):
        code3, exp, mant = c & 7, (c & 7) >> 1, c & 1
        two_m = mant if exp == 0 else (mant + 2) * 2 ** (exp - 1)
        sign = 1 - 2 * (c >> 3)
        v = sign * two_m / 2.0
        assert codec.e2m1_value(c) == v, c


def test_e2m1_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    lib = np.arange(16, dtype=np.uint8).view(ml.float4_e2m1fn).astype(np.float64)
    for c in range(16):
        assert _same(codec.E2M1_TABLE[c], lib[c]), c


# ---------------------------------------------------------- E4M3 / E5M2 ----

def test_fp8_scale_anchors_match_pages():
    tables = {"e4m3": codec.E4M3_TABLE, "e5m2": codec.E5M2_TABLE, "e8m0": codec.E8M0_TABLE}
    rows = _golden("fp8_scale_anchors.txt")
    for fmt, code, val in rows:
        c = int(code, 0)
        assert _same(tables[fmt][c], float(val)), (fmt, code)


def test_e4m3_matches_torch_all_codes():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        assert _same(codec.E4M3_TABLE[c], lib[c]), hex(c)
    assert np.isnan(codec.E4M3_TABLE[0x7F]) and np.isnan(codec.E4M3_TABLE[0xFF])
    assert np.nanmax(codec.E4M3_TABLE) == 448.0        # +-448 saturation, no inf
    assert not np.any(np.isinf(codec.E4M3_TABLE))


def test_e4m3_binade_formula_from_page():
    # fp_quantized_mma.rs: e = (code7 >> 3) - 7, m = code7 & 7; normal 2^e (1 + m/8);
    # subnormal (e_raw = 0) 2^-6 * m/8; sign 1 - 2 (code >> 7).  Checked in exact rationals.
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        c7 = c & 0x7F
        e_raw, m = c7 >> 3, c7 & 7
        mag = Fraction(m, 8) * Fraction(1, 64) if e_raw == 0 else Fraction(2) ** (e_raw - 7) * (1 + Fraction(m, 8))
        val = (1 - 2 * (c >> 7)) * mag
        assert Fraction(codec.E4M3_TABLE[c]) == val, hex(c)


def test_e5m2_is_half_high_byte():
    halves = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).double().numpy()
    for c in range(256):
        assert _same(codec.E5M2_TABLE[c], halves[c]), hex(c)
        assert _same(codec.E5M2_TABLE[c], lib[c]), hex(c)
    assert np.nanmax(codec.E5M2_TABLE[np.isfinite(codec.E5M2_TABLE)]) == 57344.0


def test_e8m0_matches_torch_and_formula():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    for c in range(256):
        assert _same(codec.E8M0_TABLE[c], lib[c]), c
        if c < 255:
            assert Fraction(codec.E8M0_TABLE[c]) == Fraction(2) ** (c - 127)
    # code 0 is 2^-127: a float32 subnormal, not zero
    assert np.float32(codec.E8M0_TABLE[0]) == np.float32(2.0 ** -127) > 0


def test_bf16_decode_matches_bit_reinterpretation():
    bits = np.arange(65536, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        lib = (bits << 16).view(np.float32).astype(np.float64)
    ours = codec.decode_bf16(bits.astype(np.uint16))
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all()
    finite = ~np.isnan(lib)
    assert (np.signbit(ours[finite]) == np.signbit(lib[finite])).all()


def test_bf16_round_matches_torch_cast():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-38).astype(np.float32),       # subnormals
        rng.integers(0, 2 ** 31, 20000, dtype=np.uint32).view(np.float32),
    ])
    v = v[np.isfinite(v)]
    ours = codec.bf16_round(v)
    lib = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)


# -------------------------------------------------------------- encoders ----

_ENC = [("e2m1", codec.E2M1_TABLE, 8, 0x8, 6.0),
        ("e4m3", codec.E4M3_TABLE, 128, 0x80, 448.0),
        ("e5m2", codec.E5M2_TABLE, 128, 0x80, 57344.0)]


def _brute_nearest(a, table, n_pos):
    """Brute force over every finite non-negative code: nearest, tie -> even code."""
    best = None
    for c in range(n_pos):
        t = table[c]
        if not np.isfinite(t):
            continue
        d = abs(Fraction(float(a)) - Fraction(float(t)))
        if best is None or d < best[0] or (d == best[0] and c % 2 == 0 and best[1] % 2 == 1):
            best = (d, c)
    return best[1]


@pytest.mark.parametrize("fmt,table,n_pos,sbit,maxf", _ENC)
def test_encode_representable_values_and_midpoints(fmt, table, n_pos, sbit, maxf):
    vals = sorted({float(table[c]) for c in range(n_pos) if np.isfinite(table[c])})
    probes = []
    for v in vals:
        probes.append(np.float32(v))
    for lo, hi in zip(vals[:-1], vals[1:]):
        mid = np.float32((lo + hi) / 2)             # exact: the grids have few mantissa bits
        assert float(mid) == (lo + hi) / 2
        probes += [mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0))]
    probes = np.array(probes, dtype=np.float32)
    for sign in (1.0, -1.0):
        p = (probes * np.float32(sign)).astype(np.float32)
        got = codec.encode_rne_sat(p, fmt)
        for v, g in zip(p, got):
            want = _brute_nearest(abs(v), table, n_pos) | (sbit if np.signbit(v) else 0)
            assert g == want, (fmt, float(v), int(g), want)


@pytest.mark.parametrize("fmt,table,n_pos,sbit,maxf", _ENC)
def test_encode_saturates_and_signs(fmt, table, n_pos, sbit, maxf):
    big = np.array([maxf * 1.5, 1e30, 3.0e38], dtype=np.float32)
    maxcode = int(np.nanargmax(np.where(np.isfinite(table[:n_pos]), table[:n_pos], -1)))
    assert (codec.encode_rne_sat(big, fmt) == maxcode).all()
    assert (codec.encode_rne_sat(-big, fmt) == (maxcode | sbit)).all()
    assert codec.encode_rne_sat(np.array([-0.0], np.float32), fmt)[0] == sbit
    assert codec.encode_rne_sat(np.array([0.0], np.float32), fmt)[0] == 0


def test_encode_matches_torch_fp8_casts_in_range():
    rng = np.random.default_rng(2)
    for fmt, tdt, lim in (("e4m3", torch.float8_e4m3fn, 448.0), ("e5m2", torch.float8_e5m2, 57344.0)):
        v = np.concatenate([rng.uniform(-lim, lim, 50000),
                            rng.standard_normal(50000) * 1e-3,
                            rng.standard_normal(50000) * 1e-6]).astype(np.float32)
        ours = codec.encode_rne_sat(v, fmt)
        lib = torch.from_numpy(v.copy()).to(tdt).view(torch.uint8).numpy()
        assert np.array_equal(ours, lib), fmt


def test_encode_matches_ml_dtypes_e2m1():
    ml = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(3)
    v = np.concatenate([rng.uniform(-6, 6, 50000), rng.uniform(-0.3, 0.3, 5000)]).astype(np.float32)
    ours = codec.encode_rne_sat(v, "e2m1")
    lib = v.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
    assert np.array_equal(ours, lib)


def test_e8m0_ceil_log2_exact():
    rng = np.random.default_rng(4)
    s = np.concatenate([
        rng.uniform(1e-3, 1e3, 3000),
        2.0 ** rng.integers(-126, 127, 300),
        np.array([2.0 ** -127, 2.0 ** -140, 1.4e-45, 3e-39, 1e-42]),
        rng.uniform(1e37, 3e38, 100),
    ]).astype(np.float32)
    got = codec.e8m0_encode_ceil(s)
    for x, g in zip(s, got):
        f = Fraction(float(x))
        e = f.numerator.bit_length() - f.denominator.bit_length()   # 2^e near f
        while Fraction(2) ** e < f:
            e += 1
        while Fraction(2) ** (e - 1) >= f:
            e -= 1
        e = max(-127, min(127, e))
        assert int(g) == e + 127, (float(x), int(g), e)
