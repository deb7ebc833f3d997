"""Pins for the oracle packer and dequant: byte layout, zero blocks, exact round trips,
value idempotence, nearest-grid quantization, and the per-format direction floors."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from block_scaled_quantized_spec_gb300 import synth
from oracle import codec, pack, reference

FMTS = pack.FORMATS
MX = ("mxfp4", "mxfp8_e4m3", "mxfp8_e5m2")          # float elements under E8M0 (mxint8 separately)


def _elem_values_lib(fmt, codes_nk):
    """Element values from library reinterpretations (not the oracle's tables)."""
    if fmt in ("mxfp4", "nvfp4", "fp4", "fp4_f16"):
        c = codes_nk.astype(np.int64)
        c3 = c & 7
        e, m = c3 >> 1, c3 & 1
        two_m = np.where(e == 0, m, (m + 2) * (2 ** np.maximum(e - 1, 0)))
        return (1 - 2 * (c >> 3)) * two_m / 2.0
    if fmt in ("mxfp8_e4m3", "nvfp8", "nvfp8_f16", "fp8_e4m3", "fp8_e4m3_f16"):
        return torch.from_numpy(codes_nk.astype(np.uint8)).view(torch.float8_e4m3fn).double().numpy()
    if fmt in ("mxfp8_e5m2", "fp8_e5m2", "fp8_e5m2_f16"):
        return (codes_nk.astype(np.uint16) << 8).view(np.float16).astype(np.float64)
    if fmt in ("mxint8", "int8", "int8_f16"):
        return torch.from_numpy(codes_nk.astype(np.uint8)).view(torch.int8).double().numpy()
    if fmt in ("int4", "int4_f16", "mxint4"):     # the nibble in the top of a byte, arithmetic shift back down
        return torch.from_numpy((codes_nk.astype(np.uint8) << 4).astype(np.uint8)).view(torch.int8).double().numpy() / 16
    return codes_nk.astype(np.float64)


def test_byte_sizes():
    # PR #250: 4-bit codes pack 8 per u32 (two per byte), 8-bit one byte per code;
    # one scale per block: E8M0/E4M3 one byte, nvfp8 FP32, int4 affine bf16 scale + bf16 bias.
    n, k = 12, 256
    w = synth.weights(n, k, seed=5)
    for fmt in FMTS:
        c, s, g = pack.pack(fmt, w)
        bits = pack.ELEM_BITS[fmt]
        assert c.nbytes == n * k * bits // 8 == pack.codes_nbytes(fmt, n, k)
        per_scale = {"nvfp8": 4, "int4_affine": 4, "nvfp8_f16": 2, "int8": 4, "int8_f16": 2, "int4": 4,
                     "int4_f16": 2, "mxfp4x2": 8, "fp4": 4, "fp4_f16": 2, "fp8_e4m3": 4, "fp8_e4m3_f16": 2,
                     "fp8_e5m2": 4, "fp8_e5m2_f16": 2, "int2": 4, "int3": 4, "int5": 4, "int6": 4,
                     "int2_f16": 2, "int3_f16": 2, "int5_f16": 2, "int6_f16": 2}.get(fmt, 1)
        assert s.nbytes == n * (k // pack.BLOCK[fmt]) * per_scale == pack.scales_nbytes(fmt, n, k)
        assert c.dtype == np.uint8 and s.dtype == np.uint8 and isinstance(g, np.float32)


def test_nibble_order_is_lsb_first():
    # Element 2i in the low nibble of byte i (8 codes per little-endian u32, code k at bits 4k).
    n, k = 1, 32
    w = np.zeros((n, k), np.float32)
    w[0, 0] = 6.0       # max code 7 at element 0 -> low nibble of byte 0
    w[0, 3] = -3.0      # element 3 -> high nibble of byte 1
    c, s, _ = pack.pack("mxfp4", w)
    assert s[0, 0] == 127                       # amax 6 -> scale 2^0
    assert c[0, 0] == 0x07 and c[0, 1] == 0xD0  # -3.0 = code 0xD
    u32 = c.view("<u4")[0, 0]
    assert (u32 >> 0) & 0xF == 7 and (u32 >> 12) & 0xF == 0xD


def test_zero_blocks():
    # rlx-cpu lowp_compute_scales: an all-zero block gets scale 1.0; lowp_quantize: codes 0.
    n, k = 2, 128
    w = np.zeros((n, k), np.float32)
    for fmt in FMTS:
        c, s, g = pack.pack(fmt, w)
        assert not c.any(), fmt
        if fmt in MX or fmt.startswith("mxint"):
            assert (s == 127).all()
        elif fmt == "nvfp4":
            assert (s == 0x38).all() and g == 1.0
        elif fmt in ("nvfp8", "int8", "int4", "mxfp4x2", "fp4", "fp8_e4m3", "fp8_e5m2", "int2", "int3", "int5", "int6"):
            assert (s.view(np.float32) == 1.0).all()
        elif fmt.endswith("_f16"):
            assert (s.view(np.float16) == 1.0).all()
        else:
            pair = s.view(np.uint16).reshape(n, -1, 2)
            assert (pair[..., 0] == 0x3F80).all() and (pair[..., 1] == 0).all()
        assert not reference.dequant_exact(fmt, c, s, g, n, k).any()


@pytest.mark.parametrize("fmt", MX)
def test_exactly_representable_roundtrip_mx(fmt):
    # W built as code values x 2^e with the block maximum at the element max: pack must
    # return exactly those codes and scales (the snapped scale equals amax / max_finite).
    rng = np.random.default_rng(7)
    n, k, blk = 8, 256, 32
    elem = {"mxfp4": "e2m1", "mxfp8_e4m3": "e4m3", "mxfp8_e5m2": "e5m2"}[fmt]
    table = {"e2m1": codec.E2M1_TABLE, "e4m3": codec.E4M3_TABLE, "e5m2": codec.E5M2_TABLE}[elem]
    ncode = 16 if elem == "e2m1" else 256
    finite = np.array([c for c in range(ncode) if np.isfinite(table[c])])
    maxcode = int(finite[np.argmax(table[finite])])
    codes = rng.choice(finite, size=(n, k))
    codes[:, ::blk] = maxcode
    e = rng.integers(-20, 10, size=(n, k // blk))
    vals = _elem_values_lib(fmt, codes).reshape(n, k // blk, blk) * (2.0 ** e)[..., None]
    w = vals.reshape(n, k).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), vals.reshape(n, k))
    c, s, g = pack.pack(fmt, w)
    assert np.array_equal(s, (e + 127).astype(np.uint8))
    got = reference.unpack_codes(fmt, c, n, k)
    # +0 and -0 both decode to zero; compare values, then the bytes away from zeros
    assert np.array_equal(_elem_values_lib(fmt, got), _elem_values_lib(fmt, codes))
    nz = _elem_values_lib(fmt, codes) != 0
    assert np.array_equal(got[nz], codes[nz].astype(np.uint8))


@pytest.mark.parametrize("fmt", [f for f in FMTS if f != "mxfp4x2"])   # a re-packed residual moves s0
def test_value_idempotence(fmt):
    # Packing the dequantized weights again reproduces the same values (the codes
    # quantized against the effective scale are self-consistent, PR #250).
    n, k = 32, 512
    w = synth.weights(n, k, seed=11, outliers=(fmt == "nvfp4"))
    c, s, g = pack.pack(fmt, w)
    wd = reference.dequant_f32(fmt, c, s, g, n, k)
    c2, s2, g2 = pack.pack(fmt, wd)
    wd2 = reference.dequant_f32(fmt, c2, s2, g2, n, k)
    if fmt == "int4_affine":
        # the affine grid re-fit on dequantized data may move by one bf16 rounding of min/scale
        scale = codec.decode_bf16(s.view(np.uint16).reshape(n, -1, 2)[..., 0])
        tol = np.repeat(scale, 64, axis=1) * 0.51 + 1e-30
        assert (np.abs(wd2.astype(np.float64) - wd) <= tol).all()
    else:
        assert np.array_equal(wd, wd2)


FLOORS = {"mxfp4": 0.98, "nvfp4": 0.98, "int4_affine": 0.99,
          "mxfp8_e5m2": 0.995, "mxfp8_e4m3": 0.999, "nvfp8": 0.999, "nvfp8_f16": 0.999, "mxint8": 0.999,
          "int8": 0.9999, "int8_f16": 0.9999, "int4": 0.99, "int4_f16": 0.99, "mxfp4x2": 0.9999, "mxint4": 0.98,
          "fp4": 0.98, "fp4_f16": 0.98, "fp8_e4m3": 0.999, "fp8_e4m3_f16": 0.999, "fp8_e5m2": 0.995,
          "fp8_e5m2_f16": 0.995, "int2": 0.75, "int3": 0.95, "int5": 0.998, "int6": 0.9995, "int2_f16": 0.75,
          "int3_f16": 0.95, "int5_f16": 0.998, "int6_f16": 0.9995, "mxint2": 0.6, "mxint3": 0.92, "mxint5": 0.997,
          "mxint6": 0.999}


@pytest.mark.parametrize("fmt", FMTS)
def test_cosine_floor(fmt):
    # PR #250: pack -> dequant judged by direction (cosine) against a per-format floor.
    n, k = 64, 1024
    w = synth.weights(n, k, seed=13, outliers=(fmt == "nvfp4"))
    c, s, g = pack.pack(fmt, w)
    wd = reference.dequant_exact(fmt, c, s, g, n, k).ravel()
    wv = w.astype(np.float64).ravel()
    cos = wv @ wd / np.linalg.norm(wv) / np.linalg.norm(wd)
    assert cos >= FLOORS[fmt], (fmt, cos)


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4", "mxfp8_e4m3", "mxfp8_e5m2", "nvfp8", "nvfp8_f16"])
def test_elements_are_nearest_grid_points(fmt):
    # Brute force over every code: each dequantized element is a closest point
    # of {value(code) * eff} to w (ties allowed either way), eff the block's effective scale.
    n, k = 2, 64
    w = synth.weights(n, k, seed=17, outliers=(fmt == "nvfp4"))
    c, s, g = pack.pack(fmt, w)
    blk = pack.BLOCK[fmt]
    mult, _ = reference.block_scales(fmt, s, g, n, k)
    eff = np.repeat(mult, blk, axis=1)
    if fmt == "nvfp4":
        eff = (eff.astype(np.float32) * g).astype(np.float64)   # effective scale is rounded to f32
    ncode = 16 if fmt in ("mxfp4", "nvfp4") else 256
    allv = _elem_values_lib(fmt, np.arange(ncode))
    allv = allv[np.isfinite(allv)]
    got = _elem_values_lib(fmt, reference.unpack_codes(fmt, c, n, k))
    for i in range(n):
        for j in range(k):
            wf = Fraction(float(w[i, j]))
            ef = Fraction(float(eff[i, j]))
            best = min(abs(wf - Fraction(float(v)) * ef) for v in allv)
            assert abs(wf - Fraction(float(got[i, j])) * ef) == best, (fmt, i, j)


def test_nvfp4_two_level_global():
    # PR #250: the global FP32 scale lets the E4M3 micro-scales fit +-448 -> the block
    # holding the tensor maximum gets micro-scale 448 (code 0x7E); global = amax / (6 * 448).
    n, k = 16, 256
    w = synth.weights(n, k, seed=19, outliers=True)
    c, s, g = pack.pack("nvfp4", w)
    amax = np.float32(np.max(np.abs(w)))
    assert g == np.float32(amax / np.float32(2688.0))
    nb = k // 16
    blk_max = np.abs(w).reshape(n, nb, 16).max(axis=2)
    i, j = np.unravel_index(np.argmax(blk_max), blk_max.shape)
    assert s.reshape(n, nb)[i, j] == 0x7E
    assert not np.isin(s, [0x7F, 0xFF]).any()


def test_no_special_codes_emitted():
    n, k = 64, 512
    for fmt in ("mxfp8_e4m3", "nvfp8", "mxfp8_e5m2", "nvfp8_f16"):
        w = synth.weights(n, k, seed=23) * np.float32(1e3)
        c, s, g = pack.pack(fmt, w)
        if fmt == "mxfp8_e5m2":
            assert not (((c >> 2) & 31) == 31).any()
        else:
            assert not ((c & 0x7F) == 0x7F).any()
        assert np.isfinite(reference.dequant_exact(fmt, c, s, g, n, k)).all()


def test_int4_affine_quantizer():
    # scale = (max - min)/15 and bias = min, both rounded to bf16; q = round-half-away
    # of (w - bias)/scale clamped to [0, 15]; error at most half a step (plus the
    # bf16 rounding of bias/scale pushed through the clamp).
    n, k = 16, 256
    w = synth.weights(n, k, seed=29)
    c, s, g = pack.pack("int4_affine", w)
    pair = s.view(np.uint16).reshape(n, k // 64, 2)
    sc = codec.decode_bf16(pair[..., 0])
    bi = codec.decode_bf16(pair[..., 1])
    wb = w.reshape(n, k // 64, 64).astype(np.float64)
    assert (np.abs(bi - wb.min(axis=2)) <= np.abs(wb.min(axis=2)) * 2.0 ** -8).all()
    true_s = (wb.max(axis=2) - wb.min(axis=2)) / 15
    assert (np.abs(sc - true_s) <= true_s * 2.0 ** -8 * 1.01).all()
    wd = reference.dequant_exact("int4_affine", c, s, g, n, k).reshape(n, k // 64, 64)
    assert (np.abs(wd - wb) <= sc[..., None] * 0.5 * 1.05 + np.abs(bi)[..., None] * 2.0 ** -7).all()


def test_pack_rejects_bad_input():
    with pytest.raises(ValueError):
        pack.pack("mxfp4", np.full((1, 32), np.nan, np.float32))
    with pytest.raises(ValueError):
        pack.pack("mxfp4", np.zeros((1, 48), np.float32))
    with pytest.raises(ValueError):
        pack.pack("bogus", np.zeros((1, 64), np.float32))


def test_nvfp8_f16_scales_are_rounded_halves_with_subnormals():
    # PR #250 fp16-scale axis: the scale is amax / 448 rounded to nearest even as
    # an IEEE half, subnormals kept (tiny blocks must not flush to zero).
    n, k = 4, 64
    w = synth.weights(n, k, seed=31)
    w[1] *= np.float32(1e-2)                      # amax / 448 in the half subnormal range
    w[2] *= np.float32(1e3)
    c, s, g = pack.pack("nvfp8_f16", w)
    amax = np.abs(w).reshape(n, k // 16, 16).max(axis=2)
    want = (amax / np.float32(448.0)).astype(np.float32).astype(np.float16)
    got = s.view(np.float16).reshape(n, k // 16)
    assert np.array_equal(got, want)
    assert (np.abs(got[1].astype(np.float64)) < 2.0 ** -14).all() and (got[1] > 0).all()
    # and a row of the twin dequantizes like nvfp8 given the same (half-exact) scales
    ref = reference.dequant_exact("nvfp8_f16", c, s, g, n, k)
    s32 = got.astype(np.float32)
    again = reference.dequant_exact("nvfp8", c, s32.view(np.uint8).reshape(n, -1), 1.0, n, k)
    assert np.array_equal(ref, again)


def test_mxint8_exactly_representable_roundtrip():
    # W = q * 2^e with q in [-127, 127] and +-127 present in every block: the
    # packer must return exactly those bytes and scales.
    rng = np.random.default_rng(37)
    n, k = 6, 256
    q = rng.integers(-127, 128, size=(n, k))
    q[:, ::32] = 127 * rng.choice([-1, 1], size=(n, k // 32))
    e = rng.integers(-30, 20, size=(n, k // 32))
    w = (q * np.repeat(2.0 ** e, 32, axis=1)).astype(np.float32)
    c, s, g = pack.pack("mxint8", w)
    assert np.array_equal(c.view(np.int8), q.astype(np.int8))
    assert np.array_equal(s.astype(np.int64), e + 127)
    assert np.array_equal(reference.dequant_exact("mxint8", c, s, g, n, k), w.astype(np.float64))


def test_mxint8_rounds_half_away_and_clamps():
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 127.0                          # scale 2^0
    w[0, 1:5] = [2.5, -2.5, 126.5, -0.5]     # ties: away from zero
    c, s, _ = pack.pack("mxint8", w)
    assert s[0, 0] == 127
    assert list(c.view(np.int8)[0, :5]) == [127, 3, -3, 127, -1]



def _int8_exact_case(rng, n, k, half, qmax=127):
    """W = q * s per group of 64 (a last group of 32 when 64 does not divide K),
    +-qmax in every group, s with few enough significant bits that qmax s / qmax
    is exact in float32 (and s is a half for the fp16-scale twin)."""
    nb = -(-k // 64)
    q = rng.integers(-qmax, qmax + 1, size=(n, k))
    q[:, ::64] = qmax * rng.choice([-1, 1], size=(n, nb))
    if half:   # 11 significant bits, exponents down into the half subnormals
        m = rng.integers(2 ** 10, 2 ** 11, size=(n, nb)).astype(np.float64)
        e = rng.integers(-34, 4, size=(n, nb))
        e = np.maximum(e, -24 - 10)            # m 2^e stays a (possibly subnormal) half
        s = (m * 2.0 ** e).astype(np.float16).astype(np.float64)
    else:      # 16 significant bits
        m = rng.integers(2 ** 15, 2 ** 16, size=(n, nb)).astype(np.float64)
        s = m * 2.0 ** rng.integers(-60, 20, size=(n, nb))
    w = (q * np.repeat(s, 64, axis=1)[:, :k]).astype(np.float32)
    return q, s, w


@pytest.mark.parametrize("fmt", ["int8", "int8_f16", "int4", "int4_f16"])
@pytest.mark.parametrize("k", [256, 96, 160])
def test_int8_exactly_representable_roundtrip(fmt, k):
    # PR #250 symmetric int8 (scale-only, +-127, group 64; the pages' ragged
    # example is this group over a dimension of 96): the packer must give back
    # exactly q and s, and the dequant exactly W -- a wrong group boundary, a
    # scale from the wrong columns or a dropped ragged group breaks it.
    rng = np.random.default_rng(41 + k)
    n = 6
    four = fmt.startswith("int4")
    q, s, w = _int8_exact_case(rng, n, k, fmt.endswith("_f16"), qmax=7 if four else 127)
    assert np.array_equal(w.astype(np.float64), q * np.repeat(s, 64, axis=1)[:, :k])
    c, sc, g = pack.pack(fmt, w)
    assert c.shape == (n, k // 2 if four else k)
    assert sc.nbytes == n * -(-k // 64) * (2 if fmt.endswith("_f16") else 4)
    if four:   # two's-complement nibbles, element 2i in the low nibble of byte i
        assert np.array_equal(c & 0xF, (q[:, 0::2] & 0xF).astype(np.uint8))
        assert np.array_equal(c >> 4, (q[:, 1::2] & 0xF).astype(np.uint8))
    else:
        assert np.array_equal(c.view(np.int8), q.astype(np.int8))
    got_s = sc.view(np.float16 if fmt.endswith("_f16") else np.float32).reshape(n, -1).astype(np.float64)
    assert np.array_equal(got_s, s)
    assert np.array_equal(reference.dequant_exact(fmt, c, sc, g, n, k), w.astype(np.float64))


@pytest.mark.parametrize("fmt", ["int8", "int8_f16"])
def test_int8_rounds_half_away_and_clamps(fmt):
    w = np.zeros((1, 64), np.float32)
    w[0, 0] = -127.0                         # scale exactly 1
    w[0, 1:5] = [2.5, -2.5, 126.5, -0.5]     # ties: away from zero
    c, s, _ = pack.pack(fmt, w)
    assert s.view(np.float32 if fmt == "int8" else np.float16)[0] == 1.0
    assert list(c.view(np.int8)[0, :5]) == [-127, 3, -3, 127, -1]


def test_int8_f16_scale_underflow_quantizes_to_zero():
    # a group whose amax / 127 rounds to a zero half stores scale 0 and zero codes
    w = np.zeros((2, 64), np.float32)
    w[0, :] = np.float32(1e-9)
    w[1, 0] = np.float32(0.5)
    c, s, g = pack.pack("int8_f16", w)
    assert s.view(np.float16)[0] == 0 and not c[0].any()
    assert not reference.dequant_exact("int8_f16", c, s, g, 2, 64)[0].any()
    assert c.view(np.int8)[1, 0] == 127


@pytest.mark.parametrize("fmt", ["int4", "int4_f16"])
def test_int4_rounds_half_away_and_clamps(fmt):
    # PR #250 intN codec: sign-extend from bit 3, clamp to +-7
    w = np.zeros((1, 64), np.float32)
    w[0, 0] = 7.0                            # scale exactly 1
    w[0, 1:6] = [2.5, -2.5, 6.5, -0.5, -7.0]
    c, s, _ = pack.pack(fmt, w)
    assert s.view(np.float16 if fmt == "int4_f16" else np.float32)[0] == 1.0
    q = reference.unpack_codes(fmt, c, 1, 64)[0, :6]
    assert list(q) == [7, 3, 0xD, 7, 0xF, 0x9]           # 3, -3, 7 (6.5 away), -1, -7 as nibbles
    assert list(reference.dequant_exact(fmt, c, s, 1.0, 1, 64)[0, :6]) == [7, 3, -3, 7, -1, -7]


def test_int4_nibble_eight_decodes_as_minus_eight():
    # the packer never writes 0x8, but a stored 0x8 sign-extends to -8
    c = np.full((1, 32), 0x88, np.uint8)
    s = np.array([1.0], np.float32).view(np.uint8).reshape(1, -1)
    assert (reference.dequant_exact("int4", c, s, 1.0, 1, 64) == -8).all()


def _x2_case(rng, n, k):
    """W = s0 v0 + s1 v1 built so that both residual levels come back exactly:
    v0, v1 on the E2M1 grid, +-6 in every block of each level (and v1 = 0 where
    v0 = +-6, so amax(W) = 6 s0), s1 = s0 / 32 (so |s1 v1| stays under half
    of the smallest E2M1 gap times s0 and level 0 rounds back to v0), s0 with
    few significant bits (every product and sum exact in float32)."""
    grid = codec.E2M1_TABLE[:8]                      # 0, .5, 1, 1.5, 2, 3, 4, 6
    nb = k // 32
    v0 = rng.choice(grid[:7], size=(n, k)) * rng.choice([-1, 1], size=(n, k))
    v1 = rng.choice(grid, size=(n, k)) * rng.choice([-1, 1], size=(n, k))
    v0[:, 0::32] = 6.0 * rng.choice([-1, 1], size=(n, nb))
    v1[:, 0::32] = 0.0
    v1[:, 1::32] = 6.0 * rng.choice([-1, 1], size=(n, nb))
    s0 = rng.integers(64, 128, size=(n, nb)) * 2.0 ** rng.integers(-20, 0, size=(n, nb))
    s1 = s0 / 32
    w = v0 * np.repeat(s0, 32, axis=1) + v1 * np.repeat(s1, 32, axis=1)
    return v0, v1, s0, s1, w.astype(np.float32)


def test_mxfp4x2_two_levels_round_trip_exactly():
    # rlx-cpu dequant_matmul_mxfp4x2 decodes w = s0 LUT[q0] + s1 LUT[q1]; the
    # packer's two residual levels must recover v0, v1, s0, s1 and the layout
    # [N, 2, K/2] codes, [N, 2, K/32] float32 scales.
    rng = np.random.default_rng(51)
    n, k = 5, 128
    v0, v1, s0, s1, w = _x2_case(rng, n, k)
    assert np.array_equal(w.astype(np.float64), v0 * np.repeat(s0, 32, axis=1) + v1 * np.repeat(s1, 32, axis=1))
    c, s, g = pack.pack("mxfp4x2", w)
    sc = s.view(np.float32).reshape(n, 2, k // 32)
    assert np.array_equal(sc[:, 0], s0) and np.array_equal(sc[:, 1], s1)
    planes = c.reshape(n, 2, k // 2)
    for p, v in ((0, v0), (1, v1)):
        q = reference.unpack_codes("mxfp4", planes[:, p], n, k)
        assert np.array_equal(codec.E2M1_TABLE[q], v), p
    assert np.array_equal(reference.dequant_exact("mxfp4x2", c, s, g, n, k), w.astype(np.float64))


def test_mxfp4x2_on_grid_weights_leave_an_empty_residual():
    # a block exactly on level 0's grid: plane 1 is all zero codes with scale 1.0
    rng = np.random.default_rng(52)
    n, k = 3, 64
    v0 = rng.choice(codec.E2M1_TABLE[:16], size=(n, k))
    v0[:, 0::32] = 6.0
    w = (v0 * 2.0 ** -5).astype(np.float32)
    c, s, _ = pack.pack("mxfp4x2", w)
    sc = s.view(np.float32).reshape(n, 2, -1)
    assert (sc[:, 0] == 2.0 ** -5).all() and (sc[:, 1] == 1.0).all()
    assert not (c.reshape(n, 2, -1)[:, 1] & 0x77).any()     # only signed zeros in plane 1


def test_mxfp4x2_error_within_second_level_step():
    # the residual is packed by level 1, so the remaining error of a block is at
    # most half the widest E2M1 gap (1.0) times s1, plus float32 rounding; and
    # far below the one-level error
    n, k = 32, 512
    w = synth.weights(n, k, seed=53)
    c, s, g = pack.pack("mxfp4x2", w)
    err = np.abs(reference.dequant_exact("mxfp4x2", c, s, g, n, k) - w)
    s1 = s.view(np.float32).reshape(n, 2, -1)[:, 1].astype(np.float64)
    assert (err <= np.repeat(s1, 32, axis=1) * (1.0 + 1e-6) + 1e-30).all()
    c1, s_1, g1 = pack.pack("mxfp4", w)
    err1 = np.abs(reference.dequant_exact("mxfp4", c1, s_1, g1, n, k) - w)
    assert err.max() < err1.max() / 8


def test_mxfp4x2_two_negative_zero_codes_give_negative_zero():
    # s0 LUT[q0] + s1 LUT[q1] with both codes the sign-set zero (0x8) is the
    # IEEE sum -0 + -0 = -0; one +0 code makes it +0
    c = np.zeros((1, 2, 16), np.uint8)
    c[0, :, 0] = 0x88                                  # k = 0, 1: -0 in both planes
    c[0, 0, 1] = 0x08                                  # k = 2: -0 in plane 0, +0 in plane 1
    s = np.array([[0.5, 0.25]], np.float32).view(np.uint8).reshape(1, -1)
    w = reference.dequant_f32("mxfp4x2", c.reshape(1, -1), s, 1.0, 1, 32)
    assert np.signbit(w[0, 0]) and np.signbit(w[0, 1]) and not np.signbit(w[0, 2])
    assert (w == 0).all()


def test_mxint4_exactly_representable_roundtrip():
    # W = q * 2^e with q in [-7, 7] and +-7 in every block of 32: the packer
    # returns exactly those nibbles and E8M0 bytes (PR #250 MXINT4)
    rng = np.random.default_rng(57)
    n, k = 4, 128
    q = rng.integers(-7, 8, size=(n, k))
    q[:, ::32] = 7 * rng.choice([-1, 1], size=(n, k // 32))
    e = rng.integers(-40, 30, size=(n, k // 32))
    w = (q * np.repeat(2.0 ** e, 32, axis=1)).astype(np.float32)
    c, s, g = pack.pack("mxint4", w)
    assert np.array_equal(s.astype(np.int64), e + 127)
    assert np.array_equal(c & 0xF, (q[:, 0::2] & 0xF).astype(np.uint8))
    assert np.array_equal(c >> 4, (q[:, 1::2] & 0xF).astype(np.uint8))
    assert np.array_equal(reference.dequant_exact("mxint4", c, s, g, n, k), w.astype(np.float64))


def test_mxint4_scale_snaps_up_and_rounds_half_away():
    # amax 6 -> 6 / 7 snapped up to 2^0; 2.5 -> 3, -2.5 -> -3, -0.5 -> -1
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 6.0
    w[0, 1:4] = [2.5, -2.5, -0.5]
    c, s, _ = pack.pack("mxint4", w)
    assert s[0, 0] == 127
    assert list(reference.dequant_exact("mxint4", c, s, 1.0, 1, 32)[0, :4]) == [6, 3, -3, -1]


LEGACY = {"fp4": ("e2m1", 6.0), "fp8_e4m3": ("e4m3", 448.0), "fp8_e5m2": ("e5m2", 57344.0)}


@pytest.mark.parametrize("fmt", ["fp4", "fp8_e4m3", "fp8_e5m2", "fp4_f16", "fp8_e4m3_f16", "fp8_e5m2_f16"])
def test_legacy_float_exactly_representable_roundtrip(fmt):
    # PR #250 legacy float formats: the element under a float scale per 32 with
    # s = amax / max_finite.  W built as grid values x s with the block maximum
    # at the element max and s of few significant bits (a half for the twins):
    # the packer must return exactly those codes and scales.
    rng = np.random.default_rng(61)
    base = fmt.replace("_f16", "")
    elem, maxf = LEGACY[base]
    table = {"e2m1": codec.E2M1_TABLE, "e4m3": codec.E4M3_TABLE, "e5m2": codec.E5M2_TABLE}[elem]
    ncode = 16 if elem == "e2m1" else 256
    finite = np.array([c for c in range(ncode) if np.isfinite(table[c])])
    maxcode = int(finite[np.argmax(table[finite])])
    n, k = 4, 128
    codes = rng.choice(finite, size=(n, k))
    codes[:, ::32] = maxcode
    m = rng.integers(512, 1024, size=(n, k // 32)).astype(np.float64)
    s = m * 2.0 ** rng.integers(-24, -12, size=(n, k // 32))      # 10 significant bits: a normal half
    vals = _elem_values_lib(base if base != "fp4" else "mxfp4", codes).reshape(n, k // 32, 32) * s[..., None]
    w = vals.reshape(n, k).astype(np.float32)
    assert np.array_equal(w.astype(np.float64), vals.reshape(n, k))
    c, sc, g = pack.pack(fmt, w)
    got_s = sc.view(np.float16 if fmt.endswith("_f16") else np.float32).reshape(n, -1).astype(np.float64)
    assert np.array_equal(got_s, s)
    assert np.array_equal(reference.dequant_exact(fmt, c, sc, g, n, k), w.astype(np.float64))


def test_legacy_float_scale_is_not_snapped():
    # unlike the MX formats, the scale is amax / max_finite itself (no power of two)
    w = np.zeros((1, 32), np.float32)
    w[0, 0] = 5.0                                    # fp4: s = 5/6, not 1
    c, s, _ = pack.pack("fp4", w)
    assert s.view(np.float32)[0] == np.float32(5.0) / np.float32(6.0)
    assert reference.dequant_f32("fp4", c, s, 1.0, 1, 32)[0, 0] == np.float32(6.0 * np.float64(s.view(np.float32)[0]))



# ----- the sub-byte integer widths (PR #250: int2-6, mxint2-6, one LSB-first bit stream) -----

SUBBYTE = ["int2", "int3", "int5", "int6", "int3_f16", "mxint2", "mxint3", "mxint5", "mxint6"]


def test_bit_stream_layout_against_integer_arithmetic():
    # code j of a row occupies bits [j N, j N + N) of the row bytes read as one
    # little-endian integer: built here with Python integers, not numpy bits
    rng = np.random.default_rng(81)
    for bits in (2, 3, 5, 6, 4):
        n, k = 3, 64
        codes = rng.integers(0, 1 << bits, size=(n, k)).astype(np.uint8)
        got = pack.pack_bits(codes, bits)
        for r in range(n):
            v = 0
            for j in range(k):
                v |= int(codes[r, j]) << (j * bits)
            assert bytes(got[r]) == v.to_bytes(k * bits // 8, "little"), bits
        assert np.array_equal(reference.unpack_codes({2: "int2", 3: "int3", 5: "int5", 6: "int6", 4: "mxfp4"}[bits],
                                                     got, n, k), codes)


def test_four_bit_stream_is_the_nibble_layout():
    # PR #250: "a 4-bit stream is byte-identical to the old nibble layout"
    rng = np.random.default_rng(82)
    codes = rng.integers(0, 16, size=(4, 96)).astype(np.uint8)
    assert np.array_equal(pack.pack_bits(codes, 4), pack._pack_nibbles(codes))


@pytest.mark.parametrize("fmt", SUBBYTE)
def test_subbyte_exactly_representable_roundtrip(fmt):
    # W = q * s per block with +-(2^(N-1) - 1) in every block and s of few
    # significant bits (a power of two for mxint): codes, scales and values back exactly
    rng = np.random.default_rng(83 + len(fmt))
    bits = pack.INTN[fmt]
    qmax = (1 << (bits - 1)) - 1
    n, k, blk = 4, 128, pack.BLOCK[fmt]
    nb = k // blk
    q = rng.integers(-qmax, qmax + 1, size=(n, k))
    q[:, ::blk] = qmax * rng.choice([-1, 1], size=(n, nb))
    if fmt.startswith("mx"):
        e = rng.integers(-30, 20, size=(n, nb))
        s = 2.0 ** e
    else:
        s = rng.integers(512, 1024, size=(n, nb)) * 2.0 ** rng.integers(-24, -12, size=(n, nb))
    w = (q * np.repeat(s, blk, axis=1)).astype(np.float32)
    c, sc, g = pack.pack(fmt, w)
    assert c.shape == (n, k * bits // 8)
    assert np.array_equal(reference.unpack_codes(fmt, c, n, k), (q & ((1 << bits) - 1)).astype(np.uint8))
    if fmt.startswith("mx"):
        assert np.array_equal(sc.astype(np.int64), e + 127)
    else:
        got_s = sc.view(np.float16 if fmt.endswith("_f16") else np.float32).reshape(n, -1).astype(np.float64)
        assert np.array_equal(got_s, s)
    assert np.array_equal(reference.dequant_exact(fmt, c, sc, g, n, k), w.astype(np.float64))


def test_subbyte_ragged_last_group():
    # int3 over K = 96: a group of 64 and a ragged group of 32 with its own scale
    n, k = 2, 96
    w = synth.weights(n, k, seed=84)
    c, s, g = pack.pack("int3", w)
    assert c.shape == (n, 36) and s.view(np.float32).shape == (n, 2)
    sc = s.view(np.float32).reshape(n, 2)
    assert np.array_equal(sc[:, 1], (np.abs(w[:, 64:]).max(axis=1) / np.float32(3.0)).astype(np.float32))
