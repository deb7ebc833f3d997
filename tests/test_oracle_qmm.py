"""Pins for the oracle's dequant value and dequantizing matmul.

* exact rational brute force (Python Fractions, element/scale values from
  library reinterpretations and explicit nibble loops) on tiny shapes;
* the all-unit-scales special case equals a library matmul of the decoded codes;
* the int4-affine algebraic split (scale * sum q x + bias * sum x) that the
  metaltile qmm correctness test uses, on that test's deterministic pattern;
* batch rows equal stacked single-row results;
* the expert-routed product: exact rational brute force over a stacked
  weight, E = 1 reduces to qmm, and relabelling the experts changes nothing;
* the batched products: exact rational brute force per matrix;
* the RMSNorm-fused product: 60-digit decimal brute force, the closed form of
  a constant row, and invariance of the normalisation under power-of-two
  scaling of x (eps = 0);
* planted mistakes (applied to the oracle on the CPU) are caught by these pins.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from block_scaled_quantized_spec_gb300 import synth
from oracle import pack, reference

FMTS = pack.FORMATS


# ----- an independent decode: explicit loops + library reinterpretations -----

def _lib_elem(fmt, c):
    if fmt in ("mxfp4", "nvfp4", "fp4", "fp4_f16"):
        # fp_quantized_mma.rs two_m_int: subnormal 2m = mant, normal 2m = (mant+2) 2^(exp-1)
        c3, s = c & 7, 1 - 2 * (c >> 3)
        e, m = c3 >> 1, c3 & 1
        two_m = m if e == 0 else (m + 2) * 2 ** (e - 1)
        return Fraction(s * two_m, 2)
    if fmt in ("mxfp8_e4m3", "nvfp8", "nvfp8_f16", "fp8_e4m3", "fp8_e4m3_f16"):
        v = torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item()
        return Fraction(v)
    if fmt in ("mxfp8_e5m2", "fp8_e5m2", "fp8_e5m2_f16"):
        return Fraction(float(np.array([c << 8], np.uint16).view(np.float16)[0]))
    if fmt in ("mxint8", "int8", "int8_f16"):
        return Fraction(c - 256 if c >= 128 else c)
    if fmt in ("int4", "int4_f16", "mxint4"):
        return Fraction(c - 16 if c >= 8 else c)
    if fmt in pack.INTN:                                  # sign bit N - 1 of an N-bit code
        nb = pack.INTN[fmt]
        return Fraction(c - (1 << nb) if c >> (nb - 1) else c)
    return Fraction(c)


def _lib_scale(fmt, sbytes, n, b):
    if fmt in ("mxfp4", "mxfp8_e4m3", "mxfp8_e5m2", "mxint8", "mxint4", "mxint2", "mxint3", "mxint5", "mxint6"):
        return Fraction(2) ** (int(sbytes[n][b]) - 127), Fraction(0)
    if fmt == "nvfp4":
        v = torch.tensor([int(sbytes[n][b])], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item()
        return Fraction(v), Fraction(0)
    if fmt in ("nvfp8", "int8", "int4", "fp4", "fp8_e4m3", "fp8_e5m2", "int2", "int3", "int5", "int6"):
        return Fraction(float(np.frombuffer(bytes(sbytes[n][4 * b:4 * b + 4]), "<f4")[0])), Fraction(0)
    if fmt.endswith("_f16"):
        return Fraction(float(np.frombuffer(bytes(sbytes[n][2 * b:2 * b + 2]), "<f2")[0])), Fraction(0)
    raw = bytes(sbytes[n][4 * b:4 * b + 4])
    s_bits, b_bits = np.frombuffer(raw, "<u2")
    f = lambda h: Fraction(float((np.array([h], np.uint32) << 16).view(np.float32)[0]))  # noqa: E731
    return f(s_bits), f(b_bits)


def _code(fmt, row, kk):
    # code kk of a row: bits [kk N, kk N + N) of the row bytes read as one
    # little-endian integer (4-bit: the nibble layout; 8-bit: the byte)
    nb = pack.ELEM_BITS[fmt]
    return (int.from_bytes(bytes(row), "little") >> (kk * nb)) & ((1 << nb) - 1)


def _x2_weight(codes_row, scales_row, kk, k):
    # rlx-cpu dequant_matmul_mxfp4x2: s0 LUT[q0] + s1 LUT[q1]; a row holds its
    # plane-0 nibbles, then its plane-1 nibbles, and its s0 floats, then its s1 floats
    nb = k // 32
    w = Fraction(0)
    for p in range(2):
        byte = codes_row[p * (k // 2) + kk // 2]
        c = (byte >> (4 * (kk % 2))) & 0xF
        o = 4 * (p * nb + kk // 32)
        sc = Fraction(float(np.frombuffer(bytes(scales_row[o:o + 4]), "<f4")[0]))
        w += _lib_elem("mxfp4", c) * sc
    return w


def _brute_qmm(fmt, codes, scales, g, x64, m, n, k):
    blk = pack.BLOCK[fmt]
    codes = [[int(v) for v in r] for r in np.asarray(codes).reshape(n, -1)]
    scales = [[int(v) for v in r] for r in np.asarray(scales).reshape(n, -1)]
    out = [[Fraction(0)] * n for _ in range(m)]
    for j in range(n):
        wrow = []
        for kk in range(k):
            if fmt == "mxfp4x2":
                wrow.append(_x2_weight(codes[j], scales[j], kk, k))
                continue
            c = _code(fmt, codes[j], kk)
            mul, add = _lib_scale(fmt, scales, j, kk // blk)
            w = _lib_elem(fmt, c) * mul + add
            if fmt == "nvfp4":
                w *= Fraction(float(g))
            wrow.append(w)
        for i in range(m):
            out[i][j] = sum(Fraction(float(x64[i][kk])) * wrow[kk] for kk in range(k))
    return out


def _tiny_case(fmt, m=3, n=5, k=64, seed=0):
    w = synth.weights(n, k, seed=seed, outliers=(fmt == "nvfp4"))
    c, s, g = pack.pack(fmt, w)
    x = synth.activations_bf16(m, k, seed=seed + 1)
    return c, s, g, x


def _check_brute(fmt, m=3, n=5, k=64, seed=0):
    c, s, g, x = _tiny_case(fmt, m, n, k, seed)
    ref, bound = reference.qmm_ref(fmt, c, s, g, x, "bf16", m, n, k)
    x64 = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = _brute_qmm(fmt, c, s, g, x64, m, n, k)
    for i in range(m):
        for j in range(n):
            # ref is an fp64 matmul: within a few fp64 ulps of the exact rational sum
            err = abs(Fraction(ref[i, j]) - exact[i][j])
            scale = sum(abs(Fraction(float(x64[i][kk]))) for kk in range(k)) + 1
            assert err <= Fraction(1, 2 ** 40) * scale, (fmt, i, j)
    return True


@pytest.mark.parametrize("fmt", FMTS)
def test_qmm_ref_matches_exact_rational_brute_force(fmt):
    assert _check_brute(fmt)


@pytest.mark.parametrize("fmt", FMTS)
def test_dequant_f32_is_one_rounding_of_exact(fmt):
    n, k = 4, 64
    c, s, g, _ = _tiny_case(fmt, 1, n, k, seed=3)
    wf = reference.dequant_f32(fmt, c, s, g, n, k)
    codes = [[int(v) for v in r] for r in np.asarray(c).reshape(n, -1)]
    scales = [[int(v) for v in r] for r in np.asarray(s).reshape(n, -1)]
    blk = pack.BLOCK[fmt]
    for j in range(n):
        for kk in range(k):
            if fmt == "mxfp4x2":
                w = _x2_weight(codes[j], scales[j], kk, k)
                assert wf[j, kk] == np.float32(float(w)), (fmt, j, kk)
                continue
            cc = _code(fmt, codes[j], kk)
            mul, add = _lib_scale(fmt, scales, j, kk // blk)
            w = _lib_elem(fmt, cc) * mul + add
            if fmt == "nvfp4":
                w *= Fraction(float(g))
            # the float32 nearest to w (ties even) via numpy's correctly rounded conversion
            # of the exactly representable float64 w
            assert float(w) == w or fmt == "int4_affine"
            assert wf[j, kk] == np.float32(float(w)), (fmt, j, kk)


def test_unit_scales_equal_library_matmul():
    # All E8M0 scales 127 (= 1.0): qmm reduces to X @ E(codes)^T, a plain library matmul.
    rng = np.random.default_rng(5)
    m, n, k = 4, 24, 128
    for fmt, elem_dt in (("mxfp8_e4m3", torch.float8_e4m3fn), ("mxfp8_e5m2", torch.float8_e5m2)):
        codes = rng.integers(0, 256, size=(n, k), dtype=np.uint8)
        bad = (codes & 0x7F) == 0x7F if fmt == "mxfp8_e4m3" else ((codes >> 2) & 31) == 31
        codes[bad] = 0
        scales = np.full((n, k // 32), 127, np.uint8)
        x = synth.activations_bf16(m, k, seed=6)
        ref, _ = reference.qmm_ref(fmt, codes, scales, 1.0, x, "bf16", m, n, k)
        e = torch.from_numpy(codes).view(elem_dt).double()
        xt = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
        lib = (xt @ e.T).numpy()
        assert np.allclose(ref, lib, rtol=1e-12, atol=1e-12)


def test_batch_rows_equal_stacked_single_rows():
    # rlx-cpu batch-M vs row-by-row M=1 equality test idea.
    fmt, m, n, k = "nvfp4", 6, 32, 256
    c, s, g, x = _tiny_case(fmt, m, n, k, seed=9)
    ref, bound = reference.qmm_ref(fmt, c, s, g, x, "bf16", m, n, k)
    for i in range(m):
        r1, b1 = reference.qmm_ref(fmt, c, s, g, x[i:i + 1], "bf16", 1, n, k)
        assert np.array_equal(r1[0], ref[i]) and np.array_equal(b1[0], bound[i])


def test_sampled_ref_equals_dense_ref():
    fmt, m, n, k = "int4_affine", 5, 40, 256
    c, s, g, x = _tiny_case(fmt, m, n, k, seed=10)
    ref, bound = reference.qmm_ref(fmt, c, s, g, x, "bf16", m, n, k)
    rows = np.array([0, 4, 2, 3, 1, 0])
    cols = np.array([39, 0, 17, 17, 5, 38])
    r, b = reference.qmm_ref_sampled(fmt, c, s, g, x, "bf16", m, n, k, rows, cols)
    assert np.allclose(r, ref[rows, cols], rtol=1e-14, atol=1e-14)
    assert np.allclose(b, bound[rows, cols], rtol=1e-14, atol=1e-14)


def test_int4_affine_algebraic_split_on_page_pattern():
    # metaltile-std tests/qmm_gpu_correctness.rs, mt_qmm_matches_cpu_reference_f32:
    # m=8, n=16, k=512, group 64; packed word i holds nibble ((i + bit) & 0xF) at bits 4*bit;
    # scales 0.1 + 0.001 i, biases 0.0001 i (rounded here to the bf16 storage);
    # x = 1 + 0.001 i (f32).  Its CPU reference accumulates s_g * sum(q x) + bias_g * sum(x)
    # per group: an algebraically different route to the same sums.
    m, n, k, gs = 8, 16, 512, 64
    words = np.array([sum(((i + bit) & 0xF) << (4 * bit) for bit in range(8))
                      for i in range(n * k // 8)], dtype="<u4")
    codes = words.view(np.uint8).reshape(n, k // 2)
    ng = k // gs
    sc = np.array([0.1 + i * 0.001 for i in range(n * ng)], np.float32)
    bi = np.array([i * 0.0001 for i in range(n * ng)], np.float32)
    sc_b = torch.from_numpy(sc).to(torch.bfloat16)
    bi_b = torch.from_numpy(bi).to(torch.bfloat16)
    pair = torch.stack([sc_b.view(torch.int16), bi_b.view(torch.int16)], dim=-1).numpy().view(np.uint16)
    scales = pair.reshape(n, ng * 2).view(np.uint8)
    x = np.array([1.0 + i * 0.001 for i in range(m * k)], np.float32).reshape(m, k)
    ref, _ = reference.qmm_ref("int4_affine", codes, scales, 1.0, x, "f32", m, n, k)
    s64, b64 = sc_b.double().numpy(), bi_b.double().numpy()
    for r in range(m):
        for col in range(n):
            acc = Fraction(0)
            for grp in range(ng):
                qdot = Fraction(0)
                xsum = Fraction(0)
                for p in range(8):
                    packed = int(words[col * k // 8 + grp * 8 + p])
                    for bit in range(8):
                        q = (packed >> (bit * 4)) & 0xF
                        xv = Fraction(float(x[r, grp * gs + p * 8 + bit]))
                        qdot += q * xv
                        xsum += xv
                acc += Fraction(float(s64[col * ng + grp])) * qdot + Fraction(float(b64[col * ng + grp])) * xsum
            assert abs(Fraction(ref[r, col]) - acc) <= abs(acc) * Fraction(1, 2 ** 45), (r, col)


def test_bound_definition():
    fmt, m, n, k = "mxfp4", 2, 8, 64
    c, s, g, x = _tiny_case(fmt, m, n, k, seed=12)
    _, bound = reference.qmm_ref(fmt, c, s, g, x, "bf16", m, n, k)
    w = reference.dequant_exact(fmt, c, s, g, n, k)
    xv = reference.x_values(x, "bf16")
    for i in range(m):
        for j in range(n):
            want = 2e-3 * sum(abs(xv[i, kk]) * abs(w[j, kk]) for kk in range(k)) + 1e-6
            assert abs(bound[i, j] - want) <= 1e-15 * want


# ---------------------- planted mistakes in the oracle are caught ----------------------

def test_planted_mistakes_are_caught(monkeypatch):
    """Each plausible oracle bug (wrong nibble order, dropped global, transposed
    operand, swapped scale/bias) must make a pin above fail."""
    orig_unpack = reference.unpack_codes
    orig_scales = reference.block_scales
    orig_exact = reference.dequant_exact

    def swapped_nibbles(fmt, codes, n, k):
        out = orig_unpack(fmt, codes, n, k)
        if fmt in ("mxfp4", "nvfp4", "int4_affine"):
            out = out.reshape(n, k // 2, 2)[..., ::-1].reshape(n, k)
        return out

    def dropped_global(fmt, codes, scales, g, n, k):
        return orig_exact(fmt, codes, scales, 1.0, n, k)

    def swapped_affine(fmt, scales, g, n, k):
        mul, add = orig_scales(fmt, scales, g, n, k)
        return (add, mul) if add is not None else (mul, add)

    plants = [("unpack_codes", swapped_nibbles, "mxfp4"),
              ("dequant_exact", dropped_global, "nvfp4"),
              ("block_scales", swapped_affine, "int4_affine")]
    for name, fn, fmt in plants:
        with monkeypatch.context() as mp:
            mp.setattr(reference, name, fn)
            with pytest.raises(AssertionError):
                _check_brute(fmt)

    # a transposed weight operand
    def transposed_ref(fmt, codes, scales, g, x, x_dtype, m, n, k):
        w = orig_exact(fmt, codes, scales, g, n, k)
        xv = reference.x_values(x, x_dtype).reshape(m, k)
        return (xv @ w.reshape(k, n)), None

    with monkeypatch.context() as mp:
        mp.setattr(reference, "qmm_ref", transposed_ref)
        with pytest.raises(AssertionError):
            _check_brute("mxfp8_e4m3")


def test_planted_mistakes_in_the_added_formats_are_caught(monkeypatch):
    """Plausible decode bugs of the formats beyond the first six -- a signed
    element read unsigned, the mxfp4x2 planes' scales swapped, a half scale read
    as bfloat16 -- must each fail the exact rational brute force."""
    orig_elem = reference.element_values
    orig_scales = reference.block_scales
    orig_exact = reference.dequant_exact

    def unsigned_ints(fmt, codes):
        if fmt in ("mxint8", "int8", "int4", "mxint4"):
            return codes.astype(np.float64)
        return orig_elem(fmt, codes)

    def swapped_planes(fmt, codes, scales, g, n, k):
        if fmt == "mxfp4x2":
            sc = np.ascontiguousarray(np.asarray(scales, dtype=np.uint8)).view(np.float32).reshape(n, 2, -1)
            scales = np.ascontiguousarray(sc[:, ::-1]).view(np.uint8).reshape(n, -1)
        return orig_exact(fmt, codes, scales, g, n, k)

    def half_as_bf16(fmt, scales, g, n, k):
        if fmt in ("int8_f16", "nvfp8_f16", "fp4_f16"):
            s = np.ascontiguousarray(np.asarray(scales, dtype=np.uint8)).view(np.uint16).reshape(n, -1)
            return reference.codec.decode_bf16(s), None
        return orig_scales(fmt, scales, g, n, k)

    plants = [("element_values", unsigned_ints, "mxint8"), ("element_values", unsigned_ints, "int4"),
              ("element_values", unsigned_ints, "mxint4"), ("dequant_exact", swapped_planes, "mxfp4x2"),
              ("block_scales", half_as_bf16, "int8_f16"), ("block_scales", half_as_bf16, "fp4_f16")]
    for name, fn, fmt in plants:
        with monkeypatch.context() as mp:
            mp.setattr(reference, name, fn)
            with pytest.raises(AssertionError):
                _check_brute(fmt)


# ----- expert-routed rows (MoE gather-qmm) -----

def _gather_case(fmt, m, n, k, e, seed):
    w = synth.weights(e * n, k, seed=seed, outliers=(fmt == "nvfp4"))
    c, s, g = pack.pack(fmt, w)
    x = synth.activations_bf16(m, k, seed=seed + 1)
    idx = np.random.default_rng(seed + 2).integers(0, e, size=m).astype(np.int32)
    return c, s, g, x, idx


def _check_gather_brute(fmt):
    # Row m against expert idx[m]'s N rows of the stack, summed exactly (the
    # explicit decode loops above over the whole [E * N, K] stack).
    m, n, k, e = 4, 3, 64, 3
    c, s, g, x, idx = _gather_case(fmt, m, n, k, e, seed=21)
    idx[:] = [2, 0, 2, 1]
    ref, _ = reference.qmm_gather_ref(fmt, c, s, g, x, "bf16", idx, m, n, k, e)
    x64 = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    exact = _brute_qmm(fmt, c, s, g, x64, m, e * n, k)        # every row against every stacked row
    for i in range(m):
        for j in range(n):
            want = exact[i][idx[i] * n + j]
            scale = sum(abs(Fraction(float(x64[i][kk]))) for kk in range(k)) + 1
            assert abs(Fraction(ref[i, j]) - want) <= Fraction(1, 2 ** 40) * scale, (fmt, i, j)
    return True


@pytest.mark.parametrize("fmt", FMTS)
def test_gather_ref_matches_exact_rational_brute_force(fmt):
    assert _check_gather_brute(fmt)


def test_planted_gather_mistake_is_caught(monkeypatch):
    """An expert-minor reading of the stack ([N, E, K] instead of [E, N, K])
    must fail the brute-force pin."""
    orig_exact = reference.dequant_exact

    def expert_minor(fmt, codes, scales, g, rows, k):
        w = orig_exact(fmt, codes, scales, g, rows, k)
        e = 3                                            # the pin's expert count
        return w.reshape(rows // e, e, k).transpose(1, 0, 2).reshape(rows, k)

    with monkeypatch.context() as mp:
        mp.setattr(reference, "dequant_exact", expert_minor)
        with pytest.raises(AssertionError):
            _check_gather_brute("mxfp4")


def test_gather_ref_with_one_expert_is_qmm():
    fmt, m, n, k = "mxfp4", 5, 24, 256
    c, s, g, x, _ = _gather_case(fmt, m, n, k, 1, seed=22)
    ref, bound = reference.qmm_gather_ref(fmt, c, s, g, x, "bf16", np.zeros(m, np.int32), m, n, k, 1)
    r2, b2 = reference.qmm_ref(fmt, c, s, g, x, "bf16", m, n, k)
    assert np.allclose(ref, r2, rtol=1e-13, atol=1e-13) and np.allclose(bound, b2, rtol=1e-13, atol=1e-13)


def test_gather_ref_invariant_under_expert_relabelling():
    # Permute the experts' slabs in the stack and remap the indices: same result.
    fmt, m, n, k, e = "mxfp8_e5m2", 6, 8, 128, 4
    c, s, g, x, idx = _gather_case(fmt, m, n, k, e, seed=23)
    perm = np.array([2, 0, 3, 1])                  # new slab j holds old expert perm[j]
    inv = np.argsort(perm)
    c2 = np.asarray(c).reshape(e, n, -1)[perm].reshape(e * n, -1)
    s2 = np.asarray(s).reshape(e, n, -1)[perm].reshape(e * n, -1)
    r1, _ = reference.qmm_gather_ref(fmt, c, s, g, x, "bf16", idx, m, n, k, e)
    r2, _ = reference.qmm_gather_ref(fmt, c2, s2, g, x, "bf16", inv[idx], m, n, k, e)
    assert np.array_equal(r1, r2)


def test_gather_ref_rejects_out_of_range_index():
    fmt, m, n, k, e = "nvfp8", 2, 4, 64, 2
    c, s, g, x, idx = _gather_case(fmt, m, n, k, e, seed=24)
    with pytest.raises(ValueError):
        reference.qmm_gather_ref(fmt, c, s, g, x, "bf16", np.array([0, 2], np.int32), m, n, k, e)


# ----- batched products and the RMSNorm-fused product -----

def test_batched_ref_matches_exact_rational_brute_force():
    fmt, m, k = "nvfp4", 2, 64
    mats, brute = [], []
    x = synth.activations_bf16(m, k, seed=51)
    x64 = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for i, n in enumerate((3, 5)):
        w = synth.weights(n, k, seed=52 + i, outliers=True)
        c, s_, g = pack.pack(fmt, w)
        mats.append((c, s_, g, n))
        brute.append(_brute_qmm(fmt, c, s_, g, x64, m, n, k))
    refs = reference.qmm_batched_ref(fmt, mats, x, "bf16", m, k)
    assert len(refs) == 2
    for (ref, _), exact, (_, _, _, n) in zip(refs, brute, mats):
        for i in range(m):
            for j in range(n):
                scale = sum(abs(Fraction(float(x64[i][kk]))) for kk in range(k)) + 1
                assert abs(Fraction(ref[i, j]) - exact[i][j]) <= Fraction(1, 2 ** 40) * scale


def _gamma_bits(k, seed):
    g = 1.0 + 0.25 * np.random.default_rng(seed).standard_normal(k)
    return (torch.from_numpy(g.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()).view(np.uint16)


@pytest.mark.parametrize("fmt", ["mxfp4", "int4_affine", "nvfp8"])
def test_rmsnorm_ref_matches_decimal_brute_force(fmt):
    from decimal import Decimal, getcontext
    getcontext().prec = 60
    m, n, k, eps = 2, 3, 64, 1e-5
    c, s_, g, x = _tiny_case(fmt, m, n, k, seed=55)
    gb = _gamma_bits(k, 56)
    ref, _ = reference.qmm_rmsnorm_ref(fmt, c, s_, g, x, "bf16", gb, eps, m, n, k)
    x64 = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    g64 = (gb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes = [[int(v) for v in r] for r in np.asarray(c).reshape(n, -1)]
    scales = [[int(v) for v in r] for r in np.asarray(s_).reshape(n, -1)]
    blk = pack.BLOCK[fmt]
    D = lambda fr: Decimal(fr.numerator) / Decimal(fr.denominator)  # noqa: E731
    for i in range(m):
        ms = sum(Decimal(float(v)) ** 2 for v in x64[i]) / k + Decimal(eps)
        inv = 1 / ms.sqrt()
        for j in range(n):
            acc = Decimal(0)
            for kk in range(k):
                byte = codes[j][kk // 2] if fmt in ("mxfp4", "nvfp4", "int4_affine") else codes[j][kk]
                cc = (byte >> (4 * (kk % 2))) & 0xF if fmt in ("mxfp4", "nvfp4", "int4_affine") else byte
                mul, add = _lib_scale(fmt, scales, j, kk // blk)
                w = _lib_elem(fmt, cc) * mul + add
                acc += Decimal(float(x64[i][kk])) * Decimal(float(g64[kk])) * inv * D(w)
            assert abs(Decimal(float(ref[i, j])) - acc) <= Decimal(2) ** -40 * (abs(acc) + 1), (fmt, i, j)


def test_rmsnorm_ref_constant_row_closed_form():
    # x[m, :] = c, gamma = 1: every normalised value is c / sqrt(c^2 + eps).
    fmt, n, k, eps = "mxfp8_e4m3", 6, 128, 0.01
    c_, s_, g, _ = _tiny_case(fmt, 1, n, k, seed=57)
    c = 0.75                                              # exact in bf16
    x = np.full((1, k), np.float32(c)).view(np.uint32) >> 16
    ones = np.full(k, 0x3F80, np.uint16)
    ref, _ = reference.qmm_rmsnorm_ref(fmt, c_, s_, g, x.astype(np.uint16), "bf16", ones, eps, 1, n, k)
    w = reference.dequant_exact(fmt, c_, s_, g, n, k)
    want = (c / np.sqrt(c * c + eps)) * w.sum(axis=1)
    assert np.allclose(ref[0], want, rtol=1e-13, atol=1e-15)


def test_rmsnorm_values_invariant_under_power_of_two_scaling():
    m, k = 3, 256
    x = synth.activations_bf16(m, k, seed=58)
    gb = _gamma_bits(k, 59)
    a = reference.rmsnorm_values(x, "bf16", gb, 0.0, m, k)
    x4 = ((x.astype(np.uint32) + (2 << 7)) & 0xFFFF).astype(np.uint16)   # exponent + 2: x * 4 (no zeros here)
    assert (x & 0x7F80).min() > 0 and (x & 0x7F80).max() < 0x7E00
    b = reference.rmsnorm_values(x4, "bf16", gb, 0.0, m, k)
    assert np.array_equal(a, b)



def test_planted_rmsnorm_mistake_is_caught(monkeypatch):
    """A normalisation by the root of the sum (not the mean) of squares must fail the decimal pin."""
    def sum_not_mean(x, x_dtype, gamma_bits, eps, m, k):
        xv = reference.x_values(x, x_dtype).reshape(m, k)
        g = reference.codec.decode_bf16(np.asarray(gamma_bits, dtype=np.uint16)).reshape(k)
        return xv * g[None, :] / np.sqrt(np.sum(xv * xv, axis=1) + eps)[:, None]

    with monkeypatch.context() as mp:
        mp.setattr(reference, "rmsnorm_values", sum_not_mean)
        with pytest.raises(AssertionError):
            test_rmsnorm_ref_matches_decimal_brute_force("mxfp4")


# ----- the gated RMSNorm (PR #250 fused gated-RMSNorm + GEMV) -----

def _bf16(a):
    return synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def test_gated_rmsnorm_zero_gate_gives_zero():
    # silu(0) = 0: every gated value vanishes
    m, k = 2, 64
    x = synth.activations_bf16(m, k, seed=71)
    v = reference.gated_rmsnorm_values(x, _bf16(np.zeros((m, k))), "bf16", _gamma_bits(k, 72), 1e-5, m, k)
    assert not v.any()


def test_gated_rmsnorm_large_gate_is_the_gate_times_rmsnorm():
    # silu(z) = z / (1 + e^-z) equals z in float64 for z = 64 (e^-64 < 2^-53 relative):
    # the gated values are 64 x the plain (separately pinned) RMSNorm values
    m, k = 2, 128
    x = synth.activations_bf16(m, k, seed=73)
    gb = _gamma_bits(k, 74)
    v = reference.gated_rmsnorm_values(x, _bf16(np.full((m, k), 64.0)), "bf16", gb, 1e-5, m, k)
    assert np.array_equal(v, 64.0 * reference.rmsnorm_values(x, "bf16", gb, 1e-5, m, k))


def test_gated_rmsnorm_odd_part_of_the_gate_is_linear():
    # silu(z) - silu(-z) = z (sigmoid(z) + sigmoid(-z) = 1): a wrong activation
    # (sigmoid alone, z (1 - sigmoid), a sign slip) breaks this identity
    m, k = 2, 256
    x = synth.activations_bf16(m, k, seed=75)
    z = synth.activations_bf16(m, k, seed=76)
    zneg = z ^ np.uint16(0x8000)
    gb = _gamma_bits(k, 77)
    a = reference.gated_rmsnorm_values(x, z, "bf16", gb, 1e-3, m, k)
    b = reference.gated_rmsnorm_values(x, zneg, "bf16", gb, 1e-3, m, k)
    zv = reference.x_values(z, "bf16").reshape(m, k)
    want = zv * reference.rmsnorm_values(x, "bf16", gb, 1e-3, m, k)
    assert np.allclose(a - b, want, rtol=1e-12, atol=1e-15)


def test_gated_rmsnorm_large_negative_gate_vanishes():
    m, k = 1, 32
    x = synth.activations_bf16(m, k, seed=78)
    v = reference.gated_rmsnorm_values(x, _bf16(np.full((m, k), -1000.0)), "bf16", _gamma_bits(k, 79), 0.0, m, k)
    assert np.all(np.abs(v) < 1e-300)


# ----- int4 affine with a ragged last group (K a multiple of 32, not of 64) -----

@pytest.mark.parametrize("k", [32, 96, 160])
def test_ragged_int4_matches_exact_rational_brute_force(k):
    assert _check_brute("int4_affine", m=2, n=4, k=k, seed=k)


def test_ragged_int4_group_round_trips_exactly():
    # Every group (the 32-wide last one too) holds b + s q with q spanning 0..15,
    # s and b exact in bf16: the packer must find exactly s and b and the codes.
    n, k = 3, 96
    rng = np.random.default_rng(61)
    w = np.empty((n, k), np.float32)
    for r in range(n):
        for g0 in range(0, k, 64):
            width = min(64, k - g0)
            s = np.float32(2.0 ** rng.integers(-6, 2)) * np.float32(1.5)
            b = np.float32(rng.integers(-40, 40)) * np.float32(0.125)
            q = rng.integers(0, 16, size=width)
            q[0], q[-1] = 0, 15
            w[r, g0:g0 + width] = b + s * q.astype(np.float32)
    c, s_, g = pack.pack("int4_affine", w)
    assert c.shape == (n, k // 2) and s_.shape == (n, 2 * 4)
    assert np.array_equal(reference.dequant_exact("int4_affine", c, s_, g, n, k), w.astype(np.float64))


# ------------------- both operands quantized: the W . A8 product ---------------

_E4M3_VALUES = None


def _e4m3_table():
    """Every finite E4M3 code and its exact value, from torch's float8_e4m3fn (a library decode)."""
    global _E4M3_VALUES
    if _E4M3_VALUES is None:
        codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
        vals = codes.view(torch.float8_e4m3fn).double().numpy()
        _E4M3_VALUES = [(int(c), Fraction(float(v))) for c, v in enumerate(vals) if np.isfinite(v)]
    return _E4M3_VALUES


def _brute_e4m3(v: Fraction) -> int:
    # nearest finite E4M3 value, an exact tie to the code with mantissa bit 0,
    # beyond +-448 the largest; the sign bit copies v's sign (zero keeps +)
    best = None
    for c, val in _e4m3_table():
        if (c & 0x80) != (0x80 if v < 0 else 0):
            continue
        d = abs(val - v)
        key = (d, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def _brute_activation_quant(xrow):
    # one row: per block of 32, s = float32(amax / 448) (1 for a zero block),
    # e = the smallest integer with 2^e >= s, codes of float32(x / 2^e)
    codes, scodes = [], []
    for b in range(0, len(xrow), 32):
        blk = np.asarray(xrow[b:b + 32], np.float32)
        amax = np.float32(np.max(np.abs(blk)))
        s = Fraction(float(np.float32(amax / np.float32(448.0)))) if amax > 0 else Fraction(1)
        e = -127
        while Fraction(2) ** e < s:
            e += 1
        scodes.append(e + 127)
        for v in blk:
            q = np.float32(v) / np.float32(2.0 ** e)
            codes.append(_brute_e4m3(Fraction(float(q))))
    return codes, scodes


def test_activation_quantizer_matches_brute_force():
    rng = np.random.default_rng(3)
    m, k = 3, 96
    x = rng.standard_normal((m, k)).astype(np.float32)
    x[0] *= np.float32(1e-3)
    x[1, 32:64] = 0.0                                                    # a zero block: scale 1.0
    x[2, :32] = np.float32(448.0) * np.float32(2.0 ** -5)                # amax / 448 exactly a power of two
    xb = synth.f32_to_bf16_bits(x)
    c, s = reference.quantize_activations("mxfp8_e4m3", xb, "bf16", m, k)
    xv = reference.x_values(xb, "bf16").reshape(m, k)
    for i in range(m):
        bc, bs = _brute_activation_quant(xv[i])
        assert list(c[i]) == bc, i
        assert list(s[i]) == bs, i


def test_a8_product_matches_exact_rational_brute_force():
    fmt, m, n, k = "mxfp4", 2, 3, 64
    cw, sw, g = _tiny_case(fmt, m=m, n=n, k=k, seed=4)[:3]
    xb = synth.activations_bf16(m, k, seed=5)
    ref, bound = reference.qmm_a8_ref(fmt, cw, sw, g, xb, "bf16", m, n, k)
    xv = reference.x_values(xb, "bf16").reshape(m, k)
    for i in range(m):
        xc, xs = _brute_activation_quant(xv[i])
        vals = dict(_e4m3_table())
        x8 = [vals[xc[kk]] * Fraction(2) ** (xs[kk // 32] - 127) for kk in range(k)]
        for j in range(n):
            exact = sum(x8[kk] * _lib_elem(fmt, _code(fmt, cw[j], kk)) * _lib_scale(fmt, sw, j, kk // 32)[0]
                        for kk in range(k))
            assert ref[i, j] == float(exact)
            assert bound[i, j] > 0


def _representable_activations(m, k, seed):
    # every block: E4M3 values times one power of two, its largest magnitude in
    # (224, 448], so the packer's scale is that power and the codes its values
    rng = np.random.default_rng(seed)
    finite = np.array([float(v) for c, v in _e4m3_table() if c < 0x7F], np.float64)
    x = np.empty((m, k), np.float32)
    for i in range(m):
        for b in range(0, k, 32):
            e = int(rng.integers(-20, 20))
            v = rng.choice(finite, 32) * rng.choice([-1.0, 1.0], 32)
            v[int(rng.integers(0, 32))] = rng.choice([256.0, 288.0, 448.0, 240.0])
            x[i, b:b + 32] = (v * 2.0 ** e).astype(np.float32)
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8_e4m3", "nvfp4", "int4_affine"])
def test_a8_is_the_exact_product_when_x_is_representable(fmt):
    # quantizing an activation that is already MXFP8 E4M3 changes nothing: the
    # W . A8 reference equals the exact bf16-activation reference bit for bit
    m, n, k = 3, 7, 128
    xb = _representable_activations(m, k, seed=6)
    c, s, g = pack.pack(fmt, synth.weights(n, k, seed=7, outliers=(fmt == "nvfp4")))
    a8, _ = reference.qmm_a8_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    exact, _ = reference.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    assert np.array_equal(a8, exact)


def test_planted_activation_quantizer_mistake_is_caught(monkeypatch):
    # snapping the activation scale down (floor) instead of up saturates the
    # block maximum: the representable-activation identity fails
    from oracle import codec
    real = codec.e8m0_encode_ceil

    def floor_snap(s):
        c = real(s)
        exact_pow2 = np.asarray(codec.E8M0_TABLE[c], np.float32) == np.asarray(s, np.float32)
        return np.where(exact_pow2, c, c - 1).astype(c.dtype)

    monkeypatch.setattr(codec, "e8m0_encode_ceil", floor_snap)
    with pytest.raises(AssertionError):
        test_a8_is_the_exact_product_when_x_is_representable("mxfp4")


# ------------------- both operands quantized: the all-FP4 W . A4 product -------------


def _brute_e2m1(v: Fraction) -> int:
    # nearest E2M1 value (the two_m_int decode above), an exact tie to the code
    # with mantissa bit 0, beyond +-6 the largest; the sign bit copies v's sign
    best = None
    for c in range(16):
        if (c & 8) != (8 if v < 0 else 0):
            continue
        key = (abs(_lib_elem("mxfp4", c) - v), c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def _brute_activation_quant_e2m1(xrow):
    # per block of 32: s = float32(amax / 6) (1 for a zero block), e = the
    # smallest integer with 2^e >= s, codes of float32(x / 2^e)
    codes, scodes = [], []
    for b in range(0, len(xrow), 32):
        blk = np.asarray(xrow[b:b + 32], np.float32)
        amax = np.float32(np.max(np.abs(blk)))
        s = Fraction(float(np.float32(amax / np.float32(6.0)))) if amax > 0 else Fraction(1)
        e = -127
        while Fraction(2) ** e < s:
            e += 1
        scodes.append(e + 127)
        for v in blk:
            codes.append(_brute_e2m1(Fraction(float(np.float32(v) / np.float32(2.0 ** e)))))
    return codes, scodes


def _a4_activations(m, k, seed):
    # N(0, 1) values, then in every row's first block the grid's midpoints
    # (0.25, 1.25, 1.75, 2.5, 3.5, 5, of either sign) under a block maximum of 6
    # times a power of two, so that the ties are exact
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k)).astype(np.float32)
    mids = np.array([6.0, 0.25, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -2.5, -5.0, -1.75, 0.75], np.float32)
    for i in range(m):
        x[i, :len(mids)] = mids * np.float32(2.0 ** (i - 1))
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8_e4m3"])
def test_a4_product_matches_exact_rational_brute_force(fmt):
    m, n, k = 2, 3, 64
    cw, sw, g = _tiny_case(fmt, m=m, n=n, k=k, seed=11)[:3]
    xb = _a4_activations(m, k, seed=12)
    ref, bound = reference.qmm_a4_ref(fmt, cw, sw, g, xb, "bf16", m, n, k)
    xv = reference.x_values(xb, "bf16").reshape(m, k)
    for i in range(m):
        xc, xs = _brute_activation_quant_e2m1(xv[i])
        x4 = [_lib_elem("mxfp4", xc[kk]) * Fraction(2) ** (xs[kk // 32] - 127) for kk in range(k)]
        for j in range(n):
            exact = sum(x4[kk] * _lib_elem(fmt, _code(fmt, cw[j], kk)) * _lib_scale(fmt, sw, j, kk // 32)[0]
                        for kk in range(k))
            assert ref[i, j] == float(exact), (fmt, i, j)
            assert bound[i, j] > 0


def _e2m1_representable_activations(m, k, seed):
    # every block: E2M1 values times one power of two, its largest magnitude
    # in (3, 6], so the packer's scale is that power and the codes its values
    rng = np.random.default_rng(seed)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    x = np.empty((m, k), np.float32)
    for i in range(m):
        for b in range(0, k, 32):
            e = int(rng.integers(-20, 20))
            v = rng.choice(grid, 32) * rng.choice([-1.0, 1.0], 32)
            v[int(rng.integers(0, 32))] = rng.choice([4.0, 6.0, -4.0, -6.0])
            x[i, b:b + 32] = (v * 2.0 ** e).astype(np.float32)
    return synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("fmt", ["mxfp4", "mxfp8_e4m3", "int4_affine"])
def test_a4_is_the_exact_product_when_x_is_representable(fmt):
    # quantizing an activation that is already MXFP4 changes nothing: the
    # W . A4 reference equals the exact bf16-activation reference bit for bit
    m, n, k = 3, 7, 128
    xb = _e2m1_representable_activations(m, k, seed=13)
    c, s, g = pack.pack(fmt, synth.weights(n, k, seed=14, outliers=(fmt == "nvfp4")))
    a4, _ = reference.qmm_a4_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    exact, _ = reference.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    assert np.array_equal(a4, exact)


def test_planted_e2m1_tie_mistake_is_caught(monkeypatch):
    # ties rounded away from zero instead of to the even code (every input
    # nudged one float32 ulp outward): the brute force over the grid's
    # midpoints catches it
    from oracle import codec
    real = codec.encode_rne_sat

    def away(v, fmt):
        if fmt != "e2m1":
            return real(v, fmt)
        v = np.asarray(v, np.float32)
        return real(np.nextafter(v, np.sign(v) * np.float32(np.inf)).astype(np.float32), fmt)

    monkeypatch.setattr(codec, "encode_rne_sat", away)
    with pytest.raises(AssertionError):
        test_a4_product_matches_exact_rational_brute_force("mxfp4")


def test_planted_a4_scale_divisor_mistake_is_caught(monkeypatch):
    # the MXFP4 scale taken from amax / 448 (E4M3's largest) instead of amax / 6:
    # the block maxima saturate and the representable-activation identity fails
    from oracle import pack as opack
    monkeypatch.setitem(opack._ELEM, "mxfp4", ("e2m1", 448.0))
    with pytest.raises(AssertionError):
        test_a4_is_the_exact_product_when_x_is_representable("mxfp4")


# ------------------- the all-FP4 product over nvfp4: NVFP4 activations -------------------


def _brute_activation_quant_nvfp4(x):
    # the whole X is one tensor: global g = float32(amax(X) / 2688) (1 for a
    # zero X); per block of 16: t = float32(float32(amax / 6) / g), its scale
    # the nearest E4M3 code (a zero block: 0x38 = 1.0), eff = float32(E4M3 * g),
    # codes the nearest E2M1 of float32(x / eff) (eff = 0: code 0)
    x = np.asarray(x, np.float32)
    amax_t = np.float32(np.max(np.abs(x)))
    g = np.float32(amax_t / np.float32(2688.0)) if amax_t > 0 else np.float32(1.0)
    vals = dict(_e4m3_table())
    codes, scodes = [], []
    for row in x:
        rc, rs = [], []
        for b in range(0, len(row), 16):
            blk = row[b:b + 16]
            amax = np.float32(np.max(np.abs(blk)))
            if amax > 0:
                t = np.float32(np.float32(amax / np.float32(6.0)) / g)
                sc = _brute_e4m3(Fraction(float(t)))
            else:
                sc = 0x38
            rs.append(sc)
            eff = np.float32(np.float32(float(vals[sc])) * g)
            for v in blk:
                rc.append(0 if eff == 0 else _brute_e2m1(Fraction(float(np.float32(v / eff)))))
        codes.append(rc)
        scodes.append(rs)
    return codes, scodes, g


def test_nvfp4_activation_quantizer_matches_brute_force():
    m, k = 3, 64
    xb = _a4_activations(m, k, seed=71)
    c, s, g = reference.quantize_activations_global("nvfp4", xb, "bf16", m, k)
    xv = reference.x_values(xb, "bf16").reshape(m, k)
    bc, bs, bg = _brute_activation_quant_nvfp4(xv)
    assert np.float32(g) == bg
    for i in range(m):
        assert [_code("nvfp4", c[i], kk) for kk in range(k)] == bc[i], i
        assert list(s[i]) == bs[i], i


def test_a4_nvfp4_product_matches_exact_rational_brute_force():
    m, n, k = 2, 3, 64
    cw, sw, gw = _tiny_case("nvfp4", m=m, n=n, k=k, seed=72)[:3]
    xb = _a4_activations(m, k, seed=73)
    ref, bound = reference.qmm_a4_ref("nvfp4", cw, sw, gw, xb, "bf16", m, n, k)
    xv = reference.x_values(xb, "bf16").reshape(m, k)
    bc, bs, bg = _brute_activation_quant_nvfp4(xv)
    vals = dict(_e4m3_table())
    for i in range(m):
        x4 = [_lib_elem("nvfp4", bc[i][kk]) * vals[bs[i][kk // 16]] * Fraction(float(bg)) for kk in range(k)]
        for j in range(n):
            exact = sum(x4[kk] * _lib_elem("nvfp4", _code("nvfp4", cw[j], kk)) * _lib_scale("nvfp4", sw, j, kk // 16)[0]
                        for kk in range(k)) * Fraction(float(gw))
            # ref is an fp64 matmul: within a few fp64 ulps of the exact rational sum
            scale = sum(abs(x4[kk] * _lib_elem("nvfp4", _code("nvfp4", cw[j], kk))
                            * _lib_scale("nvfp4", sw, j, kk // 16)[0]) for kk in range(k)) * Fraction(float(gw))
            assert abs(Fraction(ref[i, j]) - exact) <= Fraction(1, 2 ** 48) * scale, (i, j)
            assert bound[i, j] > 0


def _nvfp4_representable_activations(m, k, seed):
    # g = 2^-3: one block holds 6 * 448 * g (the tensor maximum, so the
    # global is g exactly); every block is E2M1 values times s_b g with s_b an
    # E4M3 value and one element 6 s_b g, so its scale is s_b and its codes
    # its values
    rng = np.random.default_rng(seed)
    g = 2.0 ** -3
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    e4 = [float(v) for c, v in _e4m3_table() if 0 < c < 0x7F and float(v) >= 2.0 ** -6]
    x = np.empty((m, k), np.float32)
    for i in range(m):
        for b in range(0, k, 16):
            sb = 448.0 if (i, b) == (0, 0) else float(rng.choice(e4))
            v = rng.choice(grid, 16) * rng.choice([-1.0, 1.0], 16)
            v[int(rng.integers(0, 16))] = rng.choice([6.0, -6.0])
            x[i, b:b + 16] = (v * sb * g).astype(np.float32)
    return synth.f32_to_bf16_bits(x)


def test_a4_nvfp4_is_the_exact_product_when_x_is_representable():
    m, n, k = 3, 7, 128
    xb = _nvfp4_representable_activations(m, k, seed=74)
    assert np.array_equal(reference.x_values(xb, "bf16").reshape(m, k).astype(np.float32),
                          reference.x_values(xb, "bf16").reshape(m, k))   # bf16-exact construction
    c, s, g = pack.pack("nvfp4", synth.weights(n, k, seed=75, outliers=True))
    a4, _ = reference.qmm_a4_ref("nvfp4", c, s, g, xb, "bf16", m, n, k)
    exact, _ = reference.qmm_ref("nvfp4", c, s, g, xb, "bf16", m, n, k)
    assert np.array_equal(a4, exact)


def test_planted_dropped_activation_global_is_caught(monkeypatch):
    # the NVFP4 activation dequantized without its global: the identity fails
    real = reference.quantize_activations_global

    def no_global(fmt, x, x_dtype, m, k):
        c, s, g = real(fmt, x, x_dtype, m, k)
        return c, s, np.float32(1.0)

    monkeypatch.setattr(reference, "quantize_activations_global", no_global)
    with pytest.raises(AssertionError):
        test_a4_nvfp4_is_the_exact_product_when_x_is_representable()


def test_planted_nvfp4_scale_rounding_mistake_is_caught(monkeypatch):
    # the E4M3 block scale truncated toward zero instead of rounded to nearest:
    # the brute-force quantizer catches it
    from oracle import codec
    real = codec.encode_rne_sat

    def trunc(v, fmt):
        if fmt != "e4m3":
            return real(v, fmt)
        v = np.asarray(v, np.float32)
        c = real(v, fmt)
        over = np.abs(codec.E4M3_TABLE[c]) > np.abs(v.astype(np.float64))
        return np.where(over & (c & 0x7F > 0), c - 1, c).astype(np.uint8)

    monkeypatch.setattr(codec, "encode_rne_sat", trunc)
    with pytest.raises(AssertionError):
        test_nvfp4_activation_quantizer_matches_brute_force()
