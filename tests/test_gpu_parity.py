"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

* dequant: bit-exact float32 (u32 patterns; any NaN matches any NaN).
* qmm: |out - ref| <= 2e-3 * sum_k |x||w| + 1e-6 elementwise, ref the exact
  float64 dequant-then-dot, plus the final rounding of a bf16 output (half a
  bf16 ulp of the stored value; see tests/tolerance.py).
Inputs: seeded synthetic weights packed by the oracle's packer (so no oracle
input comes from the library), bf16 activations from the shared generator.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_scaled_quantized_spec_gb300 as q  # noqa: E402
from block_scaled_quantized_spec_gb300 import synth  # noqa: E402
from oracle import pack as opack  # noqa: E402
from oracle import reference as oref  # noqa: E402
from tolerance import bf16_half_ulp, check, check_tensor  # noqa: E402

pytestmark = pytest.mark.gpu
FMTS = list(q.FORMATS)
GROUP64 = ["int4_affine", "int8", "int8_f16", "int4", "int4_f16",         # group of 64: K may end in a group of 32
           "int2", "int3", "int5", "int6", "int2_f16", "int3_f16", "int5_f16", "int6_f16"]
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_quantized_spec_gb300 import build
    build.build()
    q.load()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _packed(fmt, n, k, seed, std=0.02):
    w = synth.weights(n, k, seed=seed, std=std, outliers=(fmt == "nvfp4"))
    return opack.pack(fmt, w)


def _x(m, k, seed):
    xb = synth.activations_bf16(m, k, seed=seed)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    return xb, xt


def _check_qmm(out_t, ref, bound, what):
    return check_tensor(out_t, ref, bound, what)


# ------------------------------------------------------------------ dequant ---

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("n,k", [(1, 64), (67, 512), (256, 2048)])
def test_dequant_bit_exact(fmt, n, k):
    c, s, g = _packed(fmt, n, k, seed=n + k)
    want = oref.dequant_f32(fmt, c, s, g, n, k)
    got = q.qfmt_dequant(fmt, _dev(c), _dev(s), g, n, k).cpu().numpy()
    wb, gb = want.view(np.uint32), got.view(np.uint32)
    same = (wb == gb) | (np.isnan(want) & np.isnan(got))
    assert same.all(), (fmt, np.argwhere(~same)[:5].tolist())


@pytest.mark.parametrize("fmt", FMTS)
def test_dequant_all_codes_and_scales(fmt):
    # every code byte against every scale class, including special values the
    # packer never emits (NaN/Inf element codes, E8M0 0 and 255, subnormals)
    rng = np.random.default_rng(5)
    n, k = 64, 512
    cb = opack.codes_nbytes(fmt, n, k)
    codes = np.tile(np.arange(256, dtype=np.uint8), cb // 256 + 1)[:cb].reshape(n, -1)
    sb = opack.scales_nbytes(fmt, n, k)
    if fmt in ("mxfp4", "mxfp8_e4m3", "mxfp8_e5m2", "mxint8", "mxint4", "nvfp4") or fmt.startswith("mxint"):
        scales = np.tile(np.arange(256, dtype=np.uint8), sb // 256 + 1)[:sb]
    elif fmt in ("nvfp8", "int8", "int4", "mxfp4x2", "fp4", "fp8_e4m3", "fp8_e5m2", "int2", "int3", "int5", "int6"):
        scales = np.concatenate([rng.standard_normal(sb // 4 - 4).astype(np.float32),
                                 np.array([1e-40, 3e38, 0.0, -2.5], np.float32)]).view(np.uint8)
    elif fmt.endswith("_f16"):   # evenly spaced half bit patterns: subnormals, +-inf, NaNs, both signs
        scales = np.arange(0, 65536, 65536 // (sb // 2), dtype=np.uint16)[:sb // 2].view(np.uint8)
    else:
        sc = synth.f32_to_bf16_bits(rng.standard_normal(sb // 2).astype(np.float32) * 1e-2)
        scales = sc.view(np.uint8)
    scales = scales.reshape(n, -1)
    g = 0.75
    want = oref.dequant_f32(fmt, codes, scales, g, n, k)
    got = q.qfmt_dequant(fmt, _dev(codes), _dev(scales), g, n, k).cpu().numpy()
    same = (want.view(np.uint32) == got.view(np.uint32)) | (np.isnan(want) & np.isnan(got))
    assert same.all(), (fmt, np.argwhere(~same)[:5].tolist())


def test_dequant_bf16_output_is_rounded_f32():
    fmt, n, k = "nvfp8", 32, 256
    c, s, g = _packed(fmt, n, k, seed=3)
    want = synth.f32_to_bf16_bits(oref.dequant_f32(fmt, c, s, g, n, k))
    got = q.qfmt_dequant(fmt, _dev(c), _dev(s), g, n, k, out_dtype=torch.bfloat16)
    assert np.array_equal(got.view(torch.int16).cpu().numpy().view(np.uint16), want)


# ---------------------------------------------------------------------- qmm ---

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 2, 5, 8, 9, 16])
def test_qgemv_parity(fmt, m):
    n, k = 200, 1024                       # 12.5 row tiles (ragged), several K chunks per warp
    c, s, g = _packed(fmt, n, k, seed=m)
    xb, xt = _x(m, k, seed=100 + m)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [17, 64, 130, 256])
def test_qgemm_parity(fmt, m):
    n, k = 272, 1024
    c, s, g = _packed(fmt, n, k, seed=m)
    xb, xt = _x(m, k, seed=200 + m)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m))


@pytest.mark.parametrize("fmt", FMTS[:20])
def test_qgemm_tile_orders(fmt):
    # the bf16-decode GEMM walks the M tiles of an N tile first when the
    # activations are the smaller operand (here X 0.5 MB, W 0.6-1.3 MB), the N
    # tiles of an M tile first otherwise; both orders forced (debug key 8) over
    # 4 x 20-40 tiles with ragged last M and N tiles agree with the oracle and,
    # accumulating in the same order, with each other bit for bit
    m, n, k = 1000, 5000, 256
    c, s, g = _packed(fmt, n, k, seed=31)
    xb, xt = _x(m, k, seed=32)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    outs = []
    try:
        for order in (0, 1, 2):
            q.qfmt_debug_set(8, order)
            out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
            _check_qmm(out, ref, bound, (fmt, "order", order))
            outs.append(out.float().cpu().numpy())
    finally:
        q.qfmt_debug_set(8, 0)
    assert np.array_equal(outs[1], outs[2])


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [3, 40, 130])
def test_short_and_odd_k(fmt, m):
    # K of one block quantum and K that leave partial chunks / K steps; few terms
    # per output, so a per-weight rounding above the bound would show
    for k in (32, 64, 96, 160, 192) if fmt in GROUP64 else (32, 96, 160):   # group 64: ragged last groups too
        n = 33 if m < 17 else 300
        c, s, g = _packed(fmt, n, k, seed=k)
        xb, xt = _x(m, k, seed=k + 1)
        out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
        ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
        _check_qmm(out, ref, bound, (fmt, k))


def test_tiny_config_f32_activations():
    # mxfp4, M=8, N=16, K=512, W ~ N(0, 0.02), X f32 ~ N(0, 1), out f32, seed 0
    fmt, m, n, k = "mxfp4", 8, 16, 512
    rng = np.random.default_rng(0)
    w = synth.weights(n, k, rng=rng)
    x = synth.activations_f32(m, k, rng=rng)
    c, s, g = opack.pack(fmt, w)
    out = q.qmm_ex(fmt, _dev(c), _dev(s), g, _dev(x), n)
    assert out.dtype == torch.float32
    ref, bound = oref.qmm_ref(fmt, c, s, g, x, "f32", m, n, k)
    _check_qmm(out, ref, bound, "tiny")


@pytest.mark.parametrize("fmt", FMTS)
def test_f32_activations_all_formats(fmt):
    m, n, k = 20, 40, 256
    c, s, g = _packed(fmt, n, k, seed=7)
    x = synth.activations_f32(m, k, seed=8)
    out = q.qmm_ex(fmt, _dev(c), _dev(s), g, _dev(x), n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, x, "f32", m, n, k)
    _check_qmm(out, ref, bound, fmt)


def test_gemv_gemm_boundary_agree():
    # the same rows computed by the M<=16 and M>16 kernels agree within the bound
    fmt, n, k = "mxfp4", 256, 2048
    c, s, g = _packed(fmt, n, k, seed=1)
    xb, xt = _x(17, k, seed=2)
    o16 = q.qmm(fmt, _dev(c), _dev(s), g, xt[:16].contiguous(), n).float().cpu().numpy()
    o17 = q.qmm(fmt, _dev(c), _dev(s), g, xt, n).float().cpu().numpy()
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", 17, n, k)
    # each side within bound + its half ulp of the exact value
    assert (np.abs(o16 - o17[:16]) <= 2 * bound[:16] + bf16_half_ulp(o16) + bf16_half_ulp(o17[:16])).all()


def test_batch_rows_equal_single_rows():
    fmt, n, k, m = "nvfp4", 96, 512, 8
    c, s, g = _packed(fmt, n, k, seed=4)
    xb, xt = _x(m, k, seed=5)
    dc, ds = _dev(c), _dev(s)
    full = q.qmm(fmt, dc, ds, g, xt, n).float().cpu().numpy()
    for i in range(m):
        one = q.qmm(fmt, dc, ds, g, xt[i:i + 1].contiguous(), n).float().cpu().numpy()
        ref, bound = oref.qmm_ref(fmt, c, s, g, xb[i:i + 1], "bf16", 1, n, k)
        assert (np.abs(one[0] - full[i]) <= 2 * bound[0] + bf16_half_ulp(one[0]) + bf16_half_ulp(full[i])).all()


def test_empty_and_zero_k():
    c = torch.zeros(256, dtype=torch.uint8, device=DEV)   # the packed bytes of a [4, 64] mxfp4 weight
    s = torch.zeros(256, dtype=torch.uint8, device=DEV)
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    out = q.qmm("mxfp4", c, s, 1.0, x, 4)
    assert out.shape == (0, 4)
    x2 = torch.zeros((3, 0), dtype=torch.bfloat16, device=DEV)
    out2 = torch.full((3, 5), 7.0, dtype=torch.bfloat16, device=DEV)
    q.qmm("mxfp4", c, s, 1.0, x2, 5, out=out2)
    assert (out2.float() == 0).all()


def test_misaligned_device_pointer_rejected():
    fmt, n, k = "mxfp4", 16, 64
    c, s, g = _packed(fmt, n, k, seed=1)
    dc = _dev(np.concatenate([np.zeros(8, np.uint8), c.ravel()]))
    xb, xt = _x(1, k, seed=1)
    with pytest.raises(q.QfmtError) as e:
        q.qmm(fmt, dc[8:], _dev(s), g, xt, n)
    assert e.value.status == -3


# ------------------------------------------- full-size workloads, every output

# The workloads of the method at full size, in the launch configuration the
# benchmark times (the tile shapes, K splits and CTA plans chosen there):
# mxfp4 1x4096x4096; nvfp4 {1, 8}x14336x4096 with outliers; mxfp8 E4M3
# 2048x4096x4096; the int4-affine / mxfp8 E5M2 / nvfp8 sweep
# {1, 16, 128, 4096}x11008x4096; and one or more shapes of each added format.
FULL = [
    ("mxfp4", 1, 4096, 4096, False),
    ("nvfp4", 1, 14336, 4096, True),
    ("nvfp4", 8, 14336, 4096, True),
    ("mxfp8_e4m3", 2048, 4096, 4096, False),
    ("int4_affine", 1, 11008, 4096, False),
    ("int4_affine", 16, 11008, 4096, False),
    ("int4_affine", 128, 11008, 4096, False),
    ("int4_affine", 4096, 11008, 4096, False),
    ("mxfp8_e5m2", 1, 11008, 4096, False),
    ("mxfp8_e5m2", 16, 11008, 4096, False),
    ("mxfp8_e5m2", 128, 11008, 4096, False),
    ("mxfp8_e5m2", 4096, 11008, 4096, False),
    ("nvfp8", 1, 11008, 4096, False),
    ("nvfp8", 16, 11008, 4096, False),
    ("nvfp8", 128, 11008, 4096, False),
    ("nvfp8", 4096, 11008, 4096, False),
    ("mxint8", 1, 11008, 4096, False),
    ("mxint8", 4096, 11008, 4096, False),
    ("int8", 1, 11008, 4096, False),
    ("int8", 4096, 11008, 4096, False),
    ("int4", 1, 11008, 4096, False),
    ("int4", 16, 11008, 4096, False),
    ("int4_f16", 4096, 11008, 4096, False),
    ("mxfp4x2", 1, 4096, 4096, False),
    ("mxfp4x2", 16, 4096, 4096, False),
    ("mxfp4x2", 2048, 4096, 4096, False),
    ("mxint4", 1, 4096, 4096, False),
    ("mxint4", 8, 4096, 4096, False),
    ("mxint4", 2048, 4096, 4096, False),
    ("fp4", 1, 4096, 4096, False),
    ("fp8_e5m2_f16", 16, 11008, 4096, False),
    ("fp8_e4m3", 2048, 4096, 4096, False),
    ("int3", 1, 11008, 4096, False),          # the sub-byte bit streams on their CUDA-core kernel
    ("mxint5", 16, 4096, 4096, False),
    ("int6_f16", 128, 4096, 4096, False),
    ("int2", 1, 4096, 4096, False),
]


_PACKED = {}


def _full_packed(fmt, n, k, outl):
    key = (fmt, n, k, outl)
    if key not in _PACKED:
        _PACKED.clear()
        w = synth.weights(n, k, seed=0, outliers=outl)
        _PACKED[key] = opack.pack(fmt, w)
    return _PACKED[key]


@pytest.mark.parametrize("fmt,m,n,k,outl", FULL)
def test_full_size_every_output(fmt, m, n, k, outl):
    # every output element of the full workload against the float64 oracle
    c, s, g = _full_packed(fmt, n, k, outl)
    xb, xt = _x(m, k, seed=1 + m)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m, n, k))


# ------------------------------------------------------------ special codes ---

MX_FMTS = ["mxfp4", "mxfp8_e4m3", "mxfp8_e5m2", "mxint8", "mxint4"]


def _nonfinite_rows_only(out, ref, bound, bad_rows, what):
    # the outputs of the weight rows holding a non-finite weight are non-finite;
    # every other output is within the tolerance
    assert (~np.isfinite(out[:, bad_rows])).all(), (what, "a non-finite weight gave a finite output")
    keep = np.ones(out.shape[1], bool)
    keep[bad_rows] = False
    check(out[:, keep], ref[:, keep], bound[:, keep], what)


@pytest.mark.parametrize("fmt", MX_FMTS)
@pytest.mark.parametrize("m", [1, 2, 5, 17, 130, 2048])
def test_e8m0_special_scales(fmt, m):
    # E8M0 code 0 (2^-127, a float32 subnormal) among ordinary scales, then a
    # 255 (NaN) scale: the NaN reaches exactly the outputs of its weight row
    # (rlx-cpu lowp_scaled_matmul multiplies every block sum by its scale);
    # M spans the decode GEMVs and the tensor-core GEMM
    n, k = 48, 256
    c, s, g = _packed(fmt, n, k, seed=31)
    rng = np.random.default_rng(32)
    s = s.copy()
    s[rng.random(s.shape) < 0.2] = 0
    s[3, :] = 0
    xb, xt = _x(m, k, seed=33)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m, "zero scales"))
    s[5, 2] = 255
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n).float().cpu().numpy()
    assert np.isnan(out[:, 5]).all()
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _nonfinite_rows_only(out, ref, bound, [5], (fmt, m, "NaN scale"))


SPECIAL_CODES = {   # element codes outside the packer's range and the rows they are planted in
    "mxfp8_e4m3": [0x7F, 0xFF],            # the E4M3 NaNs
    "nvfp8": [0x7F, 0xFF],
    "fp8_e4m3": [0xFF],
    "mxfp8_e5m2": [0x7C, 0xFC, 0x7E],      # E5M2 +inf, -inf, NaN
    "fp8_e5m2_f16": [0x7C, 0xFD],
}


@pytest.mark.parametrize("fmt", list(SPECIAL_CODES))
@pytest.mark.parametrize("m", [1, 5, 17, 130, 2048])
def test_special_element_codes(fmt, m):
    # NaN / Inf element codes (the pages' E4M3 NaN S.1111.111, E5M2 as the
    # IEEE half's high byte): every output of the weight row holding one is
    # non-finite, on every path; the other outputs stay within the tolerance
    n, k = 40, 256
    c, s, g = _packed(fmt, n, k, seed=34)
    c = c.copy()
    rows = []
    for i, code in enumerate(SPECIAL_CODES[fmt]):
        r = 7 + 11 * i
        c[r, 37 + 64 * i] = code
        rows.append(r)
    xb, xt = _x(m, k, seed=35)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n).float().cpu().numpy()
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _nonfinite_rows_only(out, ref, bound, rows, (fmt, m))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [3, 12, 16])
def test_batch_gemv_split_k_ragged(fmt, m):
    # K not a multiple of 128 and large enough that 3 <= M <= 16 splits it over
    # a cluster of CTAs: the last K part ends inside a chunk; N ends inside a
    # 64-row CTA tile
    n, k = 100, (2112 if fmt == "int4_affine" else 2080)
    c, s, g = _packed(fmt, n, k, seed=40 + m)
    xb, xt = _x(m, k, seed=41 + m)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m, k))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [2, 16])
def test_gemv_fallback_long_k(fmt, m):
    # K too long for the activation slices of the register-direct GEMVs: the
    # bulk-copy GEMV takes it in several K passes
    n, k = 48, 24576
    c, s, g = _packed(fmt, n, k, seed=50 + m)
    xb, xt = _x(m, k, seed=51 + m)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m, k))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 2])
@pytest.mark.parametrize("n", [1000, 4000])
def test_staged_weight_gemv(fmt, m, n):
    # at most two 16-row tiles an SM and whole rounds of chunks: the E2M1
    # formats' M <= 2 GEMV bulk-copies each 16-warp CTA's two tiles of weight
    # and scale rows into shared memory as it starts (one tile a CTA at N =
    # 1000, two for most CTAs at N = 4000); N ends inside a tile, whose rows
    # past N are not copied; the other formats take the register form
    k = 2048
    c, s, g = _packed(fmt, n, k, seed=70 + m)
    xb, xt = _x(m, k, seed=71 + m)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m))


@pytest.mark.parametrize("fmt", MX_FMTS)
@pytest.mark.parametrize("m", [1, 2])
def test_staged_weight_gemv_special_scales(fmt, m):
    # the staged GEMV's exact E8M0 decode: zero scales among ordinary ones,
    # then a NaN scale that reaches exactly its row's outputs
    n, k = 300, 2048
    c, s, g = _packed(fmt, n, k, seed=75)
    s = s.copy()
    s[np.random.default_rng(76).random(s.shape) < 0.2] = 0
    s[7, :] = 0
    xb, xt = _x(m, k, seed=77)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m, "zero scales"))
    s[9, 40] = 255
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n).float().cpu().numpy()
    assert np.isnan(out[:, 9]).all()
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _nonfinite_rows_only(out, ref, bound, [9], (fmt, m, "NaN scale"))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [3, 8, 9, 16])
def test_batch_gemv_one_decode(fmt, m):
    # 3 <= M <= 16 with K a multiple of 256 and at least 76 16-row tiles: one
    # decode of each weight block serves every activation row (the rows are
    # the MMA's columns, 8 a set); N ends inside a tile
    n, k = 1300, 1024
    c, s, g = _packed(fmt, n, k, seed=90 + m)
    xb, xt = _x(m, k, seed=91 + m)
    dc, ds = _dev(c), _dev(s)
    out = q.qmm(fmt, dc, ds, g, xt, n)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m))
    q.qfmt_debug_set(7, 1)                 # the same rows through the K-split batch GEMV
    try:
        other = q.qmm(fmt, dc, ds, g, xt, n).float().cpu().numpy()
    finally:
        q.qfmt_debug_set(7, 0)
    a = out.float().cpu().numpy()
    assert (np.abs(a - other) <= 2 * bound + bf16_half_ulp(a) + bf16_half_ulp(other)).all()


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4", "int4_affine", "mxint4", "mxfp8_e5m2", "nvfp8", "int8", "mxfp4x2"])
def test_batch_gemv_several_tiles_a_cta(fmt):
    # 313 tiles over one CTA an SM: up to three tiles a CTA, two blocks a warp,
    # so the loads run ahead across tile ends; float32 output
    m, n, k = 16, 5000, 512
    c, s, g = _packed(fmt, n, k, seed=95)
    xb, xt = _x(m, k, seed=96)
    out = q.qmm_ex(fmt, _dev(c), _dev(s), g, xt, n, out_dtype=torch.float32)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, fmt)


@pytest.mark.parametrize("fmt", MX_FMTS)
def test_batch_gemv_special_scales(fmt):
    # E8M0 0 and 255 scales on the one-decode batch GEMV
    m, n, k = 5, 1300, 512
    c, s, g = _packed(fmt, n, k, seed=97)
    s = s.copy()
    s[np.random.default_rng(98).random(s.shape) < 0.2] = 0
    s[11, :] = 0
    xb, xt = _x(m, k, seed=99)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, "zero scales"))
    s[13, 3] = 255
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n).float().cpu().numpy()
    assert np.isnan(out[:, 13]).all()
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _nonfinite_rows_only(out, ref, bound, [13], (fmt, "NaN scale"))


@pytest.mark.parametrize("fmt", list(SPECIAL_CODES))
def test_batch_gemv_special_element_codes(fmt):
    # NaN / Inf element codes on the one-decode batch GEMV: exactly their rows'
    # outputs are non-finite
    m, n, k = 5, 1300, 512
    c, s, g = _packed(fmt, n, k, seed=36)
    c = c.copy()
    rows = []
    for i, code in enumerate(SPECIAL_CODES[fmt]):
        r = 17 + 101 * i
        c[r, 45 + 64 * i] = code
        rows.append(r)
    xb, xt = _x(m, k, seed=37)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n).float().cpu().numpy()
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _nonfinite_rows_only(out, ref, bound, rows, (fmt, m))


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4", "int4_affine", "int4", "mxint4"])
@pytest.mark.parametrize("m", [1, 2])
def test_wide_gemv_four_warp_ctas(fmt, m):
    # more 16-row tiles than two per SM: the 4-bit GEMV runs 4-warp CTAs; N
    # ends inside a tile and K leaves a partial round
    n, k = 6000, 1152
    c, s, g = _packed(fmt, n, k, seed=60 + m)
    xb, xt = _x(m, k, seed=61 + m)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m))


@pytest.mark.parametrize("fmt,m", [("mxfp4", 1), ("nvfp8", 2), ("nvfp4", 8), ("int4_affine", 16),
                                   ("mxfp8_e4m3", 64), ("mxfp8_e5m2", 200)])
def test_chained_layers_read_the_previous_output(fmt, m):
    # Every kernel lets the next launch start early (programmatic dependent
    # launch) and reads X only after waiting for the preceding kernel.  A chain
    # of square layers, X(i+1) = out(i), launched back to back on one stream:
    # each layer must match the oracle on the input it was actually given.
    n = k = 512
    layers = 6
    packed = [_packed(fmt, n, k, seed=70 + i) for i in range(layers)]
    dev = [(_dev(c), _dev(s), g) for c, s, g in packed]
    xb, xt = _x(m, k, seed=80)
    outs = [xt]
    for i in range(layers):
        dc, ds, g = dev[i]
        outs.append(q.qmm(fmt, dc, ds, g, outs[-1], n))
    torch.cuda.synchronize()
    for i in range(layers):
        xin = outs[i].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        c, s, g = packed[i]
        ref, bound = oref.qmm_ref(fmt, c, s, g, xin, "bf16", m, n, k)
        _check_qmm(outs[i + 1], ref, bound, (fmt, m, "layer", i))


@pytest.mark.parametrize("fmt", GROUP64)
@pytest.mark.parametrize("m", [1, 2, 5, 16, 40, 300])
def test_ragged_last_group_every_path(fmt, m):
    # K = 64 * 32 + 32: the last group of 64 holds 32 values (its own scale, and bias for int4 affine)
    n, k = 136, 2080
    c, s, g = _packed(fmt, n, k, seed=90 + m)
    xb, xt = _x(m, k, seed=91 + m)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m, k))
    if m == 2:   # the float32-activation path over the same weights
        xf = synth.activations_f32(m, k, seed=92)
        out_f = q.qmm_ex(fmt, _dev(c), _dev(s), g, _dev(xf), n)
        ref_f, bound_f = oref.qmm_ref(fmt, c, s, g, xf, "f32", m, n, k)
        _check_qmm(out_f, ref_f, bound_f, (fmt, "f32", k))
    if m == 1:
        want = oref.dequant_f32(fmt, c, s, g, n, k)
        got = q.qfmt_dequant(fmt, _dev(c), _dev(s), g, n, k).cpu().numpy()
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))



@pytest.mark.parametrize("fmt", GROUP64)
def test_ragged_last_group_long_k_fallback(fmt):
    # two rows of K = 64 * 384 + 32: past the single-pass GEMVs' shared-memory plans
    m, n, k = 2, 48, 24608
    c, s, g = _packed(fmt, n, k, seed=95)
    xb, xt = _x(m, k, seed=96)
    out = q.qmm(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    _check_qmm(out, ref, bound, (fmt, m, k))
