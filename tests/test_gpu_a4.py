"""GPU parity of the all-FP4 product (qmm_a4) against the oracle.

The activation is packed to MXFP4 (E2M1 codes, E8M0 scale per 32) by the
packer's rule and both operands enter kind::mxf4 packed two codes to a byte;
the result must lie within the float32-accumulation bound 2^-12 sum
|q4(x)||w| + 1e-6 of the oracle's exact Q4(X) . W^T (plus the bf16 output's
half ulp), element by element.  The forms covered: single 128-row tiles at
both widths, tall 256-row tiles (two accumulators, two scale slots in tensor
memory refilled behind the MMAs), K splits over a cluster, ragged M and N,
float32 output, and an expired wait.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_scaled_quantized_spec_gb300 as q  # noqa: E402
from block_scaled_quantized_spec_gb300 import synth  # noqa: E402
from oracle import pack as opack  # noqa: E402
from oracle import reference as oref  # noqa: E402
from tolerance import check_tensor  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
FMT = "mxfp4"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_quantized_spec_gb300 import build
    build.build()
    q.load()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _case(m, n, k, seed):
    c, s, g = opack.pack(FMT, synth.weights(n, k, seed=seed))
    xb = synth.activations_bf16(m, k, seed=seed + 1)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    return c, s, g, xb, xt


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("m", [1, 17, 128, 300])
@pytest.mark.parametrize("n,k", [(272, 1024), (40, 256), (1000, 512)])
def test_qmm_a4_parity(out_dtype, m, n, k):
    c, s, g, xb, xt = _case(m, n, k, seed=m + n + k)
    out = q.qmm_a4(FMT, _dev(c), _dev(s), xt, n, out_dtype=out_dtype)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_a4_ref(FMT, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (m, n, k, str(out_dtype)))


@pytest.mark.parametrize("m,n,k", [(2048, 4096, 4096), (4096, 11008, 4096)])
def test_qmm_a4_full_size_every_output(m, n, k):
    c, s, g, xb, xt = _case(m, n, k, seed=21)
    out = q.qmm_a4(FMT, _dev(c), _dev(s), xt, n)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_a4_ref(FMT, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (m, n, k))
    # W . A4's own error against the exact bf16-activation product, relative to qmm's bound
    exact, qbound = oref.qmm_ref(FMT, c, s, g, xb, "bf16", m, n, k)
    o = out.float().cpu().numpy()
    print(f"{m}x{n}x{k}: W.A4 |out - exact| / qmm bound: max {float((np.abs(o - exact) / qbound).max()):.3f}, "
          f"median {float(np.median(np.abs(o - exact) / qbound)):.4f}")


@pytest.mark.parametrize("m,n,k", [(300, 5000, 512), (1000, 700, 1024), (129, 2300, 256), (777, 450, 2048)])
def test_qmm_a4_tall_tiles(m, n, k):
    # 256-row tiles forced on and off (debug key 9) without a K split (key 4):
    # the last tile's second M half wholly past M (m = 300), ending inside it
    # (1000, 777) or holding one row (129); K = 256 is one step and 2048 eight,
    # so the two tensor-memory scale slots wrap several times; against the
    # oracle, and bit for bit against single tiles (the same accumulation order)
    c, s, g, xb, xt = _case(m, n, k, seed=m + 5)
    dc, ds = _dev(c), _dev(s)
    ref, bound = oref.qmm_a4_ref(FMT, c, s, g, xb, "bf16", m, n, k)
    outs = []
    try:
        for tall in (2, 1):
            q.qfmt_debug_set(9, tall)
            q.qfmt_debug_set(4, 1)
            out = q.qmm_a4(FMT, dc, ds, xt, n)
            assert q.qfmt_device_status() == 0
            check_tensor(out, ref, bound, (m, n, k, tall))
            outs.append(out.float().cpu().numpy())
    finally:
        q.qfmt_debug_set(9, 0)
        q.qfmt_debug_set(4, 0)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("bn", [224, 256])
@pytest.mark.parametrize("splits", [1, 2, 3, 4])
def test_qmm_a4_tile_width_and_k_split(bn, splits):
    # single tiles at both widths, K split over a cluster of 1-4 CTAs (K =
    # 2304: 9 steps, uneven splits), ragged N
    m, n, k = 200, 600, 2304
    c, s, g, xb, xt = _case(m, n, k, seed=31)
    ref, bound = oref.qmm_a4_ref(FMT, c, s, g, xb, "bf16", m, n, k)
    try:
        q.qfmt_debug_set(9, 1)
        q.qfmt_debug_set(3, bn)
        q.qfmt_debug_set(4, splits)
        out = q.qmm_a4(FMT, _dev(c), _dev(s), xt, n)
        assert q.qfmt_device_status() == 0
    finally:
        for key in (3, 4, 9):
            q.qfmt_debug_set(key, 0)
    check_tensor(out, ref, bound, (bn, splits))


def test_qmm_a4_representable_activation_is_the_exact_product():
    # an activation that is already MXFP4 (E2M1 values times a power of two
    # per block, block maximum in (3, 6] times it): W . A4 is then qmm's exact
    # product, within the float32-accumulation bound
    m, n, k = 130, 300, 512
    rng = np.random.default_rng(41)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    x = np.empty((m, k), np.float32)
    for i in range(m):
        for b in range(0, k, 32):
            v = rng.choice(grid, 32) * rng.choice([-1.0, 1.0], 32)
            v[int(rng.integers(0, 32))] = 6.0
            x[i, b:b + 32] = (v * 2.0 ** int(rng.integers(-10, 10))).astype(np.float32)
    xb = synth.f32_to_bf16_bits(x)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    c, s, g = opack.pack(FMT, synth.weights(n, k, seed=42))
    out = q.qmm_a4(FMT, _dev(c), _dev(s), xt, n, out_dtype=torch.float32)
    exact, _ = oref.qmm_ref(FMT, c, s, g, xb, "bf16", m, n, k)
    _, bound = oref.qmm_a4_ref(FMT, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, exact, bound, "representable")


def test_qmm_a4_tall_expired_wait():
    # the W-scale warp never signals (test hook) in a tall-tile launch: the
    # bounded waits expire, the status word reports it, nothing is stored, and
    # the next call is correct
    m, n, k = 600, 2300, 1024
    c, s, g, xb, xt = _case(m, n, k, seed=51)
    dc, ds = _dev(c), _dev(s)
    assert q.qfmt_device_status() == 0
    sentinel = torch.full((m, n), 3.0, dtype=torch.bfloat16, device=DEV)
    q.qfmt_debug_set(9, 2)
    q.qfmt_debug_set(1, 20_000_000)
    q.qfmt_debug_set(2, 1)
    try:
        q.qmm_a4(FMT, dc, ds, xt, n, out=sentinel)
        st = q.qfmt_device_status()
    finally:
        q.qfmt_debug_set(2, 0)
        q.qfmt_debug_set(1, 0)
    try:
        assert st == -6
        assert (sentinel.float() == 3.0).all()
        out = q.qmm_a4(FMT, dc, ds, xt, n)
        assert q.qfmt_device_status() == 0
    finally:
        q.qfmt_debug_set(9, 0)
    ref, bound = oref.qmm_a4_ref(FMT, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, "after the expired wait")


def test_qmm_a4_workspace_and_errors():
    assert q.qmm_a4_workspace_bytes(FMT, 300, 1024) >= 300 * 512 + 384 * 1024 // 32
    assert q.qmm_a4_workspace_bytes("mxfp8_e4m3", 300, 1024) == 0
    assert q.qmm_a4_workspace_bytes(FMT, 300, 384) == 0
    c, s, g, xb, xt = _case(32, 64, 256, seed=61)
    small = torch.empty(q.qmm_a4_workspace_bytes(FMT, 32, 256) - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(q.QfmtError) as e:
        q.qmm_a4(FMT, _dev(c), _dev(s), xt, 64, workspace=small)
    assert e.value.status == -8
    c8, s8, _ = opack.pack("mxfp8_e4m3", synth.weights(64, 256, seed=1))
    with pytest.raises(q.QfmtError) as e:
        q.qmm_a4("mxfp8_e4m3", _dev(c8), _dev(s8), xt, 64)
    assert e.value.status == -4
    c3, s3, _ = opack.pack(FMT, synth.weights(64, 384, seed=2))
    x3 = _dev(synth.activations_bf16(32, 384, seed=3).view(np.int16)).view(torch.bfloat16)
    with pytest.raises(q.QfmtError) as e:
        q.qmm_a4(FMT, _dev(c3), _dev(s3), x3, 64)
    assert e.value.status == -2
    # M = 0 and N = 0 are no-ops
    assert q.qmm_a4(FMT, _dev(c), _dev(s), xt[:0], 64).shape == (0, 64)
