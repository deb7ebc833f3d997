"""GPU parity of the all-FP4 product (qmm_a4) against the oracle.

The activation is packed in the weight's FP4 family by the packer's rule
(MXFP4 against mxfp4 weights; NVFP4 with its own global against nvfp4) and
both operands enter the tensor cores packed two codes to a byte (kind::mxf4,
kind::mxf4nvf4); the result must lie within the float32-accumulation bound
2^-12 sum |q4(x)||w| + 1e-6 of the oracle's exact Q4(X) . W^T (plus the bf16
output's half ulp), element by element.  The forms covered: single 128-row
tiles at both widths, tall 256-row tiles (two accumulators; two scale slots
in tensor memory for mxfp4, one for nvfp4, refilled behind the MMAs), K splits over a cluster,
ragged M and N, float32 output, an expired wait; and the quantized
activation the call leaves in its workspace, byte for byte against the
oracle's packer.
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
FP4 = ["mxfp4", "nvfp4"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_quantized_spec_gb300 import build
    build.build()
    q.load()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _case(fmt, m, n, k, seed):
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=seed, outliers=(fmt == "nvfp4")))
    xb = synth.activations_bf16(m, k, seed=seed + 1)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    return c, s, g, xb, xt


@pytest.mark.parametrize("fmt", FP4)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("m", [1, 17, 128, 300])
@pytest.mark.parametrize("n,k", [(272, 1024), (40, 256), (1000, 512)])
def test_qmm_a4_parity(fmt, out_dtype, m, n, k):
    c, s, g, xb, xt = _case(fmt, m, n, k, seed=m + n + k)
    out = q.qmm_a4(fmt, _dev(c), _dev(s), g, xt, n, out_dtype=out_dtype)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_a4_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, n, k, str(out_dtype)))


@pytest.mark.parametrize("fmt", FP4)
@pytest.mark.parametrize("m,n,k", [(2048, 4096, 4096), (4096, 11008, 4096)])
def test_qmm_a4_full_size_every_output(fmt, m, n, k):
    c, s, g, xb, xt = _case(fmt, m, n, k, seed=21)
    out = q.qmm_a4(fmt, _dev(c), _dev(s), g, xt, n)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_a4_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, n, k))
    # W . A4's own error against the exact bf16-activation product, relative to qmm's bound
    exact, qbound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    o = out.float().cpu().numpy()
    print(f"{fmt} {m}x{n}x{k}: W.A4 |out - exact| / qmm bound: max {float((np.abs(o - exact) / qbound).max()):.3f}, "
          f"median {float(np.median(np.abs(o - exact) / qbound)):.4f}")


def _ws_activation(fmt, ws, m, k):
    """Q4(X) as the call leaves it in the workspace: codes [M, K/2], scales [M, K/blk], global."""
    w = ws.cpu().numpy()
    codes = w[: m * k // 2].reshape(m, k // 2)
    al = lambda v: (v + 1023) // 1024 * 1024  # noqa: E731
    base = al(m * k // 2)
    cell_k = 64 if fmt == "nvfp4" else 128                 # K covered by one 4-byte scale cell
    blk = cell_k // 4
    katoms = k // cell_k
    scales = np.empty((m, k // blk), np.uint8)
    for r in range(m):
        for b in range(k // blk):
            atom = (r // 128) * katoms + b // 4
            off = 16 * (r % 32) + 4 * ((r % 128) // 32) + b % 4
            scales[r, b] = w[base + atom * 512 + off]
    g = np.float32(1.0)
    if fmt == "nvfp4":
        gofs = base + al(((m + 127) // 128) * katoms * 512) + 4096
        g = w[gofs:gofs + 4].view(np.float32)[0]
    return codes, scales, g


@pytest.mark.parametrize("fmt", FP4)
@pytest.mark.parametrize("m,k", [(5, 256), (130, 512), (300, 1024)])
def test_qmm_a4_quantized_activation_bit_exact(fmt, m, k):
    # the workspace after the call holds Q4(X): codes, scales (and the nvfp4
    # global) byte for byte the oracle packer's, with activations across
    # magnitudes, zero blocks and exact ties
    rng = np.random.default_rng(m + k)
    x = rng.standard_normal((m, k)).astype(np.float32)
    x *= np.exp2(rng.integers(-8, 8, size=(m, 1))).astype(np.float32)
    x[0, :32] = 0.0
    x[1, 16:48] = np.array([6.0, 0.25, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25] * 4, np.float32)
    xb = synth.f32_to_bf16_bits(x)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    n = 64
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=3))
    ws = torch.zeros(q.qmm_a4_workspace_bytes(fmt, m, k), dtype=torch.uint8, device=DEV)
    q.qmm_a4(fmt, _dev(c), _dev(s), g, xt, n, workspace=ws)
    torch.cuda.synchronize()
    got_c, got_s, got_g = _ws_activation(fmt, ws, m, k)
    want_c, want_s, want_g = oref.quantize_activations_global(fmt, xb, "bf16", m, k)
    assert np.float32(got_g) == np.float32(want_g), (got_g, want_g)
    assert np.array_equal(got_s, want_s), (fmt, np.argwhere(got_s != want_s)[:5].tolist())
    assert np.array_equal(got_c, want_c), (fmt, np.argwhere(got_c != want_c)[:5].tolist())


@pytest.mark.parametrize("fmt", FP4)
@pytest.mark.parametrize("m,n,k", [(300, 5000, 512), (1000, 700, 1024), (129, 2300, 256), (777, 450, 2048)])
def test_qmm_a4_tall_tiles(fmt, m, n, k):
    # 256-row tiles forced on and off (debug key 9) without a K split (key
    # 4): the last tile's second M half wholly past M (m = 300), ending inside
    # it (1000, 777) or holding one row (129); K = 256 is one step and 2048
    # eight, so the tensor-memory scale slots (two for mxfp4, one for nvfp4)
    # are refilled several times; against the oracle, and bit for bit against
    # single tiles (the same accumulation order)
    c, s, g, xb, xt = _case(fmt, m, n, k, seed=m + 5)
    dc, ds = _dev(c), _dev(s)
    ref, bound = oref.qmm_a4_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    outs = []
    try:
        for tall in (2, 1):
            q.qfmt_debug_set(9, tall)
            q.qfmt_debug_set(4, 1)
            out = q.qmm_a4(fmt, dc, ds, g, xt, n)
            assert q.qfmt_device_status() == 0
            check_tensor(out, ref, bound, (m, n, k, tall))
            outs.append(out.float().cpu().numpy())
    finally:
        q.qfmt_debug_set(9, 0)
        q.qfmt_debug_set(4, 0)
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("fmt", FP4)
@pytest.mark.parametrize("bn", [224, 256])
@pytest.mark.parametrize("splits", [1, 2, 3, 4])
def test_qmm_a4_tile_width_and_k_split(fmt, bn, splits):
    # single tiles at both widths, K split over a cluster of 1-4 CTAs (K =
    # 2304: 9 steps, uneven splits), ragged N
    m, n, k = 200, 600, 2304
    c, s, g, xb, xt = _case(fmt, m, n, k, seed=31)
    ref, bound = oref.qmm_a4_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    try:
        q.qfmt_debug_set(9, 1)
        q.qfmt_debug_set(3, bn)
        q.qfmt_debug_set(4, splits)
        out = q.qmm_a4(fmt, _dev(c), _dev(s), g, xt, n)
        assert q.qfmt_device_status() == 0
    finally:
        for key in (3, 4, 9):
            q.qfmt_debug_set(key, 0)
    check_tensor(out, ref, bound, (fmt, bn, splits))


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
    c, s, g = opack.pack("mxfp4", synth.weights(n, k, seed=42))
    out = q.qmm_a4("mxfp4", _dev(c), _dev(s), g, xt, n, out_dtype=torch.float32)
    exact, _ = oref.qmm_ref("mxfp4", c, s, g, xb, "bf16", m, n, k)
    _, bound = oref.qmm_a4_ref("mxfp4", c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, exact, bound, "representable")


@pytest.mark.parametrize("fmt", FP4)
def test_qmm_a4_expired_wait(fmt):
    # the W-scale warp never signals (test hook; mxfp4 on tall tiles, nvfp4 on
    # single ones): the bounded waits expire, the status word reports it,
    # nothing is stored, and the next call is correct
    m, n, k = 600, 2300, 1024
    c, s, g, xb, xt = _case(fmt, m, n, k, seed=51)
    dc, ds = _dev(c), _dev(s)
    assert q.qfmt_device_status() == 0
    sentinel = torch.full((m, n), 3.0, dtype=torch.bfloat16, device=DEV)
    q.qfmt_debug_set(9, 2)
    q.qfmt_debug_set(1, 20_000_000)
    q.qfmt_debug_set(2, 1)
    try:
        q.qmm_a4(fmt, dc, ds, g, xt, n, out=sentinel)
        st = q.qfmt_device_status()
    finally:
        q.qfmt_debug_set(2, 0)
        q.qfmt_debug_set(1, 0)
    try:
        assert st == -6
        assert (sentinel.float() == 3.0).all()
        out = q.qmm_a4(fmt, dc, ds, g, xt, n)
        assert q.qfmt_device_status() == 0
    finally:
        q.qfmt_debug_set(9, 0)
    ref, bound = oref.qmm_a4_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, "after the expired wait"))


def test_qmm_a4_nvfp4_non_finite_activation_gives_nan():
    # an infinity in X: the activation's global is NaN, hence every output
    m, n, k = 40, 64, 256
    c, s, g, xb, xt = _case("nvfp4", m, n, k, seed=61)
    xt = xt.clone()
    xt[3, 7] = float("inf")
    out = q.qmm_a4("nvfp4", _dev(c), _dev(s), g, xt, n, out_dtype=torch.float32)
    assert q.qfmt_device_status() == 0
    assert torch.isnan(out).all()


def test_qmm_a4_workspace_and_errors():
    assert q.qmm_a4_workspace_bytes("mxfp4", 300, 1024) >= 300 * 512 + 384 * 1024 // 32
    assert q.qmm_a4_workspace_bytes("nvfp4", 300, 1024) >= 300 * 512 + 384 * 1024 // 16 + 4100
    assert q.qmm_a4_workspace_bytes("mxfp8_e4m3", 300, 1024) == 0
    assert q.qmm_a4_workspace_bytes("mxfp4", 300, 384) == 0
    c, s, g, xb, xt = _case("mxfp4", 32, 64, 256, seed=61)
    small = torch.empty(q.qmm_a4_workspace_bytes("mxfp4", 32, 256) - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(q.QfmtError) as e:
        q.qmm_a4("mxfp4", _dev(c), _dev(s), g, xt, 64, workspace=small)
    assert e.value.status == -8
    c8, s8, _ = opack.pack("mxfp8_e4m3", synth.weights(64, 256, seed=1))
    with pytest.raises(q.QfmtError) as e:
        q.qmm_a4("mxfp8_e4m3", _dev(c8), _dev(s8), 1.0, xt, 64)
    assert e.value.status == -4
    c3, s3, _ = opack.pack("mxfp4", synth.weights(64, 384, seed=2))
    x3 = _dev(synth.activations_bf16(32, 384, seed=3).view(np.int16)).view(torch.bfloat16)
    with pytest.raises(q.QfmtError) as e:
        q.qmm_a4("mxfp4", _dev(c3), _dev(s3), 1.0, x3, 64)
    assert e.value.status == -2
    # M = 0 is a no-op
    assert q.qmm_a4("mxfp4", _dev(c), _dev(s), g, xt[:0], 64).shape == (0, 64)
