"""GPU parity of the quantized-activation path against the oracle.

* qfmt_quantize: an activation packed on the GPU as a weight of mxfp4 /
  mxfp8 E4M3 / E5M2 -- bit-exact against the oracle's packer applied to the
  same values (codes and scales, byte for byte).
* qmm_a8: both operands quantized (the activation to MXFP8 E4M3 by that
  rule), one block-scaled MMA per block -- within the float32-accumulation
  bound 2^-12 sum |q(x)||w| + 1e-6 of the oracle's exact Q(X) . W^T (plus the
  bf16 output's half ulp).  Its distance from the exact bf16-activation
  product is reported, not bounded: it is W . A8's own quantization error.
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
MXB = ["mxfp4", "mxfp8_e4m3", "mxfp8_e5m2"]
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


def _activations(m, k, seed):
    # N(0, 1) rows at magnitudes across the float32 range, zero blocks, single
    # tiny values, exact ties between adjacent codes, subnormal float32 values
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((m, k)).astype(np.float32)
    x *= np.exp2(rng.integers(-60, 60, size=(m, 1))).astype(np.float32)
    x[0, :32] = 0.0
    if m > 1 and k > 32:
        x[1, 32:64] *= np.float32(1e-30)
    if m > 2 and k > 64:
        x[2, 64:96] = np.float32(2.0 ** -140)
    if m > 3:
        x[3, :32] = np.float32(448.0) * np.arange(32, dtype=np.float32) / np.float32(16.0)   # midpoints of the grid
    return x


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("x_dtype", ["bf16", "f32"])
@pytest.mark.parametrize("m,k", [(1, 32), (5, 96), (64, 1024), (130, 4096)])
def test_quantize_bit_exact(fmt, x_dtype, m, k):
    x = _activations(m, k, seed=m + k)
    if x_dtype == "bf16":
        xb = synth.f32_to_bf16_bits(x)
        xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
        xin = xb
    else:
        xt = _dev(x)
        xin = x
    codes, scales = q.qfmt_quantize(fmt, xt)
    want_c, want_s = oref.quantize_activations(fmt, xin, x_dtype, m, k)
    got_c, got_s = codes.cpu().numpy().reshape(want_c.shape), scales.cpu().numpy().reshape(want_s.shape)
    assert np.array_equal(got_s, want_s), (fmt, np.argwhere(got_s != want_s)[:5].tolist())
    assert np.array_equal(got_c, want_c), (fmt, np.argwhere(got_c != want_c)[:5].tolist())


def test_quantize_of_a_weight_equals_the_host_packer():
    # the same matrix packed by the host packer (as a weight) and quantized on
    # the GPU (as an activation): the same bytes
    w = synth.weights(96, 512, seed=9)
    for fmt in MXB:
        c, s, _ = q.qfmt_pack(fmt, w)
        gc, gs = q.qfmt_quantize(fmt, _dev(w))
        assert np.array_equal(gc.cpu().numpy().reshape(c.shape), c), fmt
        assert np.array_equal(gs.cpu().numpy().reshape(s.shape), s), fmt


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("m", [1, 17, 128, 300])
@pytest.mark.parametrize("n,k", [(272, 1024), (40, 128)])
def test_qmm_a8_parity(fmt, m, n, k):
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=m + n))
    xb = synth.activations_bf16(m, k, seed=m + k)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    out = q.qmm_a8(fmt, _dev(c), _dev(s), xt, n)
    ref, bound = oref.qmm_a8_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, n, k))


@pytest.mark.parametrize("fmt,m,n,k", [("mxfp8_e4m3", 2048, 4096, 4096), ("mxfp4", 2048, 4096, 4096),
                                       ("mxfp8_e5m2", 4096, 11008, 4096)])
def test_qmm_a8_full_size_every_output(fmt, m, n, k):
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=0))
    xb = synth.activations_bf16(m, k, seed=1 + m)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    out = q.qmm_a8(fmt, _dev(c), _dev(s), xt, n)
    ref, bound = oref.qmm_a8_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, n, k))
    # W . A8's own error against the exact bf16-activation product, relative to qmm's bound
    exact, qbound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    o = out.float().cpu().numpy()
    print(f"{fmt} {m}x{n}x{k}: W.A8 |out - exact| / qmm bound: max {float((np.abs(o - exact) / qbound).max()):.3f}, "
          f"median {float(np.median(np.abs(o - exact) / qbound)):.4f}")


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("m,n,k", [(300, 5000, 512), (1000, 700, 1024), (129, 2300, 256)])
def test_qmm_a8_tall_tiles(fmt, m, n, k):
    # 256-row tiles (two 128-row accumulators sharing each stage's W tile),
    # forced on and off (debug key 9): the last tile's second M half lies
    # wholly past M (m = 300), ends inside it (m = 1000) or holds one row
    # (m = 129); against the oracle, and bit for bit against single tiles (the
    # same accumulation order)
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=m + 3))
    xb = synth.activations_bf16(m, k, seed=m + 4)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    dc, ds = _dev(c), _dev(s)
    ref, bound = oref.qmm_a8_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    outs = []
    try:
        for tall in (2, 1):
            q.qfmt_debug_set(9, tall)
            q.qfmt_debug_set(4, 1)   # no K split: the tall form's condition
            out = q.qmm_a8(fmt, dc, ds, xt, n)
            assert q.qfmt_device_status() == 0
            check_tensor(out, ref, bound, (fmt, m, n, k, tall))
            outs.append(out.float().cpu().numpy())
    finally:
        q.qfmt_debug_set(9, 0)
        q.qfmt_debug_set(4, 0)
    assert np.array_equal(outs[0], outs[1])


def test_qmm_a8_tall_expired_wait():
    # the W-scale warp never signals (test hook) in a tall-tile launch: the
    # bounded waits expire, the status word reports it, nothing is stored, and
    # the next call is correct
    fmt, m, n, k = "mxfp8_e4m3", 600, 2300, 512
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=8))
    xb = synth.activations_bf16(m, k, seed=9)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    dc, ds = _dev(c), _dev(s)
    assert q.qfmt_device_status() == 0
    sentinel = torch.full((m, n), 3.0, dtype=torch.bfloat16, device=DEV)
    q.qfmt_debug_set(9, 2)
    q.qfmt_debug_set(1, 20_000_000)
    q.qfmt_debug_set(2, 1)
    try:
        q.qmm_a8(fmt, dc, ds, xt, n, out=sentinel)
        st = q.qfmt_device_status()
    finally:
        q.qfmt_debug_set(2, 0)
        q.qfmt_debug_set(1, 0)
    try:
        assert st == -6
        assert (sentinel.float() == 3.0).all()
        out = q.qmm_a8(fmt, dc, ds, xt, n)
        assert q.qfmt_device_status() == 0
    finally:
        q.qfmt_debug_set(9, 0)
    ref, bound = oref.qmm_a8_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, "after the expired wait"))


def test_qmm_a8_workspace_and_errors():
    assert q.qmm_a8_workspace_bytes("mxfp8_e4m3", 300, 1024) >= 300 * 1024 + 384 * 1024 // 32
    assert q.qmm_a8_workspace_bytes("nvfp4", 300, 1024) == 0
    assert q.qmm_a8_workspace_bytes("mxfp4", 300, 96) == 0
    c, s, g = opack.pack("mxfp8_e4m3", synth.weights(64, 256, seed=1))
    xt = _dev(synth.activations_bf16(32, 256, seed=2).view(np.int16)).view(torch.bfloat16)
    small = torch.empty(q.qmm_a8_workspace_bytes("mxfp8_e4m3", 32, 256) - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(q.QfmtError) as e:
        q.qmm_a8("mxfp8_e4m3", _dev(c), _dev(s), xt, 64, workspace=small)
    assert e.value.status == -8
    cn, sn, gn = opack.pack("nvfp4", synth.weights(64, 256, seed=1))
    with pytest.raises(q.QfmtError) as e:
        q.qmm_a8("nvfp4", _dev(cn), _dev(sn), xt, 64)
    assert e.value.status == -4
