"""GPU parity of the fused decode forms against the oracle.

* qmm_batched: up to four weight matrices sharing one activation (the
  batched Q/K/V and 4-way projections of metaltile PR #250), one launch for
  M <= 2 and one qmm per matrix beyond;
* qmm_rmsnorm: RMSNorm of the activation fused in front of the decode GEMV
  (PR #250, the fused RMSNorm + GEMV commit);
* qmm_gated_rmsnorm: the same times silu(gate) (the fused gated-RMSNorm +
  GEMV commit).
Tolerance as qmm (plus half a bf16 ulp of each stored output; tests/tolerance.py); inputs packed by the
oracle's packer from seeded generators.
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
FMTS = [f for f in q.FORMATS if f not in q.SUB_BYTE]   # the 2/3/5/6-bit formats take qmm only
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


def _x(m, k, seed):
    xb = synth.activations_bf16(m, k, seed=seed)
    return xb, _dev(xb.view(np.int16)).view(torch.bfloat16)


def _check(out_t, ref, bound, what):
    return check_tensor(out_t, ref, bound, what)


def _gamma(k, seed):
    g = 1.0 + 0.25 * np.random.default_rng(seed).standard_normal(k)
    gt = torch.from_numpy(g.astype(np.float32)).to(torch.bfloat16)
    return gt.view(torch.int16).numpy().view(np.uint16), gt.to(DEV)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 2, 5])
def test_batched_qkv_parity(fmt, m):
    # grouped-query shapes: Q wide, K and V narrow (ragged tiles), K = 1024
    k, ns = 1024, (200, 40, 40)
    mats, dev = [], []
    for i, n in enumerate(ns):
        w = synth.weights(n, k, seed=60 + i, outliers=(fmt == "nvfp4"))
        c, s, g = opack.pack(fmt, w)
        mats.append((c, s, g, n))
        dev.append((_dev(c), _dev(s), g))
    xb, xt = _x(m, k, seed=63 + m)
    outs = q.qmm_batched(fmt, [d[0] for d in dev], [d[1] for d in dev], [d[2] for d in dev], xt, list(ns))
    for o, (ref, bound), n in zip(outs, oref.qmm_batched_ref(fmt, mats, xb, "bf16", m, k), ns):
        assert o.shape == (m, n)
        _check(o, ref, bound, (fmt, m, n))


def test_batched_four_way_equals_separate_calls():
    fmt, m, k = "mxfp4", 1, 4096
    ns = (4096, 1024, 1024, 512)
    dev = []
    for i, n in enumerate(ns):
        c, s, g = opack.pack(fmt, synth.weights(n, k, seed=70 + i))
        dev.append((_dev(c), _dev(s), g))
    _, xt = _x(m, k, seed=74)
    outs = q.qmm_batched(fmt, [d[0] for d in dev], [d[1] for d in dev], [d[2] for d in dev], xt, list(ns))
    for o, (c, s, g), n in zip(outs, dev, ns):
        assert torch.equal(o, q.qmm(fmt, c, s, g, xt, n))    # the same single-matrix decode GEMV


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 2])
def test_rmsnorm_parity(fmt, m):
    n, k, eps = 200, 1024, 1e-5
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=80, outliers=(fmt == "nvfp4")))
    xb, xt = _x(m, k, seed=81 + m)
    gb, gt = _gamma(k, 83)
    out = q.qmm_rmsnorm(fmt, _dev(c), _dev(s), g, xt, gt, eps, n)
    ref, bound = oref.qmm_rmsnorm_ref(fmt, c, s, g, xb, "bf16", gb, eps, m, n, k)
    _check(out, ref, bound, (fmt, m))


def test_rmsnorm_full_width_and_large_activations():
    # N = K = 4096, activations scaled by 2^40 (normalisation removes the scale)
    fmt, m, n, k, eps = "nvfp4", 2, 4096, 4096, 1e-6
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=84, outliers=True))
    xb = synth.activations_bf16(m, k, seed=85)
    zero = (xb & 0x7F80) == 0
    xb = ((xb.astype(np.uint32) + (40 << 7)) & 0xFFFF).astype(np.uint16)
    xb[zero] = 0
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    gb, gt = _gamma(k, 86)
    out = q.qmm_rmsnorm(fmt, _dev(c), _dev(s), g, xt, gt, eps, n)
    ref, bound = oref.qmm_rmsnorm_ref(fmt, c, s, g, xb, "bf16", gb, eps, m, n, k)
    _check(out, ref, bound, fmt)


def test_rmsnorm_rejects_batches_above_two():
    fmt, n, k = "mxfp4", 32, 256
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=87))
    _, xt = _x(3, k, seed=88)
    _, gt = _gamma(k, 89)
    with pytest.raises(q.QfmtError) as e:
        q.qmm_rmsnorm(fmt, _dev(c), _dev(s), g, xt, gt, 1e-5, n)
    assert e.value.status == -4


# ---- the gated RMSNorm (PR #250, the fused gated-RMSNorm + GEMV commit) ----

@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 2])
def test_gated_rmsnorm_parity(fmt, m):
    n, k, eps = 200, 1024, 1e-5
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=90, outliers=(fmt == "nvfp4")))
    xb, xt = _x(m, k, seed=91 + m)
    zb, zt = _x(m, k, seed=93 + m)
    gb, gt = _gamma(k, 95)
    out = q.qmm_gated_rmsnorm(fmt, _dev(c), _dev(s), g, xt, zt, gt, eps, n)
    ref, bound = oref.qmm_gated_rmsnorm_ref(fmt, c, s, g, xb, zb, "bf16", gb, eps, m, n, k)
    _check(out, ref, bound, (fmt, m))


def test_gated_rmsnorm_extreme_gates_and_full_width():
    # N = K = 4096; gates far negative (silu -> -0), zero, and large (silu -> z)
    fmt, m, n, k, eps = "mxfp4", 2, 4096, 4096, 1e-6
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=96))
    xb, xt = _x(m, k, seed=97)
    z = np.random.default_rng(98).standard_normal((m, k)).astype(np.float32) * 4
    z[:, ::7] = -300.0
    z[:, 1::7] = 0.0
    z[:, 2::7] = 300.0
    zb = synth.f32_to_bf16_bits(z)
    zt = _dev(zb.view(np.int16)).view(torch.bfloat16)
    gb, gt = _gamma(k, 99)
    out = q.qmm_gated_rmsnorm(fmt, _dev(c), _dev(s), g, xt, zt, gt, eps, n)
    ref, bound = oref.qmm_gated_rmsnorm_ref(fmt, c, s, g, xb, zb, "bf16", gb, eps, m, n, k)
    _check(out, ref, bound, fmt)


def test_gated_rmsnorm_with_a_zero_gate_is_zero_and_a_large_gate_scales_rmsnorm():
    fmt, m, n, k, eps = "nvfp8", 1, 256, 512, 1e-5
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=100))
    xb, xt = _x(m, k, seed=101)
    gb, gt = _gamma(k, 102)
    zero = torch.zeros((m, k), dtype=torch.bfloat16, device=DEV)
    assert not q.qmm_gated_rmsnorm(fmt, _dev(c), _dev(s), g, xt, zero, gt, eps, n).float().any()
    big = torch.full((m, k), 64.0, dtype=torch.bfloat16, device=DEV)   # silu(64) = 64 in float32
    a = q.qmm_gated_rmsnorm(fmt, _dev(c), _dev(s), g, xt, big, gt, eps, n).float()
    b = q.qmm_rmsnorm(fmt, _dev(c), _dev(s), g, xt, gt, eps, n).float()
    ref, bound = oref.qmm_rmsnorm_ref(fmt, c, s, g, xb, "bf16", gb, eps, m, n, k)
    _check(a / 64.0, ref, bound, "gate 64")
    _check(b, ref, bound, "plain")


@pytest.mark.parametrize("fmt", ["int3", "mxint5", "int6_f16"])
def test_sub_byte_formats_are_refused_by_the_fused_forms(fmt):
    m, n, k = 1, 64, 256
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=1))
    xb, xt = _x(m, k, seed=2)
    gamma = torch.ones(k, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(q.QfmtError) as e:
        q.qmm_rmsnorm(fmt, _dev(c), _dev(s), g, xt, gamma, 1e-5, n)
    assert e.value.status == -4
    with pytest.raises(q.QfmtError) as e:
        q.qmm_batched(fmt, [_dev(c)], [_dev(s)], [g], xt, [n])
    assert e.value.status == -4
