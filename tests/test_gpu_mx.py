"""GPU parity of the block-scaled tensor-core GEMM (path B) against the oracle.

With a workspace (``qmm_workspace_bytes``), ``qmm_ex`` runs mxfp4 / mxfp8 E4M3
/ E5M2 at M > 16 on tcgen05 kind::mxf8f6f4: X split into two MXFP8 E4M3 terms
(hi + lo, E8M0 per 32), the weights as stored, both scales applied by the
MMA.  The tolerance is qmm's (tests/tolerance.py): the split is exact for
every activation within 2^14 of its block's largest, so the seeded N(0, 1)
inputs land far inside the bound.
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


def _x(m, k, seed):
    xb = synth.activations_bf16(m, k, seed=seed)
    return xb, _dev(xb.view(np.int16)).view(torch.bfloat16)


def _qmm_b(fmt, dc, ds, g, xt, n, out=None):
    m, k = xt.shape
    wsb = q.qmm_workspace_bytes(fmt, m, k)
    assert wsb > 0
    ws = torch.empty(wsb, dtype=torch.uint8, device=DEV)
    return q.qmm_ex(fmt, dc, ds, g, xt, n, out=out, workspace=ws)


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("m", [17, 64, 128, 130, 256, 300])
@pytest.mark.parametrize("n,k", [(272, 1024), (300, 512), (256, 128), (40, 384)])
def test_block_scaled_gemm_parity(fmt, m, n, k):
    # tiles ragged in M and N, K of one to eight stages
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=m + n))
    xb, xt = _x(m, k, seed=m + k)
    out = _qmm_b(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, n, k))


FULL_B = [
    ("mxfp8_e4m3", 2048, 4096, 4096),     # the mxfp8 E4M3 prefill workload
    ("mxfp8_e5m2", 128, 11008, 4096),     # the sweep's mxfp8 E5M2 rows
    ("mxfp8_e5m2", 4096, 11008, 4096),
    ("mxfp4", 2048, 4096, 4096),
    ("mxfp4", 128, 4096, 4096),
]


@pytest.mark.parametrize("fmt,m,n,k", FULL_B)
def test_block_scaled_full_size_every_output(fmt, m, n, k):
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=0))
    xb, xt = _x(m, k, seed=1 + m)
    out = _qmm_b(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, n, k))


@pytest.mark.parametrize("fmt", MXB)
def test_paths_agree(fmt):
    # the same product through the bf16-decode GEMM (no workspace) and the
    # block-scaled GEMM: each within bound + half a bf16 ulp of the exact value
    m, n, k = 200, 520, 1024
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=3))
    xb, xt = _x(m, k, seed=4)
    dc, ds = _dev(c), _dev(s)
    a = q.qmm(fmt, dc, ds, g, xt, n).float().cpu().numpy()
    b = _qmm_b(fmt, dc, ds, g, xt, n).float().cpu().numpy()
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    assert (np.abs(a - b) <= 2 * bound + bf16_half_ulp(a) + bf16_half_ulp(b)).all()


@pytest.mark.parametrize("fmt", MXB)
def test_activation_extremes(fmt):
    # rows of very different magnitude, blocks holding values 2^-20 of their
    # largest, exact zeros and whole zero blocks: the two-term split and its
    # scale choice at the edges of the E4M3 range
    m, n, k = 130, 96, 512
    rng = np.random.default_rng(9)
    x = rng.standard_normal((m, k)).astype(np.float32)
    x *= np.exp2(rng.integers(-40, 40, size=(m, 1))).astype(np.float32)
    x[:, 5::32] *= np.float32(2.0 ** -20)
    x[:, 7::64] = 0.0
    x[3, 64:96] = 0.0
    x[4, :] = np.float32(2.0 ** -130)                 # subnormal in float32, a subnormal bf16
    xb = synth.f32_to_bf16_bits(x)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=10))
    out = _qmm_b(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, "extremes"))


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("m", [17, 130])
def test_block_scaled_special_scales_and_codes(fmt, m):
    # E8M0 0 (2^-127) scales give exact tiny weights; a 255 (NaN) scale and a
    # NaN / Inf element code make exactly their weight row's outputs non-finite
    n, k = 48, 256
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=31))
    rng = np.random.default_rng(32)
    s = s.copy()
    s[rng.random(s.shape) < 0.2] = 0
    s[3, :] = 0
    xb, xt = _x(m, k, seed=33)
    out = _qmm_b(fmt, _dev(c), _dev(s), g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, "zero scales"))
    s[5, 2] = 255
    c = c.copy()
    bad = [5]
    if fmt != "mxfp4":
        c[9, 40] = 0x7F if fmt == "mxfp8_e4m3" else 0x7C    # E4M3 NaN / E5M2 +inf
        bad.append(9)
    out = _qmm_b(fmt, _dev(c), _dev(s), g, xt, n).float().cpu().numpy()
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    assert (~np.isfinite(out[:, bad])).all()
    keep = np.ones(n, bool)
    keep[bad] = False
    check(out[:, keep], ref[:, keep], bound[:, keep], (fmt, m, "non-finite rows"))


def test_workspace_query_and_errors():
    # the workspace size: X's two code planes plus their scale atoms for the
    # MX formats the block-scaled MMA reads; 0 where the call needs none
    for fmt in MXB:
        assert q.qmm_workspace_bytes(fmt, 300, 1024) >= 2 * 300 * 1024 + 2 * 384 * 1024 // 32
        assert q.qmm_workspace_bytes(fmt, 16, 1024) == 0          # the decode GEMVs
        assert q.qmm_workspace_bytes(fmt, 300, 96) == 0           # K not a multiple of 128: bf16-decode GEMM
    for fmt in ("nvfp4", "int4_affine", "nvfp8", "mxint8"):
        assert q.qmm_workspace_bytes(fmt, 300, 1024) == 0
    m, n, k = 64, 128, 256
    c, s, g = opack.pack("mxfp8_e4m3", synth.weights(n, k, seed=1))
    xb, xt = _x(m, k, seed=2)
    small = torch.empty(q.qmm_workspace_bytes("mxfp8_e4m3", m, k) - 1, dtype=torch.uint8, device=DEV)
    with pytest.raises(q.QfmtError) as e:
        q.qmm_ex("mxfp8_e4m3", _dev(c), _dev(s), g, xt, n, workspace=small)
    assert e.value.status == -8


@pytest.mark.parametrize("m,n,k", [(256, 512, 1024), (2000, 2300, 256)])
def test_expired_wait_block_scaled(m, n, k):
    # the W-scale warp never signals (test hook): the MMA warp's bounded wait
    # expires, the status word reports it, no output is written, and the next
    # call is correct (a K-split cluster; 176 tiles of two K steps)
    fmt = "mxfp8_e4m3"
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=5))
    xb, xt = _x(m, k, seed=6)
    dc, ds = _dev(c), _dev(s)
    assert q.qfmt_device_status() == 0
    sentinel = torch.full((m, n), 3.0, dtype=torch.bfloat16, device=DEV)
    q.qfmt_debug_set(1, 20_000_000)
    q.qfmt_debug_set(2, 1)
    try:
        _qmm_b(fmt, dc, ds, g, xt, n, out=sentinel)
        st = q.qfmt_device_status()
    finally:
        q.qfmt_debug_set(2, 0)
        q.qfmt_debug_set(1, 0)
    assert st == -6
    assert (sentinel.float() == 3.0).all()
    out = _qmm_b(fmt, dc, ds, g, xt, n)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, "after the expired wait"))


@pytest.mark.parametrize("fmt", MXB)
def test_chained_layers_block_scaled(fmt):
    # square layers X(i+1) = out(i) back to back on one stream: the activation
    # split of each layer waits for the previous layer's output
    m, n = 256, 512
    layers = 5
    packed = [opack.pack(fmt, synth.weights(n, n, seed=70 + i)) for i in range(layers)]
    xb, xt = _x(m, n, seed=80)
    ws = torch.empty(q.qmm_workspace_bytes(fmt, m, n), dtype=torch.uint8, device=DEV)
    outs = [xt]
    for c, s, g in packed:
        outs.append(q.qmm_ex(fmt, _dev(c), _dev(s), g, outs[-1], n, workspace=ws))
    torch.cuda.synchronize()
    for i, (c, s, g) in enumerate(packed):
        xin = outs[i].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        ref, bound = oref.qmm_ref(fmt, c, s, g, xin, "bf16", m, n, n)
        check_tensor(outs[i + 1], ref, bound, (fmt, "layer", i))


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("m", [1, 2, 8, 9, 16])
@pytest.mark.parametrize("k", [128, 384, 512, 768, 1024])
def test_tensor_core_decode_gemv(fmt, m, k):
    # M <= 16 with K <= 1024: the decode GEMV on the block-scaled MMA (weights
    # as stored, activations split in the CTA, one CTA per 128 rows or a pair
    # summed through distributed shared memory); N ends inside a 128-row tile
    n = 300
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=m + k))
    xb, xt = _x(m, k, seed=m * k)
    dc, ds = _dev(c), _dev(s)
    out = q.qmm(fmt, dc, ds, g, xt, n)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, k))
    # the same rows through the mma.sync decode GEMV (measurement hook 5)
    q.qfmt_debug_set(5, 1)
    try:
        other = q.qmm(fmt, dc, ds, g, xt, n).float().cpu().numpy()
    finally:
        q.qfmt_debug_set(5, 0)
    a = out.float().cpu().numpy()
    assert (np.abs(a - other) <= 2 * bound + bf16_half_ulp(a) + bf16_half_ulp(other)).all()


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("m,n,k", [(3, 4096, 4096), (9, 4000, 4096), (16, 4096, 3072)])
def test_tensor_core_decode_gemv_long_k(fmt, m, n, k):
    # 3-16 activation rows at long K: the tensor-core decode GEMV split into
    # 512-column slabs (8 and 6 CTAs a cluster) where that grid lands 1.5-2
    # CTAs on every SM (N = 4000 ends inside a tile); against the oracle at
    # every output and against the CUDA-core batch GEMV (hook 5)
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=m + 11))
    xb, xt = _x(m, k, seed=m + 12)
    dc, ds = _dev(c), _dev(s)
    out = q.qmm(fmt, dc, ds, g, xt, n)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out, ref, bound, (fmt, m, n, k))
    q.qfmt_debug_set(5, 1)
    try:
        other = q.qmm(fmt, dc, ds, g, xt, n).float().cpu().numpy()
    finally:
        q.qfmt_debug_set(5, 0)
    a = out.float().cpu().numpy()
    assert (np.abs(a - other) <= 2 * bound + bf16_half_ulp(a) + bf16_half_ulp(other)).all()


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("m,n,k", [(130, 300, 128), (300, 520, 384), (2000, 2300, 640), (1200, 4100, 1152)])
def test_stage_ring_wraps(fmt, m, n, k):
    # three stages: 1, 3, 5 and 9 K steps leave the stage ring at every
    # offset; the planner's tiles and forced tile widths and K splits (debug
    # keys 3, 4) all agree with the oracle, and the quantized-activation
    # product runs the same ring
    c, s, g = opack.pack(fmt, synth.weights(n, k, seed=m + 1))
    xb, xt = _x(m, k, seed=m + 2)
    dc, ds = _dev(c), _dev(s)
    ws = torch.empty(q.qmm_workspace_bytes(fmt, m, k), dtype=torch.uint8, device=DEV)
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    try:
        for bn, sk in ((0, 0), (224, 1), (256, 2), (256, 3)):
            q.qfmt_debug_set(3, bn)
            q.qfmt_debug_set(4, sk)
            out = q.qmm_ex(fmt, dc, ds, g, xt, n, workspace=ws)
            assert q.qfmt_device_status() == 0
            check_tensor(out, ref, bound, (fmt, m, n, k, bn, sk))
    finally:
        q.qfmt_debug_set(3, 0)
        q.qfmt_debug_set(4, 0)
    out8 = q.qmm_a8(fmt, dc, ds, xt, n)
    assert q.qfmt_device_status() == 0
    ref8, bound8 = oref.qmm_a8_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check_tensor(out8, ref8, bound8, (fmt, "a8", m, n, k))
