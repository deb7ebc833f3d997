"""GPU parity of the expert-routed product (MoE gather-qmm) against the oracle.

Row m of the output is x[m] against rows [e N, e N + N) of one stacked
[E * N, K] packed weight, e = expert_idx[m] (metaltile PR #250, the MoE
gather-qmm commit).  Tolerance as qmm: |out - ref| <= 2e-3 sum_k |x||w| + 1e-6
plus half an ulp of the bf16 output.  Inputs: weights packed by the oracle's
packer, activations and expert numbers from seeded generators.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_scaled_quantized_spec_gb300 as q  # noqa: E402
from block_scaled_quantized_spec_gb300 import synth  # noqa: E402
from oracle import pack as opack  # noqa: E402
from oracle import reference as oref  # noqa: E402
from tolerance import bf16_half_ulp, check_tensor  # noqa: E402

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


def _case(fmt, m, n, k, e, seed):
    w = synth.weights(e * n, k, seed=seed, outliers=(fmt == "nvfp4"))
    c, s, g = opack.pack(fmt, w)
    xb = synth.activations_bf16(m, k, seed=seed + 1)
    xt = _dev(xb.view(np.int16)).view(torch.bfloat16)
    idx = np.random.default_rng(seed + 2).integers(0, e, size=m).astype(np.int32)
    return c, s, g, xb, xt, idx


def _check(out_t, ref, bound, what):
    return check_tensor(out_t, ref, bound, what)


def _x(m, k, seed):
    xb = synth.activations_bf16(m, k, seed=seed)
    return xb, _dev(xb.view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("m", [1, 5, 9])
def test_gather_parity(fmt, m):
    n, k, e = 200, 1024, 3                 # ragged row tiles, several chunks per warp
    c, s, g, xb, xt, idx = _case(fmt, m, n, k, e, seed=30 + m)
    idx[0] = e - 1                         # the last slab is reached
    out = q.qmm_gather(fmt, _dev(c), _dev(s), g, xt, _dev(idx), n, e)
    ref, bound = oref.qmm_gather_ref(fmt, c, s, g, xb, "bf16", idx, m, n, k, e)
    _check(out, ref, bound, (fmt, m))
    assert q.qfmt_device_status() == 0


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4", "int4_affine", "mxfp8_e5m2"])
def test_gather_wider_shape_and_repeated_experts(fmt):
    # eight rows over four experts (each twice), N = 1024, K = 2048
    m, n, k, e = 8, 1024, 2048, 4
    c, s, g, xb, xt, idx = _case(fmt, m, n, k, e, seed=40)
    idx[:] = [3, 1, 0, 2, 1, 3, 0, 2]
    out = q.qmm_gather(fmt, _dev(c), _dev(s), g, xt, _dev(idx), n, e)
    ref, bound = oref.qmm_gather_ref(fmt, c, s, g, xb, "bf16", idx, m, n, k, e)
    _check(out, ref, bound, fmt)


def test_gather_one_expert_equals_qmm():
    fmt, m, n, k = "nvfp8", 4, 96, 512
    c, s, g, xb, xt, _ = _case(fmt, m, n, k, 1, seed=41)
    idx = _dev(np.zeros(m, np.int32))
    a = q.qmm_gather(fmt, _dev(c), _dev(s), g, xt, idx, n, 1)
    b = torch.cat([q.qmm(fmt, _dev(c), _dev(s), g, xt[i:i + 1], n) for i in range(m)])
    assert torch.equal(a, b)               # the same single-row GEMV on the same weights


def test_gather_out_of_range_index_zeroes_the_row():
    fmt, m, n, k, e = "mxfp8_e4m3", 4, 64, 256, 2
    c, s, g, xb, xt, idx = _case(fmt, m, n, k, e, seed=42)
    bad = idx.copy()
    bad[1], bad[3] = 2, -1
    q.qfmt_device_status()                 # start clean
    out = q.qmm_gather(fmt, _dev(c), _dev(s), g, xt, _dev(bad), n, e)
    assert q.qfmt_device_status() == -9    # QFMT_EINDEX, then cleared
    assert q.qfmt_device_status() == 0
    o = out.float().cpu().numpy()
    assert (o[1] == 0).all() and (o[3] == 0).all()
    good = [0, 2]
    ref, bound = oref.qmm_gather_ref(fmt, c, s, g, xb[good], "bf16", bad[good], 2, n, k, e)
    _check(out[good], ref, bound, "good rows")


def test_gather_reads_indices_written_by_the_preceding_kernel():
    # The router's output (here a device op enqueued right before) must be
    # read only after it completes: the call waits on the preceding kernel.
    fmt, m, n, k, e = "mxfp4", 6, 512, 4096, 5
    c, s, g, xb, xt, _ = _case(fmt, m, n, k, e, seed=43)
    dc, ds = _dev(c), _dev(s)
    idx_t = torch.full((m,), 0, dtype=torch.int32, device=DEV)
    outs = []
    for r in range(4):
        seq = torch.arange(m, device=DEV, dtype=torch.int32)
        idx_t.copy_((seq * 3 + r) % e)     # written on the stream just before the call
        outs.append((q.qmm_gather(fmt, dc, ds, g, xt, idx_t, n, e), ((np.arange(m) * 3 + r) % e).astype(np.int32)))
    for out, want_idx in outs:
        ref, bound = oref.qmm_gather_ref(fmt, c, s, g, xb, "bf16", want_idx, m, n, k, e)
        _check(out, ref, bound, "chained")


# ------------------------------ expert-grouped rows on the tensor-core GEMM ---

MXB = ["mxfp4", "mxfp8_e4m3", "mxfp8_e5m2"]


def _routing(m, e, seed, kind):
    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return rng.integers(0, e, m).astype(np.int32)
    if kind == "skewed":            # most rows to one expert, some experts empty
        idx = np.where(rng.random(m) < 0.7, 1, rng.integers(0, e, m))
        idx[idx == e - 1] = 0
        return idx.astype(np.int32)
    return np.full(m, e - 1, np.int32)   # every row to the last expert


@pytest.mark.parametrize("fmt", MXB)
@pytest.mark.parametrize("m", [1, 64, 200, 512])
@pytest.mark.parametrize("kind", ["uniform", "skewed", "one"])
def test_grouped_matches_oracle(fmt, m, kind):
    n, k, e = 272, 1024, 8
    c, s, g = opack.pack(fmt, synth.weights(e * n, k, seed=m + 3))
    xb, xt = _x(m, k, seed=m + 4)
    idx = _routing(m, e, seed=m, kind=kind)
    out = q.qmm_grouped(fmt, _dev(c), _dev(s), xt, _dev(idx), n, e)
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_gather_ref(fmt, c, s, g, xb, "bf16", idx, m, n, k, e)
    _check(out, ref, bound, (fmt, m, kind))


@pytest.mark.parametrize("fmt", MXB)
def test_grouped_agrees_with_gather(fmt):
    # the same routed rows through the per-row decode form and the grouped GEMM
    m, n, k, e = 96, 512, 2048, 4
    c, s, g = opack.pack(fmt, synth.weights(e * n, k, seed=11))
    xb, xt = _x(m, k, seed=12)
    idx = _dev(_routing(m, e, seed=13, kind="uniform"))
    a = q.qmm_gather(fmt, _dev(c), _dev(s), g, xt, idx, n, e).float().cpu().numpy()
    b = q.qmm_grouped(fmt, _dev(c), _dev(s), xt, idx, n, e).float().cpu().numpy()
    ref, bound = oref.qmm_gather_ref(fmt, c, s, g, xb, "bf16", idx.cpu().numpy(), m, n, k, e)
    assert (np.abs(a - b) <= 2 * bound + bf16_half_ulp(a) + bf16_half_ulp(b)).all()


def test_grouped_bad_index_zeroes_its_row():
    fmt, m, n, k, e = "mxfp8_e4m3", 130, 128, 512, 3
    c, s, g = opack.pack(fmt, synth.weights(e * n, k, seed=21))
    xb, xt = _x(m, k, seed=22)
    idx = _routing(m, e, seed=23, kind="uniform")
    idx[7] = e
    idx[50] = -1
    out = q.qmm_grouped(fmt, _dev(c), _dev(s), xt, _dev(idx), n, e).float().cpu().numpy()
    assert q.qfmt_device_status() == -9
    assert (out[7] == 0).all() and (out[50] == 0).all()
    good = np.ones(m, bool)
    good[[7, 50]] = False
    ref, bound = oref.qmm_gather_ref(fmt, c, s, g, xb[good], "bf16", idx[good], int(good.sum()), n, k, e)
    _check(torch.from_numpy(out[good]).to(torch.bfloat16), ref, bound, "good rows")


def test_grouped_chained_with_a_router_kernel():
    # the routing indices written by a preceding kernel on the same stream
    fmt, m, n, k, e = "mxfp4", 256, 256, 256, 8
    c, s, g = opack.pack(fmt, synth.weights(e * n, k, seed=31))
    dc, ds = _dev(c), _dev(s)
    xb, xt = _x(m, k, seed=32)
    idx_host = _routing(m, e, seed=33, kind="skewed")
    idx = torch.zeros(m, dtype=torch.int32, device=DEV)
    src = _dev(idx_host)
    for _ in range(3):
        idx.zero_()
        idx.add_(src)                                  # the "router" writes the indices
        out = q.qmm_grouped(fmt, dc, ds, xt, idx, n, e)
    torch.cuda.synchronize()
    ref, bound = oref.qmm_gather_ref(fmt, c, s, g, xb, "bf16", idx_host, m, n, k, e)
    _check(out, ref, bound, "chained")
