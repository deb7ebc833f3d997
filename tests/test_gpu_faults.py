"""Failure detection on the GPU without a fault: every pipeline wait of the
tensor-core GEMMs and every weight-copy wait of the decode GEMV is bounded.
A test hook makes a stage never signal (the GEMMs' decoder or scale warps skip
their arrivals; the decode GEMVs do not issue their weight or activation
copies), the wait
runs out after a short limit, the kernel records QFMT_ETIMEOUT in the device
status word and stores nothing; the context stays usable for the next correct
call."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import block_scaled_quantized_spec_gb300 as q  # noqa: E402
from block_scaled_quantized_spec_gb300 import synth  # noqa: E402
from oracle import pack as opack  # noqa: E402
from oracle import reference as oref  # noqa: E402
from tolerance import check  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_scaled_quantized_spec_gb300 import build
    build.build()
    q.load()


@pytest.mark.parametrize("fmt,m,n,k", [
    ("mxfp8_e4m3", 128, 256, 512),     # one CTA a tile (no K split)
    ("mxfp4", 128, 2048, 4096),        # 8 tiles of one M row: K split over clusters of CTAs
    ("mxfp4", 1, 4096, 4096),          # the decode GEMV's staged weight copies (not issued)
    ("nvfp4", 2, 1000, 2048),          # the same, M = 2, a ragged last tile
    ("mxint8", 8, 1300, 1024),         # the one-decode batch GEMV's activation copies (not issued)
])
def test_expired_wait_reports_timeout_and_context_survives(fmt, m, n, k):
    w = synth.weights(n, k, seed=3)
    c, s, g = opack.pack(fmt, w)
    xb = synth.activations_bf16(m, k, seed=4)
    dc = torch.from_numpy(c).cuda()
    ds = torch.from_numpy(s).cuda()
    xt = torch.from_numpy(xb.view(np.int16)).cuda().view(torch.bfloat16)
    assert q.qfmt_device_status() == 0
    q.qfmt_debug_set(1, 20_000_000)          # 20 ms per wait
    q.qfmt_debug_set(2, 1)                   # decoders never signal
    sentinel = torch.full((m, n), 3.0, dtype=torch.bfloat16, device="cuda")
    try:
        q.qmm(fmt, dc, ds, g, xt, n, out=sentinel)
        st = q.qfmt_device_status()
        msg = q.qfmt_last_error()
    finally:
        q.qfmt_debug_set(2, 0)
        q.qfmt_debug_set(1, 0)
    assert st == -6
    assert "expired" in msg
    # a kernel that gave up writes no output (a K split: no CTA of the cluster)
    assert (sentinel.float() == 3.0).all()
    # the context is intact: the next call is correct and reports no error
    out = q.qmm(fmt, dc, ds, g, xt, n).float().cpu().numpy()
    assert q.qfmt_device_status() == 0
    ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
    check(out, ref, bound, (fmt, "after the expired wait"))


def test_debug_set_rejects_unknown_key():
    with pytest.raises(q.QfmtError):
        q.qfmt_debug_set(99, 1)
