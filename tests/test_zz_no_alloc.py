"""qmm_noalloc: the block-scaled GEMM for callers that cannot allocate device
memory (an engine plugin that is handed only its inputs and outputs, a path
that cannot take cudaMalloc's synchronisation), its scratch in the library's
static device array.

The GPU test calls the entry point through the C ABI twice in a row, on
different shapes (the second call reuses the array the first one left
behind), and compares each output with the existing entry point's (qmm_ex
with a caller workspace) within the tolerance every qmm test uses.  This
file is collected last, so a run that stops at its first failure has already
run every other test; it passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest

import block_scaled_quantized_spec_gb300 as q
from block_scaled_quantized_spec_gb300 import synth
from oracle import pack as opack
from oracle import reference as oref
from tolerance import bf16_half_ulp, check


def _lib():
    from block_scaled_quantized_spec_gb300 import build
    build.build()
    return q.load()


def test_noalloc_refuses_before_any_device_work():
    # format, shape and size checks come before the device is touched: a
    # scratch need above the static array is QFMT_ENOSPACE with its sizes
    lib = _lib()
    p = ctypes.c_void_p(0x1000)
    assert lib.qmm_noalloc(3, p, p, 1.0, p, p, 4096, 256, 8192, 0, None) == -8       # 2 x 32 MiB of codes
    assert b"static scratch" in lib.qfmt_last_error()
    assert lib.qmm_noalloc(2, p, p, 1.0, p, p, 256, 256, 1024, 0, None) == -4        # nvfp4: not block-scaled here
    assert lib.qmm_noalloc(3, p, p, 1.0, p, p, 16, 256, 1024, 0, None) == -4         # the decode GEMV's M
    assert lib.qmm_noalloc(3, p, p, 1.0, p, p, 256, 256, 96, 0, None) == -4          # K not a multiple of 128
    assert lib.qmm_noalloc(1, ctypes.c_void_p(0x1010), p, 1.0, p, p, 256, 256, 1024, 0, None) == -3   # E2M1: 32-byte codes
    assert lib.qmm_noalloc(3, p, p, 1.0, p, p, 0, 256, 1024, 0, None) == 0           # empty: a no-op


@pytest.mark.gpu
def test_noalloc_matches_the_workspace_entry_point_twice():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _lib()
    dev = "cuda:0"
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for i, (fmt, m, n, k) in enumerate([("mxfp8_e4m3", 300, 520, 1024), ("mxfp4", 130, 272, 512)]):
        c, s, g = opack.pack(fmt, synth.weights(n, k, seed=20 + i))
        xb = synth.activations_bf16(m, k, seed=30 + i)
        dc, ds = torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)
        xt = torch.from_numpy(xb.view(np.int16)).to(dev).view(torch.bfloat16)
        out = torch.full((m, n), 7.0, dtype=torch.bfloat16, device=dev)
        st = lib.qmm_noalloc(q.FORMATS[fmt], ctypes.c_void_p(dc.data_ptr()), ctypes.c_void_p(ds.data_ptr()), g,
                             ctypes.c_void_p(xt.data_ptr()), ctypes.c_void_p(out.data_ptr()), m, n, k, 0, stream)
        assert st == 0, lib.qfmt_last_error()
        ws = torch.empty(q.qmm_workspace_bytes(fmt, m, k), dtype=torch.uint8, device=dev)
        want = q.qmm_ex(fmt, dc, ds, g, xt, n, workspace=ws)
        torch.cuda.synchronize()
        assert q.qfmt_device_status() == 0
        a = out.float().cpu().numpy()
        b = want.float().cpu().numpy()
        ref, bound = oref.qmm_ref(fmt, c, s, g, xb, "bf16", m, n, k)
        assert np.isfinite(a).all()
        assert (np.abs(a - b) <= 2 * bound + bf16_half_ulp(a) + bf16_half_ulp(b)).all(), (fmt, "call", i)
        check(a, ref, bound, (fmt, "qmm_noalloc call", i))
