"""CPU tests of libqfmt: it loads, exports every symbol the header declares, its
host packer matches the oracle byte for byte, and argument validation
rejects bad calls before any device work (no GPU needed)."""
import ctypes
import os
import re

import numpy as np
import pytest

import block_scaled_quantized_spec_gb300 as q
from block_scaled_quantized_spec_gb300 import synth
from oracle import pack as opack

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qfmt.h")


@pytest.fixture(scope="module")
def lib():
    from block_scaled_quantized_spec_gb300 import build
    build.build()
    return q.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_abi():
    names = _declared_functions()
    for must in ("qfmt_pack", "qfmt_dequant", "qmm", "qmm_ex", "qfmt_last_error", "qfmt_codes_bytes",
                 "qfmt_scales_bytes", "qfmt_block_size", "qmm_workspace_bytes", "qfmt_version"):
        assert must in names, must


def test_library_exports_every_declared_symbol(lib):
    cdll = ctypes.CDLL(q.lib_path())
    for name in _declared_functions():
        assert hasattr(cdll, name), name
    assert q.qfmt_version() >= 100


def test_sizes_and_blocks(lib):
    for name, f in q.FORMATS.items():
        blk = opack.BLOCK[name]
        assert q.qfmt_block_size(name) == blk
        assert q.qfmt_block_size(name, blk) == blk            # the format's own block, stated
        assert q.qfmt_codes_bytes(name, 7, 256) == opack.codes_nbytes(name, 7, 256)
        assert q.qfmt_scales_bytes(name, 7, 256) == opack.scales_nbytes(name, 7, 256)
        assert q.qfmt_codes_bytes(name, 7, 256, blk) == opack.codes_nbytes(name, 7, 256)
    assert q.qfmt_scales_bytes("int4_affine", 4, 96) == 4 * 2 * 4   # a ragged last group of 32
    assert q.qfmt_codes_bytes("mxfp8_e4m3", (1 << 31) - 1, 32) == ((1 << 31) - 1) * 32
    assert q.qfmt_codes_bytes("mxfp4x2", (1 << 30) - 1, 32) == ((1 << 30) - 1) * 32


def test_size_queries_error_returns(lib):
    # every size query through the C ABI: 0 (block) or SIZE_MAX (bytes) on an
    # unknown format, a group the format does not take, or a shape the packer
    # refuses, with the reason in qfmt_last_error
    SMAX = q.SIZE_ERROR
    assert lib.qfmt_block_size(99, 0) == 0 and b"unknown format" in lib.qfmt_last_error()
    assert lib.qfmt_block_size(1, 64) == 0 and b"group" in lib.qfmt_last_error()
    assert lib.qfmt_block_size(6, 32) == 0
    assert lib.qfmt_last_error() != b""
    assert lib.qfmt_block_size(6, 0) == 64 and lib.qfmt_last_error() == b""
    for fn in (lib.qfmt_codes_bytes, lib.qfmt_scales_bytes):
        assert fn(99, 4, 64, 0) == SMAX and b"unknown format" in lib.qfmt_last_error()
        assert fn(1, 4, 64, 16) == SMAX and b"group" in lib.qfmt_last_error()
        assert fn(1, 4, 48, 0) == SMAX and b"multiple" in lib.qfmt_last_error()     # K not a multiple of 32
        assert fn(6, 4, 80, 0) == SMAX                                               # int4 affine too
        assert fn(1, -1, 64, 0) == SMAX and b"negative" in lib.qfmt_last_error()
        assert fn(3, 1 << 31, 32, 0) == SMAX                                         # 2^31 code rows
        assert fn(13, 1 << 30, 32, 0) == SMAX                                        # mxfp4x2: 2N code rows
        assert fn(1, 0, 64, 0) == 0 and lib.qfmt_last_error() == b""
    with pytest.raises(q.QfmtError):
        q.qfmt_codes_bytes("mxfp4", 4, 48)


CASES = [
    (16, 512, 0, 0.02, False),
    (37, 1024, 1, 0.02, True),
    (8, 256, 2, 1e-20, False),      # tiny weights: subnormal scales / codes
    (8, 256, 3, 3e3, False),        # large weights
    (4, 2048, 4, 0.02, True),
    (5, 96, 5, 0.02, False),        # K = 96: int4 affine's ragged last group of 32
    (3, 4128, 6, 0.02, True),       # K = 64 * 64 + 32
]


@pytest.mark.parametrize("fmt", list(q.FORMATS))
@pytest.mark.parametrize("n,k,seed,std,outl", CASES)
def test_host_pack_matches_oracle_bytes(lib, fmt, n, k, seed, std, outl):
    w = synth.weights(n, k, seed=seed, std=std, outliers=outl)
    c_lib, s_lib, g_lib = q.qfmt_pack(fmt, w)
    c_or, s_or, g_or = opack.pack(fmt, w)
    assert np.array_equal(c_lib, c_or), fmt
    assert np.array_equal(s_lib, s_or), fmt
    assert np.float32(g_lib) == g_or


@pytest.mark.parametrize("fmt", list(q.FORMATS))
def test_host_pack_special_blocks(lib, fmt):
    n, k = 6, 256
    w = synth.weights(n, k, seed=9)
    w[0] = 0.0                                  # all-zero row
    w[1, :64] = 0.0                             # zero blocks
    w[2, 5] = -0.0
    w[3, :] = np.float32(1e-40)                 # subnormal weights
    w[4, 0] = np.float32(5.0e4)                 # a block with a large maximum
    w[5, ::2] = -w[5, 1::2]                     # exact ties in magnitude
    c_lib, s_lib, g_lib = q.qfmt_pack(fmt, w)
    c_or, s_or, g_or = opack.pack(fmt, w)
    assert np.array_equal(c_lib, c_or) and np.array_equal(s_lib, s_or) and np.float32(g_lib) == g_or


def test_host_pack_exhaustive_midpoints(lib):
    # Every representable value and midpoint of each element grid, placed in a
    # block whose amax pins the scale to 1: the library's arithmetic encoder and
    # the oracle's table search must agree on every tie and on saturation.
    from oracle import codec
    for fmt, table, maxf in (("mxfp4", codec.E2M1_TABLE[:8], 6.0),
                             ("mxfp8_e4m3", codec.E4M3_TABLE[:127], 448.0),
                             ("mxfp8_e5m2", codec.E5M2_TABLE[:124], 57344.0)):
        vals = np.sort(table[np.isfinite(table)])
        mids = (vals[:-1] + vals[1:]) / 2
        probes = np.concatenate([vals, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                                 np.nextafter(mids.astype(np.float32), np.float32(1e9))]).astype(np.float32)
        probes = np.concatenate([probes, -probes])
        blocks = -(-len(probes) // 31)
        w = np.zeros((blocks, 32), np.float32)
        w[:, 0] = maxf
        w[:, 1:].reshape(-1)[:len(probes)] = probes
        w = w.reshape(1, -1)
        c_lib, s_lib, _ = q.qfmt_pack(fmt, w)
        c_or, s_or, _ = opack.pack(fmt, w)
        assert (s_or == 127).all()
        assert np.array_equal(c_lib, c_or), fmt
        assert np.array_equal(s_lib, s_or), fmt


def test_host_pack_rejects_bad_input(lib):
    with pytest.raises(q.QfmtError) as e:
        q.qfmt_pack("mxfp4", np.full((2, 32), np.inf, np.float32))
    assert e.value.status == -7
    with pytest.raises(q.QfmtError) as e:
        q.qfmt_pack("mxfp4", np.zeros((2, 32), np.float32), group=16)
    assert e.value.status == -4
    with pytest.raises(q.QfmtError):
        q.qfmt_pack(42, np.zeros((2, 32), np.float32))
    with pytest.raises(q.QfmtError):
        q.qfmt_pack("nvfp4", np.zeros((2, 40), np.float32))


def _call_qmm(lib, **kw):
    a = dict(fmt=1, codes=0x1000, scales=0x1000, g=1.0, x=0x1000, xd=1, out=0x1000, od=1,
             M=4, N=4, K=64, group=0)
    a.update(kw)
    return lib.qmm_ex(a["fmt"], a["codes"], a["scales"], a["g"], a["x"], a["xd"], a["out"], a["od"],
                      a["M"], a["N"], a["K"], a["group"], None, 0, None)


def test_device_entry_validation_without_gpu(lib):
    # each of these fails in host-side validation, before any CUDA call
    assert _call_qmm(lib, fmt=0) == -1
    assert _call_qmm(lib, fmt=33) == -1
    assert _call_qmm(lib, K=48) == -2
    assert _call_qmm(lib, M=-1) == -2
    assert _call_qmm(lib, group=64) == -4
    assert _call_qmm(lib, xd=5) == -1
    assert _call_qmm(lib, od=9) == -1
    assert _call_qmm(lib, codes=0x1008) == -3
    assert _call_qmm(lib, x=0x1004) == -3
    assert _call_qmm(lib, out=0x1002) == -3
    assert _call_qmm(lib, scales=0x1002) == -3
    assert _call_qmm(lib, codes=None) == -1
    assert _call_qmm(lib, fmt=2, g=0.0) == -1
    assert _call_qmm(lib, fmt=2, g=float("nan")) == -1
    assert _call_qmm(lib, fmt=6, K=80) == -2
    assert b"multiple" in lib.qfmt_last_error()
    # more 128-row GEMM tiles than the grid's y dimension holds: refused before any launch
    assert _call_qmm(lib, M=65535 * 128 + 1) == -2
    assert b"65535" in lib.qfmt_last_error()
    # empty problems are legal no-ops
    assert _call_qmm(lib, M=0) == 0
    assert _call_qmm(lib, N=0) == 0
    assert lib.qfmt_dequant(1, None, None, 1.0, None, 0, 0, 64, 0, None) == 0
    assert lib.qfmt_dequant(1, 0x1000, 0x1000, 1.0, 0x1000, 3, 4, 64, 0, None) == -1
    assert lib.qfmt_dequant(1, 0x1000, 0x1000, 1.0, 0x1004, 0, 4, 64, 0, None) == -3


def _call_gather(lib, **kw):
    a = dict(fmt=1, codes=0x1000, scales=0x1000, g=1.0, x=0x1000, idx=0x2000, out=0x1000,
             M=4, N=4, K=64, E=2, group=0)
    a.update(kw)
    return lib.qmm_gather(a["fmt"], a["codes"], a["scales"], a["g"], a["x"], a["idx"], a["out"],
                          a["M"], a["N"], a["K"], a["E"], a["group"], None)


def test_gather_entry_validation_without_gpu(lib):
    # each fails in host-side validation, before any CUDA call
    assert _call_gather(lib, E=0) == -1
    assert _call_gather(lib, M=70000) == -2
    assert _call_gather(lib, E=1 << 20, N=1 << 12) == -2          # E * N above 2^31
    assert _call_gather(lib, E=1 << 19, N=1 << 12) == -2          # E * N = 2^31
    assert _call_gather(lib, K=48) == -2
    assert _call_gather(lib, idx=None) == -1
    assert _call_gather(lib, idx=0x2002) == -3
    assert _call_gather(lib, x=0x1004) == -3
    assert _call_gather(lib, fmt=2, g=0.0) == -1
    assert _call_gather(lib, group=32, fmt=6) == -4
    assert b"expert" in lib.qfmt_last_error() or _call_gather(lib, E=0) == -1
    assert _call_gather(lib, M=0) == 0 and _call_gather(lib, N=0) == 0


def test_batched_and_rmsnorm_validation_without_gpu(lib):
    P = ctypes.c_void_p
    arr = lambda *v: (P * len(v))(*v)  # noqa: E731
    f = lambda *v: (ctypes.c_float * len(v))(*v)  # noqa: E731
    n = lambda *v: (ctypes.c_int64 * len(v))(*v)  # noqa: E731
    ok = dict(codes=arr(0x1000, 0x1000), scales=arr(0x1000, 0x1000), g=f(1.0, 1.0), N=n(4, 4),
              out=arr(0x1000, 0x1000))

    def batched(count=2, x=0x1000, M=1, K=64, **kw):
        a = dict(ok)
        a.update(kw)
        return lib.qmm_batched(1, count, a["codes"], a["scales"], a["g"], a["N"], x, a["out"], M, K, 0, None)

    assert batched(count=0) == -1
    assert batched(count=5) == -1
    assert batched(K=48) == -2
    assert batched(out=arr(0x1000, 0x1004)) == -3
    assert batched(codes=arr(0x1000, 0x1008)) == -3
    assert batched(x=0x1002) == -3
    assert batched(M=0) == 0

    def rms(M=1, eps=1e-5, gamma=0x1000, K=64, N=4):
        return lib.qmm_rmsnorm(1, 0x1000, 0x1000, 1.0, 0x1000, gamma, eps, 0x1000, M, N, K, 0, None)

    assert rms(M=3) == -4
    assert rms(eps=-1.0) == -1
    assert rms(eps=float("inf")) == -1
    assert rms(K=0) == -2
    assert rms(gamma=0x1008) == -3
    assert rms(gamma=None) == -1
    assert rms(M=0) == 0 and rms(N=0) == 0

    def gated(M=1, eps=1e-5, gate=0x2000, gamma=0x1000, K=64, N=4):
        return lib.qmm_gated_rmsnorm(1, 0x1000, 0x1000, 1.0, 0x1000, gate, gamma, eps, 0x1000, M, N, K, 0, None)

    assert gated(gate=None) == -1
    assert gated(gate=0x2004) == -3
    assert gated(M=3) == -4
    assert gated(eps=float("nan")) == -1
    assert gated(K=0) == -2
    assert gated(M=0) == 0


def test_binding_rejects_bad_tensors_before_the_call(lib):
    # the binding checks every tensor before a pointer crosses the C ABI:
    # contiguity, dtype, shape, buffer size, then the device (CPU tensors here,
    # so every rejection below happens on the host)
    import torch
    fmt, n, k = "mxfp4", 8, 64
    codes = torch.zeros(q.qfmt_codes_bytes(fmt, n, k), dtype=torch.uint8)
    scales = torch.zeros(q.qfmt_scales_bytes(fmt, n, k), dtype=torch.uint8)
    x = torch.zeros((2, k), dtype=torch.bfloat16)

    def rejects(fn, *a, match, **kw):
        with pytest.raises(q.QfmtError) as e:
            fn(*a, **kw)
        assert match in str(e.value), (match, str(e.value))

    rejects(q.qmm, fmt, codes, scales, 1.0, x.float(), n, match="must be torch.bfloat16")
    rejects(q.qmm, fmt, codes, scales, 1.0, torch.zeros((2, 2 * k), dtype=torch.bfloat16)[:, ::2], n,
            match="contiguous")
    rejects(q.qmm, fmt, codes, scales, 1.0, torch.zeros((2, 1, k), dtype=torch.bfloat16), n, match="2-D")
    rejects(q.qmm, fmt, codes[:-1], scales, 1.0, x, n, match="codes holds")
    rejects(q.qmm, fmt, codes, scales[:-1], 1.0, x, n, match="scales holds")
    rejects(q.qmm, fmt, codes, scales, 1.0, x, n, out=torch.zeros((2, n), dtype=torch.float32),
            match="out must be torch.bfloat16")
    rejects(q.qmm, fmt, codes, scales, 1.0, x, n, out=torch.zeros((2, n + 1), dtype=torch.bfloat16),
            match="shape")
    rejects(q.qmm, fmt, codes, scales, 1.0, x, n, match="CUDA tensor")
    rejects(q.qmm, fmt, codes, scales, 1.0, torch.zeros((2, 48), dtype=torch.bfloat16), n, match="multiple")
    rejects(q.qmm_ex, fmt, codes, scales, 1.0, x.to(torch.float16), n, match="must be")
    rejects(q.qfmt_dequant, fmt, codes, scales, 1.0, n, k, out=torch.zeros((n, k), dtype=torch.float16),
            match="float32 or bfloat16")
    rejects(q.qmm_gather, fmt, codes, scales, 1.0, x, torch.zeros(2, dtype=torch.int64), n, 1,
            match="int32")
    rejects(q.qmm_gather, fmt, codes, scales, 1.0, x, torch.zeros(2, dtype=torch.int32), n, 2,
            match="codes holds")                                  # two experts need twice the codes
    rejects(q.qmm_rmsnorm, fmt, codes, scales, 1.0, x, torch.zeros(k + 1, dtype=torch.bfloat16), 1e-5, n,
            match="norm_weight must have shape")
    rejects(q.qmm_gated_rmsnorm, fmt, codes, scales, 1.0, x, torch.zeros((2, k), dtype=torch.float32),
            torch.zeros(k, dtype=torch.bfloat16), 1e-5, n, match="gate must be torch.bfloat16")
    rejects(q.qmm_batched, fmt, [codes] * 5, [scales] * 5, [1.0] * 5, x, [n] * 5, match="1..4")


def test_debug_keys_without_gpu(lib):
    # the test and measurement settings are host state: every documented key
    # takes its default value, unknown keys and values are refused
    for key in range(1, 10):
        q.qfmt_debug_set(key, 0)
    for key in (8, 9):
        for value in (1, 2, 0):
            q.qfmt_debug_set(key, value)
    for key, value in ((0, 0), (10, 0), (-1, 1), (8, 3), (8, -1), (9, 3)):
        with pytest.raises(q.QfmtError) as e:
            q.qfmt_debug_set(key, value)
        assert e.value.status == -1


def test_quantized_activation_workspace_sizes(lib):
    # codes, then 512-byte scale atoms per 128-row tile (a 4-byte cell per row
    # covers 128 K for E8M0 per 32, 64 K for nvfp4's E4M3 per 16), then for
    # nvfp4 the maxima scratch and the global; each part 1 KiB aligned
    al = lambda v: (v + 1023) // 1024 * 1024  # noqa: E731
    for m, k in [(1, 256), (300, 1024), (2048, 4096)]:
        mp = (m + 127) // 128 * 128
        assert q.qmm_a8_workspace_bytes("mxfp8_e4m3", m, k) == al(m * k) + al(mp * k // 32)
        assert q.qmm_a4_workspace_bytes("mxfp4", m, k) == al(m * k // 2) + al(mp * k // 32)
        assert q.qmm_a4_workspace_bytes("nvfp4", m, k) == al(m * k // 2) + al(mp * k // 16) + al(4 * 1025)
    assert q.qmm_a4_workspace_bytes("mxfp8_e4m3", 8, 256) == 0
    assert q.qmm_a4_workspace_bytes("mxfp4", 8, 384) == 0
    assert q.qmm_a4_workspace_bytes("nvfp4", 0, 256) == 0


def test_qmm_a4_rejects_before_device_work(lib):
    f = q.FORMATS
    args = lambda fmt, m, k: (f[fmt], None, None, 1.0, None, None, 1, m, 64, k, None, 0, None)  # noqa: E731
    assert lib.qmm_a4(*args("mxfp8_e4m3", 8, 256)) == -4     # a weight format with no FP4 pairing
    assert lib.qmm_a4(*args("mxfp4", 8, 384)) == -2          # K not a multiple of 256
    assert lib.qmm_a4(*args("nvfp4", 8, 256)) == -8          # no workspace
    assert lib.qmm_a4(*args("mxfp4", 0, 256)) == 0           # M = 0: nothing to do
