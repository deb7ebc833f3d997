"""Python binding of libqfmt (argument marshalling only).

Every function has the name of the C-ABI entry point it wraps (declared in
``include/qfmt.h``) and does nothing but check Python-side types, pass raw
pointers and sizes, and raise ``QfmtError`` on a non-zero status.  All
arithmetic runs in the library: the host packer in C++ and every device step
in the CUDA kernels.  If ``libqfmt.so`` has not been built the first call
raises; there is no fallback.

PyTorch supplies device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "FORMATS", "QfmtError", "load", "lib_path",
    "qfmt_block_size", "qfmt_codes_bytes", "qfmt_scales_bytes",
    "qfmt_pack", "qfmt_dequant", "qmm", "qmm_ex", "qmm_workspace_bytes", "qmm_gather", "qmm_batched", "qmm_rmsnorm",
    "qmm_gated_rmsnorm",
    "qfmt_last_error",
    "qfmt_version", "qfmt_device_status", "qfmt_debug_set",
]

FORMATS = {"mxfp4": 1, "nvfp4": 2, "mxfp8_e4m3": 3, "mxfp8_e5m2": 4, "nvfp8": 5, "int4_affine": 6,
           "nvfp8_f16": 7, "mxint8": 8, "int8": 9, "int8_f16": 10,
           "int4": 11, "int4_f16": 12, "mxfp4x2": 13, "mxint4": 14,
           "fp4": 15, "fp4_f16": 16, "fp8_e4m3": 17, "fp8_e4m3_f16": 18, "fp8_e5m2": 19, "fp8_e5m2_f16": 20}
F32, BF16 = 0, 1
STATUS = {0: "QFMT_OK", -1: "QFMT_EINVAL", -2: "QFMT_ESHAPE", -3: "QFMT_EALIGN", -4: "QFMT_EUNSUPPORTED",
          -5: "QFMT_ECUDA", -6: "QFMT_ETIMEOUT", -7: "QFMT_ENONFINITE", -8: "QFMT_ENOSPACE", -9: "QFMT_EINDEX"}

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB = None


class QfmtError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {message}")
        self.status = status


def lib_path() -> str:
    return os.path.join(_HERE, "libqfmt.so")


_SIGS = {
    "qfmt_version": (ctypes.c_int, []),
    "qfmt_last_error": (ctypes.c_char_p, []),
    "qfmt_block_size": (ctypes.c_int, [ctypes.c_int]),
    "qfmt_codes_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]),
    "qfmt_scales_bytes": (ctypes.c_int64, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]),
    "qfmt_pack": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_float)]),
    "qfmt_dequant": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                    ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                    ctypes.c_int, ctypes.c_void_p]),
    "qmm": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                           ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                           ctypes.c_void_p]),
    "qmm_ex": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                              ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                              ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "qmm_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]),
    "qmm_gather": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]),
    "qmm_batched": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_void_p),
                                   ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_float),
                                   ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p),
                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]),
    "qmm_rmsnorm": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_int, ctypes.c_void_p]),
    "qmm_gated_rmsnorm": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float,
                                         ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                         ctypes.c_void_p]),
    "qfmt_device_status": (ctypes.c_int, [ctypes.c_void_p]),
    "qfmt_debug_set": (ctypes.c_int, [ctypes.c_int, ctypes.c_int64]),
}


def load() -> ctypes.CDLL:
    """Load libqfmt.so (built by ``build.build()``); raise if it is missing."""
    global _LIB
    if _LIB is None:
        path = lib_path()
        if not os.path.exists(path):
            raise QfmtError(-5, "load", f"{path} not built: run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        return FORMATS[fmt]
    return int(fmt)


def _check(status: int, where: str):
    if status != 0:
        raise QfmtError(status, where, load().qfmt_last_error().decode())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return ctypes.c_void_p(t.ctypes.data)
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    return ctypes.c_void_p(t.data_ptr())


def qfmt_version() -> int:
    return load().qfmt_version()


def qfmt_last_error() -> str:
    return load().qfmt_last_error().decode()


def qfmt_device_status(stream=None) -> int:
    """Wait for the stream; return (and clear) the device status: 0, QFMT_ETIMEOUT (-6) or QFMT_EINDEX (-9)."""
    st = load().qfmt_device_status(_stream(stream))
    if st not in (0, -6, -9):
        _check(st, "qfmt_device_status")
    return st


def qfmt_debug_set(key: int, value: int) -> None:
    _check(load().qfmt_debug_set(key, value), "qfmt_debug_set")


def qfmt_block_size(fmt) -> int:
    return load().qfmt_block_size(_fmt(fmt))


def qfmt_codes_bytes(fmt, N: int, K: int) -> int:
    return load().qfmt_codes_bytes(_fmt(fmt), N, K)


def qfmt_scales_bytes(fmt, N: int, K: int) -> int:
    return load().qfmt_scales_bytes(_fmt(fmt), N, K)


def qmm_workspace_bytes(fmt, M: int, N: int, K: int) -> int:
    return load().qmm_workspace_bytes(_fmt(fmt), M, N, K)


def qfmt_pack(fmt, W: np.ndarray, group: int = 0):
    """Host packer: float32 W [N, K] -> (codes uint8 [N, *], scales uint8 [N, *], global_scale float)."""
    lib = load()
    f = _fmt(fmt)
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    cb, sb = lib.qfmt_codes_bytes(f, N, K), lib.qfmt_scales_bytes(f, N, K)
    if cb < 0 or sb < 0:
        raise QfmtError(-2, "qfmt_pack", f"bad format/shape {fmt} {N}x{K}")
    codes = np.zeros(cb, np.uint8)
    scales = np.zeros(sb, np.uint8)
    g = ctypes.c_float(0.0)
    _check(lib.qfmt_pack(f, _ptr(W), N, K, group, _ptr(codes), _ptr(scales), ctypes.byref(g)), "qfmt_pack")
    return codes.reshape(N, -1) if N else codes, scales.reshape(N, -1) if N else scales, float(g.value)


def qfmt_dequant(fmt, codes, scales, global_scale: float, N: int, K: int, out=None, out_dtype=None,
                 group: int = 0, stream=None):
    """Device dequant into ``out`` (a new [N, K] tensor if None); float32 unless out_dtype is bf16."""
    import torch
    if out is None:
        out = torch.empty((N, K), dtype=out_dtype or torch.float32, device=codes.device)
    od = BF16 if out.dtype == torch.bfloat16 else F32
    _check(load().qfmt_dequant(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(out), od,
                               N, K, group, _stream(stream)), "qfmt_dequant")
    return out


def qmm(fmt, codes, scales, global_scale: float, x, N: int, out=None, group: int = 0, stream=None):
    """out [M, N] bf16 = x [M, K] bf16 . dequant(W)^T on the device."""
    import torch
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().qmm(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), _ptr(out),
                      M, N, K, group, _stream(stream)), "qmm")
    return out


def qmm_ex(fmt, codes, scales, global_scale: float, x, N: int, out=None, out_dtype=None, group: int = 0,
           workspace=None, stream=None):
    """qmm with x in bf16 or float32 and out in bf16 or float32 (default: x's dtype)."""
    import torch
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or x.dtype, device=x.device)
    xd = F32 if x.dtype == torch.float32 else BF16
    od = F32 if out.dtype == torch.float32 else BF16
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().qmm_ex(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), xd, _ptr(out), od,
                         M, N, K, group, _ptr(workspace), ws_bytes, _stream(stream)), "qmm_ex")
    return out


def qmm_gather(fmt, codes, scales, global_scale: float, x, expert_idx, N: int, E: int, out=None, group: int = 0,
               stream=None):
    """out [M, N] bf16: row m = x[m] . dequant(W[expert_idx[m] * N : + N])^T over a stacked [E * N, K] weight.

    ``expert_idx`` is a device int32 tensor [M].
    """
    import torch
    M, K = x.shape
    if expert_idx.dtype != torch.int32 or expert_idx.numel() != M:
        raise QfmtError(-1, "qmm_gather", "expert_idx must be an int32 tensor of M entries")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().qmm_gather(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), _ptr(expert_idx),
                             _ptr(out), M, N, K, E, group, _stream(stream)), "qmm_gather")
    return out


def qmm_batched(fmt, codes, scales, global_scales, x, Ns, outs=None, group: int = 0, stream=None):
    """Products of up to four weights with one activation: outs[i] [M, Ns[i]] bf16 = x . dequant(W_i)^T."""
    import torch
    M, K = x.shape
    count = len(codes)
    if not (len(scales) == len(global_scales) == len(Ns) == count):
        raise QfmtError(-1, "qmm_batched", "codes, scales, global_scales and Ns differ in length")
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.bfloat16, device=x.device) for n in Ns]
    arr = lambda ts: (ctypes.c_void_p * count)(*[t.data_ptr() for t in ts])  # noqa: E731
    _check(load().qmm_batched(_fmt(fmt), count, arr(codes), arr(scales),
                              (ctypes.c_float * count)(*[float(g) for g in global_scales]),
                              (ctypes.c_int64 * count)(*[int(n) for n in Ns]), _ptr(x), arr(outs), M, K, group,
                              _stream(stream)), "qmm_batched")
    return outs


def qmm_rmsnorm(fmt, codes, scales, global_scale: float, x, norm_weight, eps: float, N: int, out=None,
                group: int = 0, stream=None):
    """out [M, N] bf16 = rmsnorm(x; norm_weight, eps) . dequant(W)^T, M <= 2 (x and norm_weight bf16)."""
    import torch
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().qmm_rmsnorm(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), _ptr(norm_weight),
                              float(eps), _ptr(out), M, N, K, group, _stream(stream)), "qmm_rmsnorm")
    return out


def qmm_gated_rmsnorm(fmt, codes, scales, global_scale: float, x, gate, norm_weight, eps: float, N: int, out=None,
                      group: int = 0, stream=None):
    """out [M, N] bf16 = (rmsnorm(x; norm_weight, eps) * silu(gate)) . dequant(W)^T, M <= 2 (bf16 x, gate)."""
    import torch
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _check(load().qmm_gated_rmsnorm(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), _ptr(gate),
                                    _ptr(norm_weight), float(eps), _ptr(out), M, N, K, group, _stream(stream)),
           "qmm_gated_rmsnorm")
    return out

