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
    "qmm_gated_rmsnorm", "qmm_noalloc", "qfmt_quantize", "qmm_a8", "qmm_a8_workspace_bytes", "qmm_a4",
    "qmm_a4_workspace_bytes", "qmm_grouped", "qmm_grouped_workspace_bytes",
    "qfmt_last_error",
    "qfmt_version", "qfmt_device_status", "qfmt_debug_set",
]

FORMATS = {"mxfp4": 1, "nvfp4": 2, "mxfp8_e4m3": 3, "mxfp8_e5m2": 4, "nvfp8": 5, "int4_affine": 6,
           "nvfp8_f16": 7, "mxint8": 8, "int8": 9, "int8_f16": 10,
           "int4": 11, "int4_f16": 12, "mxfp4x2": 13, "mxint4": 14,
           "fp4": 15, "fp4_f16": 16, "fp8_e4m3": 17, "fp8_e4m3_f16": 18, "fp8_e5m2": 19, "fp8_e5m2_f16": 20,
           "int2": 21, "int3": 22, "int5": 23, "int6": 24, "int2_f16": 25, "int3_f16": 26, "int5_f16": 27,
           "int6_f16": 28, "mxint2": 29, "mxint3": 30, "mxint5": 31, "mxint6": 32}
# the 2/3/5/6-bit formats (one bit stream per row): qmm / qmm_ex and dequant only
SUB_BYTE = ("int2", "int3", "int5", "int6", "int2_f16", "int3_f16", "int5_f16", "int6_f16",
            "mxint2", "mxint3", "mxint5", "mxint6")
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
    "qfmt_block_size": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "qfmt_codes_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int]),
    "qfmt_scales_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int]),
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
    "qmm_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]),
    "qfmt_quantize": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                     ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]),
    "qmm_a8": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                              ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                              ctypes.c_size_t, ctypes.c_void_p]),
    "qmm_a8_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]),
    "qmm_a4": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                              ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                              ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "qmm_a4_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]),
    "qmm_grouped": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                   ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "qmm_grouped_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]),
    "qmm_noalloc": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                                   ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_void_p]),
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


SIZE_ERROR = (1 << (8 * ctypes.sizeof(ctypes.c_size_t))) - 1   # SIZE_MAX: a size query's error return


def qfmt_block_size(fmt, group: int = 0) -> int:
    """The block along K (0 for an unknown format or a group the format does not take)."""
    return load().qfmt_block_size(_fmt(fmt), group)


def _size(v: int, where: str) -> int:
    if v == SIZE_ERROR:
        raise QfmtError(-2, where, load().qfmt_last_error().decode())
    return v


def qfmt_codes_bytes(fmt, N: int, K: int, group: int = 0) -> int:
    """Bytes of the packed codes of an [N, K] weight; raises QfmtError where the C call returns SIZE_MAX."""
    return _size(load().qfmt_codes_bytes(_fmt(fmt), N, K, group), "qfmt_codes_bytes")


def qfmt_scales_bytes(fmt, N: int, K: int, group: int = 0) -> int:
    """Bytes of the block scales of an [N, K] weight; raises QfmtError where the C call returns SIZE_MAX."""
    return _size(load().qfmt_scales_bytes(_fmt(fmt), N, K, group), "qfmt_scales_bytes")


def qmm_workspace_bytes(fmt, M: int, K: int) -> int:
    return load().qmm_workspace_bytes(_fmt(fmt), M, K)


def qfmt_pack(fmt, W: np.ndarray, group: int = 0):
    """Host packer: float32 W [N, K] -> (codes uint8 [N, *], scales uint8 [N, *], global_scale float)."""
    lib = load()
    f = _fmt(fmt)
    W = np.ascontiguousarray(W, dtype=np.float32)
    N, K = W.shape
    cb, sb = lib.qfmt_codes_bytes(f, N, K, group), lib.qfmt_scales_bytes(f, N, K, group)
    g = ctypes.c_float(0.0)
    if cb == SIZE_ERROR or sb == SIZE_ERROR:   # the packer's own status for the refused format / group / shape
        _check(lib.qfmt_pack(f, _ptr(W), N, K, group, None, None, ctypes.byref(g)), "qfmt_pack")
        raise QfmtError(-2, "qfmt_pack", f"bad format/group/shape {fmt} {N}x{K}")
    codes = np.zeros(cb, np.uint8)
    scales = np.zeros(sb, np.uint8)
    g = ctypes.c_float(0.0)
    _check(lib.qfmt_pack(f, _ptr(W), N, K, group, _ptr(codes), _ptr(scales), ctypes.byref(g)), "qfmt_pack")
    return codes.reshape(N, -1) if N else codes, scales.reshape(N, -1) if N else scales, float(g.value)


def _fail(where: str, msg: str, status: int = -1):
    raise QfmtError(status, where, msg)


def _tensor(t, where: str, name: str, dtype=None, nbytes=None, shape=None):
    """Check one tensor's layout, dtype, shape and size before its pointer crosses the C ABI."""
    import torch
    if not isinstance(t, torch.Tensor):
        _fail(where, f"{name} must be a torch tensor")
    if not t.is_contiguous():
        _fail(where, f"{name} must be contiguous (row-major)")
    if dtype is not None and t.dtype != dtype:
        _fail(where, f"{name} must be {dtype} (is {t.dtype})")
    if shape is not None and tuple(t.shape) != tuple(shape):
        _fail(where, f"{name} must have shape {tuple(shape)} (has {tuple(t.shape)})")
    if nbytes is not None and t.numel() * t.element_size() < nbytes:
        _fail(where, f"{name} holds {t.numel() * t.element_size()} bytes, the call reads {nbytes}")


def _on_device(where: str, **tensors):
    """Every tensor is a CUDA tensor on the device of the first one."""
    dev = None
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            _fail(where, f"{name} must be a CUDA tensor (is on {t.device})")
        dev = dev or t.device
        if t.device != dev:
            _fail(where, f"{name} is on {t.device}, the call runs on {dev}")


def _weights(where, fmt, codes, scales, rows, K, group):
    """codes / scales: device tensors holding at least the packed bytes of a [rows, K] weight."""
    cb = _size(load().qfmt_codes_bytes(_fmt(fmt), rows, K, group), where)
    sb = _size(load().qfmt_scales_bytes(_fmt(fmt), rows, K, group), where)
    _tensor(codes, where, "codes", nbytes=cb)
    _tensor(scales, where, "scales", nbytes=sb)


def _activations(where, x, dtypes=None):
    import torch
    dtypes = dtypes or (torch.bfloat16,)
    if not isinstance(x, torch.Tensor):
        _fail(where, "x must be a torch tensor")
    if x.dim() != 2:
        _fail(where, f"x must be 2-D [M, K] (has {x.dim()} dimensions)")
    if x.dtype not in dtypes:
        _fail(where, f"x must be {' or '.join(str(d) for d in dtypes)} (is {x.dtype})")
    _tensor(x, where, "x")
    return x.shape[0], x.shape[1]


def qfmt_dequant(fmt, codes, scales, global_scale: float, N: int, K: int, out=None, out_dtype=None,
                 group: int = 0, stream=None):
    """Device dequant into ``out`` (a new [N, K] tensor if None); float32 unless out_dtype is bf16."""
    import torch
    where = "qfmt_dequant"
    _weights(where, fmt, codes, scales, N, K, group)
    if out is None:
        out = torch.empty((N, K), dtype=out_dtype or torch.float32, device=codes.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        _fail(where, f"out must be float32 or bfloat16 (is {out.dtype})")
    _tensor(out, where, "out", shape=(N, K))
    _on_device(where, codes=codes, scales=scales, out=out)
    od = BF16 if out.dtype == torch.bfloat16 else F32
    _check(load().qfmt_dequant(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(out), od,
                               N, K, group, _stream(stream)), where)
    return out


def qmm(fmt, codes, scales, global_scale: float, x, N: int, out=None, group: int = 0, stream=None):
    """out [M, N] bf16 = x [M, K] bf16 . dequant(W)^T on the device."""
    import torch
    where = "qmm"
    M, K = _activations(where, x)
    _weights(where, fmt, codes, scales, N, K, group)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _tensor(out, where, "out", dtype=torch.bfloat16, shape=(M, N))
    _on_device(where, x=x, codes=codes, scales=scales, out=out)
    _check(load().qmm(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), _ptr(out),
                      M, N, K, group, _stream(stream)), where)
    return out


def qmm_ex(fmt, codes, scales, global_scale: float, x, N: int, out=None, out_dtype=None, group: int = 0,
           workspace=None, stream=None):
    """qmm with x in bf16 or float32 and out in bf16 or float32 (default: x's dtype).

    ``workspace``: None, or a device tensor of at least ``qmm_workspace_bytes(fmt, M, K)`` bytes.
    """
    import torch
    where = "qmm_ex"
    M, K = _activations(where, x, (torch.bfloat16, torch.float32))
    _weights(where, fmt, codes, scales, N, K, group)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or x.dtype, device=x.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        _fail(where, f"out must be float32 or bfloat16 (is {out.dtype})")
    _tensor(out, where, "out", shape=(M, N))
    ws_bytes = 0
    if workspace is not None:
        _tensor(workspace, where, "workspace")
        ws_bytes = workspace.numel() * workspace.element_size()
    _on_device(where, x=x, codes=codes, scales=scales, out=out, workspace=workspace)
    xd = F32 if x.dtype == torch.float32 else BF16
    od = F32 if out.dtype == torch.float32 else BF16
    _check(load().qmm_ex(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), xd, _ptr(out), od,
                         M, N, K, group, _ptr(workspace), ws_bytes, _stream(stream)), where)
    return out


def qfmt_quantize(fmt, x, codes=None, scales=None, stream=None):
    """Device: an activation [M, K] (bf16 or float32) packed as a weight of an MX format -> (codes, scales)."""
    import torch
    where = "qfmt_quantize"
    M, K = _activations(where, x, (torch.bfloat16, torch.float32))
    cb = _size(load().qfmt_codes_bytes(_fmt(fmt), M, K, 0), where)
    sb = _size(load().qfmt_scales_bytes(_fmt(fmt), M, K, 0), where)
    if codes is None:
        codes = torch.empty((M, cb // max(M, 1)), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((M, sb // max(M, 1)), dtype=torch.uint8, device=x.device)
    _tensor(codes, where, "codes", nbytes=cb)
    _tensor(scales, where, "scales", nbytes=sb)
    _on_device(where, x=x, codes=codes, scales=scales)
    _check(load().qfmt_quantize(_fmt(fmt), _ptr(x), F32 if x.dtype == torch.float32 else BF16, _ptr(codes),
                                _ptr(scales), M, K, _stream(stream)), where)
    return codes, scales


def qmm_a8_workspace_bytes(fmt, M: int, K: int) -> int:
    return load().qmm_a8_workspace_bytes(_fmt(fmt), M, K)


def qmm_a4_workspace_bytes(fmt, M: int, K: int) -> int:
    return load().qmm_a4_workspace_bytes(_fmt(fmt), M, K)


def qmm_a8(fmt, codes, scales, x, N: int, out=None, out_dtype=None, workspace=None, stream=None):
    """out [M, N] = Q(x) . dequant(W)^T, Q(x) the activation packed to MXFP8 E4M3 (both operands quantized)."""
    return _qmm_quantized_x("qmm_a8", fmt, codes, scales, x, N, out, out_dtype, workspace, stream)


def qmm_a4(fmt, codes, scales, global_scale: float, x, N: int, out=None, out_dtype=None, workspace=None, stream=None):
    """out [M, N] = Q4(x) . dequant(W)^T, the all-FP4 product: Q4(x) the activation packed in W's FP4
    family (MXFP4 for mxfp4 W; NVFP4 with its own global for nvfp4 W, whose global is global_scale)."""
    return _qmm_quantized_x("qmm_a4", fmt, codes, scales, x, N, out, out_dtype, workspace, stream,
                            global_scale=global_scale)


def _qmm_quantized_x(where, fmt, codes, scales, x, N, out, out_dtype, workspace, stream, global_scale=None):
    import torch
    M, K = _activations(where, x)
    _weights(where, fmt, codes, scales, N, K, 0)
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=x.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        _fail(where, f"out must be float32 or bfloat16 (is {out.dtype})")
    _tensor(out, where, "out", shape=(M, N))
    lib = load()
    wsb = getattr(lib, where + "_workspace_bytes")
    if workspace is None:
        workspace = torch.empty(max(1, wsb(_fmt(fmt), M, K)), dtype=torch.uint8, device=x.device)
    _tensor(workspace, where, "workspace")
    _on_device(where, x=x, codes=codes, scales=scales, out=out, workspace=workspace)
    head = (_fmt(fmt), _ptr(codes), _ptr(scales)) + (() if global_scale is None else (float(global_scale),))
    _check(getattr(lib, where)(*head, _ptr(x), _ptr(out), F32 if out.dtype == torch.float32 else BF16, M, N, K,
                               _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)), where)
    return out


def qmm_grouped_workspace_bytes(fmt, M: int, K: int, E: int) -> int:
    return load().qmm_grouped_workspace_bytes(_fmt(fmt), M, K, E)


def qmm_grouped(fmt, codes, scales, x, expert_idx, N: int, E: int, out=None, out_dtype=None, workspace=None,
                stream=None):
    """out [M, N]: row m = x[m] . dequant(W[expert_idx[m] N : + N])^T, rows of one expert grouped on the tensor cores."""
    import torch
    where = "qmm_grouped"
    M, K = _activations(where, x)
    if E < 1:
        _fail(where, f"expert count E={E} must be >= 1")
    _weights(where, fmt, codes, scales, E * N, K, 0)
    _tensor(expert_idx, where, "expert_idx", dtype=torch.int32)
    if expert_idx.numel() != M:
        _fail(where, "expert_idx must be an int32 tensor of M entries")
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=x.device)
    if out.dtype not in (torch.float32, torch.bfloat16):
        _fail(where, f"out must be float32 or bfloat16 (is {out.dtype})")
    _tensor(out, where, "out", shape=(M, N))
    if workspace is None:
        workspace = torch.empty(max(1, qmm_grouped_workspace_bytes(fmt, M, K, E)), dtype=torch.uint8, device=x.device)
    _tensor(workspace, where, "workspace")
    _on_device(where, x=x, codes=codes, scales=scales, expert_idx=expert_idx, out=out, workspace=workspace)
    _check(load().qmm_grouped(_fmt(fmt), _ptr(codes), _ptr(scales), _ptr(x), _ptr(expert_idx), _ptr(out),
                              F32 if out.dtype == torch.float32 else BF16, M, N, K, E, _ptr(workspace),
                              workspace.numel() * workspace.element_size(), _stream(stream)), where)
    return out


def qmm_noalloc(fmt, codes, scales, x, N: int, out=None, group: int = 0, stream=None):
    """qmm_ex's block-scaled GEMM with the library's static scratch instead of a workspace (no allocation)."""
    import torch
    where = "qmm_noalloc"
    M, K = _activations(where, x)
    _weights(where, fmt, codes, scales, N, K, group)
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _tensor(out, where, "out", dtype=torch.bfloat16, shape=(M, N))
    _on_device(where, x=x, codes=codes, scales=scales, out=out)
    _check(load().qmm_noalloc(_fmt(fmt), _ptr(codes), _ptr(scales), 1.0, _ptr(x), _ptr(out), M, N, K, group,
                              _stream(stream)), where)
    return out


def qmm_gather(fmt, codes, scales, global_scale: float, x, expert_idx, N: int, E: int, out=None, group: int = 0,
               stream=None):
    """out [M, N] bf16: row m = x[m] . dequant(W[expert_idx[m] * N : + N])^T over a stacked [E * N, K] weight.

    ``expert_idx`` is a device int32 tensor [M].
    """
    import torch
    where = "qmm_gather"
    M, K = _activations(where, x)
    if E < 1:
        _fail(where, f"expert count E={E} must be >= 1")
    _weights(where, fmt, codes, scales, E * N, K, group)
    _tensor(expert_idx, where, "expert_idx", dtype=torch.int32)
    if expert_idx.numel() != M:
        _fail(where, "expert_idx must be an int32 tensor of M entries")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _tensor(out, where, "out", dtype=torch.bfloat16, shape=(M, N))
    _on_device(where, x=x, codes=codes, scales=scales, expert_idx=expert_idx, out=out)
    _check(load().qmm_gather(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), _ptr(expert_idx),
                             _ptr(out), M, N, K, E, group, _stream(stream)), where)
    return out


def qmm_batched(fmt, codes, scales, global_scales, x, Ns, outs=None, group: int = 0, stream=None):
    """Products of up to four weights with one activation: outs[i] [M, Ns[i]] bf16 = x . dequant(W_i)^T."""
    import torch
    where = "qmm_batched"
    M, K = _activations(where, x)
    count = len(codes)
    if not (len(scales) == len(global_scales) == len(Ns) == count):
        _fail(where, "codes, scales, global_scales and Ns differ in length")
    if not 1 <= count <= 4:
        _fail(where, f"count={count} must be 1..4")
    for c, sc, n in zip(codes, scales, Ns):
        _weights(where, fmt, c, sc, int(n), K, group)
    if outs is None:
        outs = [torch.empty((M, n), dtype=torch.bfloat16, device=x.device) for n in Ns]
    if len(outs) != count:
        _fail(where, "outs differs in length from codes")
    for o, n in zip(outs, Ns):
        _tensor(o, where, "out", dtype=torch.bfloat16, shape=(M, int(n)))
    _on_device(where, x=x, **{f"codes[{i}]": t for i, t in enumerate(codes)},
               **{f"scales[{i}]": t for i, t in enumerate(scales)}, **{f"outs[{i}]": t for i, t in enumerate(outs)})
    arr = lambda ts: (ctypes.c_void_p * count)(*[t.data_ptr() for t in ts])  # noqa: E731
    _check(load().qmm_batched(_fmt(fmt), count, arr(codes), arr(scales),
                              (ctypes.c_float * count)(*[float(g) for g in global_scales]),
                              (ctypes.c_int64 * count)(*[int(n) for n in Ns]), _ptr(x), arr(outs), M, K, group,
                              _stream(stream)), where)
    return outs


def _norm_args(where, fmt, codes, scales, x, norm_weight, N, out, group, gate=None):
    import torch
    M, K = _activations(where, x)
    _weights(where, fmt, codes, scales, N, K, group)
    _tensor(norm_weight, where, "norm_weight", dtype=torch.bfloat16, shape=(K,))
    if gate is not None:
        _tensor(gate, where, "gate", dtype=torch.bfloat16, shape=(M, K))
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    _tensor(out, where, "out", dtype=torch.bfloat16, shape=(M, N))
    _on_device(where, x=x, codes=codes, scales=scales, norm_weight=norm_weight, gate=gate, out=out)
    return M, K, out


def qmm_rmsnorm(fmt, codes, scales, global_scale: float, x, norm_weight, eps: float, N: int, out=None,
                group: int = 0, stream=None):
    """out [M, N] bf16 = rmsnorm(x; norm_weight, eps) . dequant(W)^T, M <= 2 (x and norm_weight bf16)."""
    where = "qmm_rmsnorm"
    M, K, out = _norm_args(where, fmt, codes, scales, x, norm_weight, N, out, group)
    _check(load().qmm_rmsnorm(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), _ptr(norm_weight),
                              float(eps), _ptr(out), M, N, K, group, _stream(stream)), where)
    return out


def qmm_gated_rmsnorm(fmt, codes, scales, global_scale: float, x, gate, norm_weight, eps: float, N: int, out=None,
                      group: int = 0, stream=None):
    """out [M, N] bf16 = (rmsnorm(x; norm_weight, eps) * silu(gate)) . dequant(W)^T, M <= 2 (bf16 x, gate)."""
    where = "qmm_gated_rmsnorm"
    if gate is None:
        _fail(where, "gate is None")
    M, K, out = _norm_args(where, fmt, codes, scales, x, norm_weight, N, out, group, gate=gate)
    _check(load().qmm_gated_rmsnorm(_fmt(fmt), _ptr(codes), _ptr(scales), float(global_scale), _ptr(x), _ptr(gate),
                                    _ptr(norm_weight), float(eps), _ptr(out), M, N, K, group, _stream(stream)),
           where)
    return out
