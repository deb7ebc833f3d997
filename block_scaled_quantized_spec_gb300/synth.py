"""Seeded synthetic inputs for the block-scaled dequantizing matmul.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no element/scale codecs, no packing, no matmul). Both the
CPU oracle's tests and the CUDA path's tests and benchmark take their inputs
from here, so the two sides see identical bytes.

Workload recipe (the shapes come from the fused dequantizing-matmul workloads
described for the block-scaled formats: an mxfp4 decode GEMV at N = K = 4096,
an nvfp4 batch GEMV on a 14336 x 4096 projection, an mxfp8 prefill GEMM and a
format sweep on an 11008 x 4096 projection):

* W: float32, i.i.d. N(0, 0.02^2), drawn row-major [N, K] from
  ``numpy.random.default_rng(seed)``.  The nvfp4 workload multiplies a 0.1 %
  random subset of entries by 20 (outliers), selected by
  ``rng.random(N*K) < 1e-3`` drawn after W.
* X: float32 N(0, 1) [M, K] drawn after W (and after the outlier mask), then
  rounded to bfloat16 with round-to-nearest-even; the bf16 bit patterns are the
  input (uint16).  The tiny workload keeps X as float32.
* Raw code/scale bytes for throughput-only runs are uniform random bytes from
  the same generator (the pages' benchmarks use random packed buffers).
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "weights",
    "activations_bf16",
    "activations_f32",
    "bf16_bits_to_f32",
    "f32_to_bf16_bits",
    "random_bytes",
    "WORKLOADS",
]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns uint16 bits.

    NaN inputs are not expected (the generators never draw them).
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = (u + 0x7FFF + lsb) >> 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns (uint16) to float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def weights(n: int, k: int, seed: int = 0, std: float = 0.02,
            outliers: bool = False, rng: np.random.Generator | None = None) -> np.ndarray:
    """W ~ N(0, std^2) float32 [n, k]; with ``outliers`` 0.1 % of entries x20."""
    rng = np.random.default_rng(seed) if rng is None else rng
    w = rng.standard_normal((n, k), dtype=np.float32) * np.float32(std)
    if outliers:
        mask = rng.random(n * k) < 1e-3
        w.reshape(-1)[mask] *= np.float32(20.0)
    return w


def activations_f32(m: int, k: int, seed: int = 0,
                    rng: np.random.Generator | None = None) -> np.ndarray:
    """X ~ N(0, 1) float32 [m, k]."""
    rng = np.random.default_rng(seed) if rng is None else rng
    return rng.standard_normal((m, k), dtype=np.float32)


def activations_bf16(m: int, k: int, seed: int = 0,
                     rng: np.random.Generator | None = None) -> np.ndarray:
    """X ~ N(0, 1) rounded to bfloat16; returns the uint16 bit patterns [m, k]."""
    return f32_to_bf16_bits(activations_f32(m, k, seed, rng))


def random_bytes(nbytes: int, seed: int = 0,
                 rng: np.random.Generator | None = None) -> np.ndarray:
    """Uniform random bytes (uint8) for data-independent throughput runs."""
    rng = np.random.default_rng(seed) if rng is None else rng
    return rng.integers(0, 256, size=nbytes, dtype=np.uint8)


# Named workloads: (format, M values, N, K, X dtype, outliers).
WORKLOADS = {
    "mxfp4_tiny": dict(fmt="mxfp4", Ms=(8,), N=16, K=512, x_dtype="f32", outliers=False),
    "mxfp4_gemv": dict(fmt="mxfp4", Ms=(1,), N=4096, K=4096, x_dtype="bf16", outliers=False),
    "nvfp4_gemv": dict(fmt="nvfp4", Ms=(1, 8), N=14336, K=4096, x_dtype="bf16", outliers=True),
    "mxfp8e4_gemm": dict(fmt="mxfp8_e4m3", Ms=(2048,), N=4096, K=4096, x_dtype="bf16", outliers=False),
    "sweep_int4a": dict(fmt="int4_affine", Ms=(1, 16, 128, 4096), N=11008, K=4096, x_dtype="bf16", outliers=False),
    "sweep_mxfp8e5": dict(fmt="mxfp8_e5m2", Ms=(1, 16, 128, 4096), N=11008, K=4096, x_dtype="bf16", outliers=False),
    "sweep_nvfp8": dict(fmt="nvfp8", Ms=(1, 16, 128, 4096), N=11008, K=4096, x_dtype="bf16", outliers=False),
}
