"""Oracle dequant and dequantizing matmul (TEST INFRASTRUCTURE ONLY).

* ``dequant_exact``: the spec value of every weight, exact in float64.
* ``dequant_f32``: that value rounded once to float32 (the bit-exact contract
  of the library's dequant kernel).
* ``qmm_ref``: out[m, n] = sum_k x[m, k] * w[n, k] in float64 with w the exact
  spec value, plus the error bound 2e-3 * sum_k |x||w| + 1e-6.

Value definitions (page title, then the section):

* mxint8 / mxint4: w = q * 2^(scale_bits - 127), q the signed byte (nibble)
  -- PR #250, the MXINT axis (symmetric integer element, E8M0 block scale).
* mxfp4 / mxfp8: w = elem(code) * 2^(scale_bits - 127) -- metaltile PR #250,
  commit "First spec-conformant block-scaled dequant kernel: mt_mxfp4_dequant"
  and the commit completing the mxfp8 dequant kernels.
* nvfp4: w = (e2m1(code) * e4m3(micro)) * global -- rlx-cpu
  ``thunk/ops/quant.rs`` ``dequant_matmul_nvfp4`` (E2M1 nibble times the E4M3
  block scale times the global FP32 scale, block 16 along K).  The inner
  product is exact, so the single float32 rounding is well defined.
* nvfp8: w = e4m3(code) * scale_f32 (block 16) -- PR #250 format list; its
  fp16-scale twin nvfp8_f16 the same with the scale an IEEE half -- PR #250,
  the fp16-scale axis.
* int8 / int8_f16: w = q * scale, q the signed byte, one float32 (or IEEE
  half) scale per group of 64 -- PR #250, the symmetric integer formats on the
  FP32 per-group scale path and their fp16-scale twin.
* int4 / int4_f16: the same with q the signed nibble (sign-extended from its
  bit 3) -- PR #250, the symmetric intN formats (FP32 group 64) and the
  fp16-scale twin.
* mxfp4x2: w = s0 e2m1(q0) + s1 e2m1(q1), the two residual planes' values
  under their float32 block scales -- rlx-cpu ``dequant_matmul_mxfp4x2``
  (codes [N, 2, K/2], scales [N, 2, K/32]; each product is exact in float64,
  their sum is rounded once in float64, then once to float32 by dequant_f32).
* fp4 / fp8_e4m3 / fp8_e5m2 and their *_f16 twins: w = elem(code) * scale,
  a float32 (IEEE half) scale per 32 -- PR #250, the legacy float formats
  on the FP32 per-group scale path and the fp16-scale axis.
* int2 / int3 / int5 / int6 (and *_f16) and mxint2 / 3 / 5 / 6: w = q * scale
  with q the N-bit code of the row's LSB-first bit stream, sign-extended from
  bit N-1 -- PR #250, the symmetric intN / MXINT formats and the sub-byte
  bit-stream packing.
* int4 affine: w = scale * q + bias with q the LSB-first nibble, group 64 --
  metaltile-std ``tests/qmm_gpu_correctness.rs``, ``cpu_qmm_reference``;
  scale and bias are bf16.  float64 evaluation of s*q + b is exact or, when
  the terms are more than 2^41 apart, already rounds to the float32 answer, so
  one float32 rounding of it equals fmaf(s, q, b).
* qmm: "dequant-then-dot" -- PR #250 qgemv/qmm commits (the oracle the GPU
  kernels are checked against) and rlx-cpu ``lowp_scaled_matmul`` (a
  decode-and-accumulate reference kept for correctness, not speed).
* qmm_batched: up to four products sharing one activation, each the qmm
  value -- PR #250, the batched Q/K/V and batched-4 GEMV commits.
* qmm_rmsnorm: the qmm value of the RMS-normalised activation x * gamma /
  sqrt(mean(x^2) + eps) -- PR #250, the fused RMSNorm + GEMV commit (phase 1
  the sum of squares and its inverse root, phase 2 the GEMV over
  x * norm_weight * inv_rms).
* qmm_gated_rmsnorm: the qmm value of x * gamma * silu(gate) / sqrt(mean(x^2)
  + eps), silu(z) = z sigmoid(z) -- PR #250, the fused gated-RMSNorm + GEMV
  commit (a silu gate times the per-row inverse RMS times the norm weight,
  staged, then the block-scaled GEMV over it); the RMS is of x alone.
* quantize_activations / qmm_a8_ref / qmm_a4_ref: both operands quantized (rlx-cpu
  ``thunk/ops/quant.rs``: ``lowp_compute_scales`` / ``lowp_snap_scale`` /
  ``lowp_quantize`` applied to the activation, then ``lowp_scaled_matmul``,
  acc += (a_s * b_s) * sum_k dec(a) dec(b)): the activation is packed exactly
  as a weight of that format (amax / max_finite in float32, E8M0 snapped up,
  round-to-nearest-even saturating codes) and the product of the two exact
  dequantized operands is taken in float64.  qmm_a8_ref packs the activation
  as MXFP8 E4M3, qmm_a4_ref in the weight's FP4 family (the all-FP4 product:
  MXFP4 against mxfp4, NVFP4 with the activation's own global against nvfp4).
* qmm_gather: expert-routed rows over one stacked [E * N, K] weight, row m
  against rows [e N, e N + N) with e = expert_idx[m] -- PR #250, the MoE
  gather-qmm commit (weight row expert_ids[m] * out_dim + n, one stacked
  packed tensor, one nvfp4 global), and rlx-cpu ``lowp_scaled_grouped_matmul``
  (one row per token against its routed expert).
"""
from __future__ import annotations

import numpy as np

from . import codec
from .pack import BLOCK, ELEM_BITS, FORMATS, INTN, SCALE_BYTES, pack

BOUND_REL = 2e-3
BOUND_ABS = 1e-6
# The quantized-activation product is exact up to float32 accumulation: K
# terms summed in float32 are within K u (u = 2^-24) of the exact sum, relative
# to the sum of the terms' magnitudes; K <= 4096 gives 2^-12.
A8_REL = 2.0 ** -12


def unpack_codes(fmt: str, codes: np.ndarray, n: int, k: int) -> np.ndarray:
    """Packed code bytes -> [N, K] integer codes (nibble 2i is the low nibble of byte i)."""
    b = np.asarray(codes, dtype=np.uint8).reshape(n, -1)
    if ELEM_BITS[fmt] == 8:
        return b.reshape(n, k)
    if ELEM_BITS[fmt] not in (4, 8):   # a row's LSB-first bit stream of `bits`-bit codes
        bits = ELEM_BITS[fmt]
        stream = np.unpackbits(b, axis=1, bitorder="little")[:, : k * bits].reshape(n, k, bits)
        return (stream.astype(np.uint32) << np.arange(bits, dtype=np.uint32)).sum(axis=2).astype(np.uint8)
    out = np.empty((n, k), dtype=np.uint8)
    out[:, 0::2] = b & 0x0F
    out[:, 1::2] = b >> 4
    return out


def block_scales(fmt: str, scales: np.ndarray, global_scale: float, n: int, k: int):
    """Decoded per-block scale terms, each [N, ceil(K/block)] float64.

    Returns (mult, add): w = elem * mult (+ add for int4 affine).  For nvfp4
    ``mult`` is the E4M3 micro-scale only; the global is applied separately so
    that the product order (e2m1 * e4m3) * global is kept.
    """
    nb = -(-k // BLOCK[fmt])
    s = np.asarray(scales, dtype=np.uint8).reshape(n, -1)
    if fmt in ("mxfp4", "mxfp8_e4m3", "mxfp8_e5m2", "mxint8", "mxint4") or fmt.startswith("mxint"):
        return codec.E8M0_TABLE[s.reshape(n, nb)], None
    if fmt == "nvfp4":
        return codec.E4M3_TABLE[s.reshape(n, nb)], None
    if fmt in ("nvfp8", "int8", "int4", "fp4", "fp8_e4m3", "fp8_e5m2") or fmt in ("int2", "int3", "int5", "int6"):
        return np.ascontiguousarray(s).view(np.float32).reshape(n, nb).astype(np.float64), None
    if fmt.endswith("_f16"):
        return np.ascontiguousarray(s).view(np.float16).reshape(n, nb).astype(np.float64), None
    pair = np.ascontiguousarray(s).view(np.uint16).reshape(n, nb, 2)
    return codec.decode_bf16(pair[..., 0]), codec.decode_bf16(pair[..., 1])


def element_values(fmt: str, codes: np.ndarray) -> np.ndarray:
    if fmt in ("mxfp4", "nvfp4", "fp4", "fp4_f16"):
        return codec.E2M1_TABLE[codes]
    if fmt in ("mxfp8_e4m3", "nvfp8", "nvfp8_f16", "fp8_e4m3", "fp8_e4m3_f16"):
        return codec.E4M3_TABLE[codes]
    if fmt in ("mxfp8_e5m2", "fp8_e5m2", "fp8_e5m2_f16"):
        return codec.E5M2_TABLE[codes]
    if fmt in ("mxint8", "int8", "int8_f16"):            # the two's-complement byte
        return codes.astype(np.uint8).view(np.int8).astype(np.float64)
    if fmt in ("int4", "int4_f16", "mxint4"):            # the two's-complement nibble, sign-extended from bit 3
        c = codes.astype(np.int64)
        return np.where(c >= 8, c - 16, c).astype(np.float64)
    if fmt in INTN:                                      # N-bit two's complement, sign-extended from bit N-1
        bits = INTN[fmt]
        c = codes.astype(np.int64)
        return np.where(c >= 1 << (bits - 1), c - (1 << bits), c).astype(np.float64)
    return codes.astype(np.float64)                      # int4 affine: q itself


def dequant_exact(fmt: str, codes, scales, global_scale, n: int, k: int) -> np.ndarray:
    """Exact spec value of W [N, K] in float64."""
    if fmt not in FORMATS:
        raise ValueError(fmt)
    blk = BLOCK[fmt]
    if fmt == "mxfp4x2":
        b = np.asarray(codes, dtype=np.uint8).reshape(n, 2, k // 2)
        s = np.ascontiguousarray(np.asarray(scales, dtype=np.uint8)).view(np.float32).reshape(n, 2, -1)
        col = np.arange(k) // blk
        t0, t1 = (codec.E2M1_TABLE[unpack_codes("mxfp4", b[:, p], n, k)] * s[:, p, col].astype(np.float64)
                  for p in range(2))
        return t0 + t1                                   # the IEEE sum (two signed zeros stay -0)
    e = element_values(fmt, unpack_codes(fmt, codes, n, k))
    mult, add = block_scales(fmt, scales, global_scale, n, k)
    col = np.arange(k) // blk                            # the block of every column (a ragged last one too)
    with np.errstate(invalid="ignore", over="ignore"):
        w = e * mult[:, col]
        if add is not None:
            w = w + add[:, col]
        if fmt == "nvfp4":
            w = w * np.float64(np.float32(global_scale))
    return w


def dequant_f32(fmt: str, codes, scales, global_scale, n: int, k: int) -> np.ndarray:
    """Spec value rounded once to float32 (overflow to +-inf, subnormals kept)."""
    with np.errstate(over="ignore", invalid="ignore"):
        return dequant_exact(fmt, codes, scales, global_scale, n, k).astype(np.float32)


def x_values(x: np.ndarray, x_dtype: str) -> np.ndarray:
    """Activation values in float64: bf16 bit patterns (uint16) or float32."""
    if x_dtype == "bf16":
        return codec.decode_bf16(x)
    if x_dtype == "f32":
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    raise ValueError(x_dtype)


def qmm_ref(fmt, codes, scales, global_scale, x, x_dtype, m, n, k):
    """(ref, bound) for out = X . dequant(W)^T, both [M, N] float64."""
    w = dequant_exact(fmt, codes, scales, global_scale, n, k)
    xv = x_values(x, x_dtype).reshape(m, k)
    ref = xv @ w.T
    bound = BOUND_REL * (np.abs(xv) @ np.abs(w).T) + BOUND_ABS
    return ref, bound


def qmm_ref_sampled(fmt, codes, scales, global_scale, x, x_dtype, m, n, k, rows, cols):
    """(ref, bound) at the sampled (rows[i], cols[i]) pairs only, decoding just those W rows."""
    rows = np.asarray(rows)
    cols = np.asarray(cols)
    uniq, inv = np.unique(cols, return_inverse=True)
    per_row_codes = ELEM_BITS[fmt] * k // 8
    per_row_scales = -(-k // BLOCK[fmt]) * SCALE_BYTES[fmt]
    c = np.asarray(codes, dtype=np.uint8).reshape(n, per_row_codes)[uniq]
    s = np.asarray(scales, dtype=np.uint8).reshape(n, per_row_scales)[uniq]
    w = dequant_exact(fmt, c, s, global_scale, len(uniq), k)[inv]
    xv = x_values(x, x_dtype).reshape(m, k)[rows]
    ref = np.einsum("ik,ik->i", xv, w)
    bound = BOUND_REL * np.einsum("ik,ik->i", np.abs(xv), np.abs(w)) + BOUND_ABS
    return ref, bound


def qmm_gather_ref(fmt, codes, scales, global_scale, x, x_dtype, expert_idx, m, n, k, e):
    """(ref, bound) for the expert-routed product, both [M, N] float64.

    ``codes``/``scales`` hold the stacked [E * N, K] weight; ``expert_idx`` the
    M expert numbers, each in [0, E) (anything else raises ValueError).
    """
    idx = np.asarray(expert_idx).reshape(m)
    if m and (idx.min() < 0 or idx.max() >= e):
        raise ValueError("expert index outside [0, E)")
    w = dequant_exact(fmt, codes, scales, global_scale, e * n, k).reshape(e, n, k)
    xv = x_values(x, x_dtype).reshape(m, k)
    ref = np.empty((m, n))
    bound = np.empty((m, n))
    for i in range(m):
        we = w[idx[i]]
        ref[i] = we @ xv[i]
        bound[i] = BOUND_REL * (np.abs(we) @ np.abs(xv[i])) + BOUND_ABS
    return ref, bound


def qmm_batched_ref(fmt, mats, x, x_dtype, m, k):
    """[(ref, bound)] of each matrix in ``mats`` = [(codes, scales, global_scale, n), ...] against x."""
    return [qmm_ref(fmt, c, s, g, x, x_dtype, m, n, k) for (c, s, g, n) in mats]


def rmsnorm_values(x, x_dtype, gamma_bits, eps, m, k):
    """x * gamma / sqrt(mean_k x^2 + eps), float64 [M, K]; gamma as bf16 bit patterns [K]."""
    xv = x_values(x, x_dtype).reshape(m, k)
    g = codec.decode_bf16(np.asarray(gamma_bits, dtype=np.uint16)).reshape(k)
    inv = 1.0 / np.sqrt(np.mean(xv * xv, axis=1) + eps)
    return xv * g[None, :] * inv[:, None]


def silu(z):
    """z * sigmoid(z) = z / (1 + exp(-z)), float64 (0 in the limit z -> -inf)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def gated_rmsnorm_values(x, gate, x_dtype, gamma_bits, eps, m, k):
    """x * gamma * silu(gate) / sqrt(mean_k x^2 + eps), float64 [M, K]; the root mean square is of x."""
    z = x_values(gate, x_dtype).reshape(m, k)
    return rmsnorm_values(x, x_dtype, gamma_bits, eps, m, k) * silu(z)


def qmm_gated_rmsnorm_ref(fmt, codes, scales, global_scale, x, gate, x_dtype, gamma_bits, eps, m, n, k):
    """(ref, bound) for out = gated_rmsnorm(x, gate) . dequant(W)^T, bound on the gated activation."""
    w = dequant_exact(fmt, codes, scales, global_scale, n, k)
    xt = gated_rmsnorm_values(x, gate, x_dtype, gamma_bits, eps, m, k)
    ref = xt @ w.T
    bound = BOUND_REL * (np.abs(xt) @ np.abs(w).T) + BOUND_ABS
    return ref, bound


def qmm_rmsnorm_ref(fmt, codes, scales, global_scale, x, x_dtype, gamma_bits, eps, m, n, k):
    """(ref, bound) for out = rmsnorm(x) . dequant(W)^T, bound on the normalised activation."""
    w = dequant_exact(fmt, codes, scales, global_scale, n, k)
    xt = rmsnorm_values(x, x_dtype, gamma_bits, eps, m, k)
    ref = xt @ w.T
    bound = BOUND_REL * (np.abs(xt) @ np.abs(w).T) + BOUND_ABS
    return ref, bound



def quantize_activations_global(fmt, x, x_dtype, m, k):
    """(codes, scales, global) of the activation X [M, K] packed as a weight of ``fmt``.

    mxfp4 / mxfp8 E4M3 / E5M2 (global 1.0), or nvfp4: the whole X is one
    tensor to the packer, so its global is amax(X) / (6 * 448).  bf16 and
    float32 values are exact in float32, so the packer sees X itself.
    """
    if fmt not in ("mxfp4", "mxfp8_e4m3", "mxfp8_e5m2", "nvfp4"):
        raise ValueError(fmt)
    xv = x_values(x, x_dtype).reshape(m, k).astype(np.float32)
    return pack(fmt, xv)


def quantize_activations(fmt, x, x_dtype, m, k):
    """(codes, scales) of the activation X [M, K] packed as a weight of ``fmt`` (mxfp4 / mxfp8 E4M3 / E5M2)."""
    if fmt == "nvfp4":
        raise ValueError("nvfp4 carries a global: quantize_activations_global")
    c, s, _ = quantize_activations_global(fmt, x, x_dtype, m, k)
    return c, s


def _qmm_quantized_x_ref(act_fmt, fmt, codes, scales, global_scale, x, x_dtype, m, n, k):
    xc, xs, xg = quantize_activations_global(act_fmt, x, x_dtype, m, k)
    xq = dequant_exact(act_fmt, xc, xs, xg, m, k)
    w = dequant_exact(fmt, codes, scales, global_scale, n, k)
    return xq @ w.T, A8_REL * (np.abs(xq) @ np.abs(w).T) + BOUND_ABS


def qmm_a8_ref(fmt, codes, scales, global_scale, x, x_dtype, m, n, k):
    """(ref, bound) of the both-operands-quantized product: X8 . dequant(W)^T, X8 the MXFP8 E4M3 activation.

    ref is exact in float64; the bound is the float32 accumulation's,
    A8_REL * sum_k |x8||w| + BOUND_ABS.
    """
    return _qmm_quantized_x_ref("mxfp8_e4m3", fmt, codes, scales, global_scale, x, x_dtype, m, n, k)


def qmm_a4_ref(fmt, codes, scales, global_scale, x, x_dtype, m, n, k):
    """(ref, bound) of X4 . dequant(W)^T, the all-FP4 product.

    X4 is the activation packed in W's own FP4 family: MXFP4 (E2M1, E8M0
    scale per 32) against mxfp4 weights, NVFP4 (E2M1, E4M3 scale per 16, the
    tensor's global) against nvfp4 weights.  The same float32-accumulation
    bound as qmm_a8_ref: A8_REL * sum_k |x4||w| + BOUND_ABS.
    """
    act = "nvfp4" if fmt == "nvfp4" else "mxfp4"
    return _qmm_quantized_x_ref(act, fmt, codes, scales, global_scale, x, x_dtype, m, n, k)
