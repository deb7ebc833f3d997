"""The parity tolerance of the dequantizing matmul, as every GPU test applies it.

The method bounds the float32-accumulated result v of each output:

    |v - ref| <= 2e-3 * sum_k |x[m,k]| |w[n,k]| + 1e-6,

ref the exact float64 dequant-then-dot.  A bf16 output is v rounded once to
the nearest bf16, which moves it by at most half a bf16 ulp of the stored
value (2^(e - 8) for a stored value in [2^e, 2^(e+1)); bf16 keeps 8
significant bits).  The bound alone cannot cover that rounding: when few terms
of one sign make |ref| close to sum |x||w| (K = 32, say), the correctly rounded
exact result already lies up to 2^-8 |ref| > 2e-3 sum |x||w| away.  So a bf16
output is checked against

    |out - ref| <= bound + ulp_bf16(out) / 2,

and a float32 output against the bound alone.  Every failure message gives the
largest err / bound both without the half-ulp term and with it.
"""
import numpy as np


def bf16_half_ulp(out: np.ndarray) -> np.ndarray:
    """Half a bf16 ulp of each (bf16-representable) value: 2^(floor(log2|v|) - 8), 2^-134 at zero."""
    a = np.abs(np.asarray(out, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)                 # the subnormal range keeps the ulp of 2^-126
    return np.where(np.isfinite(a), np.ldexp(1.0, (e - 8).astype(np.int64)), 0.0)


def check(out, ref, bound, what, bf16=True):
    """Assert |out - ref| <= bound (+ half a bf16 ulp of out); return (max err/bound, max err/allowed)."""
    out = np.asarray(out, dtype=np.float64)
    assert np.isfinite(out).all(), (what, "non-finite output", np.argwhere(~np.isfinite(out))[:5].tolist())
    err = np.abs(out - ref)
    allowed = bound + (bf16_half_ulp(out) if bf16 else 0.0)
    raw = float((err / bound).max()) if err.size else 0.0
    rel = float((err / allowed).max()) if err.size else 0.0
    ok = err <= allowed
    assert ok.all(), (what, f"max err/bound {raw:.4g} (without the bf16 half ulp), {rel:.4g} (with it)",
                      np.argwhere(~ok)[:5].tolist())
    return raw, rel


def check_tensor(out_t, ref, bound, what):
    """check() for a torch output tensor (bf16 or float32)."""
    import torch
    return check(out_t.float().cpu().numpy(), ref, bound, what, bf16=out_t.dtype == torch.bfloat16)
