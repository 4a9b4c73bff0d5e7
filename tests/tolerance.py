"""Parity tolerance between the CUDA path and the oracle.

The bound is the one stated for the method's evaluation: every element within
``2^-7 * |ref| + 1e-2 * rms(ref row)`` and, over all compared elements, the
normalised difference ``1 - 2*sum(x*y) / sum(x^2 + y^2)`` below 1e-4.  All
arithmetic here is fp64 on bf16 values decoded exactly.
"""
from __future__ import annotations

import numpy as np

REL = 2.0 ** -7
ROW_RMS = 1e-2
GLOBAL = 1e-4


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def check(gpu_bits: np.ndarray, ref_bits: np.ndarray, what: str = "") -> dict:
    """gpu_bits, ref_bits: uint16 bf16 bit patterns, [rows][N].  Raises
    AssertionError with the worst offender when the bound is broken."""
    x = bf16_bits_to_f64(gpu_bits).reshape(-1, gpu_bits.shape[-1])
    r = bf16_bits_to_f64(ref_bits).reshape(-1, ref_bits.shape[-1])
    assert x.shape == r.shape, (x.shape, r.shape)
    assert np.isfinite(r).all(), f"{what}: reference has non-finite values"
    if not np.isfinite(x).all():
        bad = np.argwhere(~np.isfinite(x))[0]
        raise AssertionError(f"{what}: GPU value not finite at {tuple(bad)}")
    rms = np.sqrt(np.mean(r * r, axis=1, keepdims=True))
    bound = REL * np.abs(r) + ROW_RMS * rms
    err = np.abs(x - r)
    excess = err - bound
    if (excess > 0).any():
        i = np.unravel_index(np.argmax(excess), excess.shape)
        raise AssertionError(
            f"{what}: element {i} gpu={x[i]!r} ref={r[i]!r} |diff|={err[i]:.4g} "
            f"bound={bound[i]:.4g} ({int((excess > 0).sum())} elements over)")
    den = float(np.sum(x * x + r * r))
    diff = 0.0 if den == 0.0 else 1.0 - 2.0 * float(np.sum(x * r)) / den
    assert diff < GLOBAL, f"{what}: global normalised diff {diff:.3g} >= {GLOBAL}"
    return {"max_err_over_bound": float(np.max(err / np.maximum(bound, 1e-300))),
            "global_diff": diff, "elements": int(x.size)}
