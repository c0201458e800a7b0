"""Shared checking helpers for the GPU parity tests.

Tolerance, per element, against the oracle's fp16 result D_ref:

    |D_gpu - D_ref| <= 2e-3 * |D_ref| + 1e-3 * sqrt(K)

The relative term covers the fp16 rounding of the output (half an ulp is
2^-11 ≈ 4.9e-4 relative, and the GPU's fp32 sum may round to the other
neighbour: one ulp, 9.8e-4); the absolute term covers fp32 accumulation
error, which grows like sqrt(K) times the size of the products for random
inputs.  Because that absolute term alone can exceed |D| for the
normal(0, 1/sqrt(K)) workloads, a second, non-vacuous check bounds the
relative Frobenius error over the compared entries by 1e-3 (output rounding
alone gives ≈ 2.8e-4), and D is pre-filled with NaN so any element the
kernel fails to write fails the comparison.
"""
from __future__ import annotations

import math

import numpy as np

REL_TOL = 2e-3
ABS_TOL_PER_SQRT_K = 1e-3
FRO_TOL = 1e-3


# bf16 keeps 8 significant bits: one output ulp is up to 2^-7 ≈ 7.8e-3 relative,
# half an ulp of rounding alone gives a relative Frobenius error near 2.3e-3
BF16_REL_TOL = 1e-2
BF16_FRO_TOL = 6e-3


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns (the top half of an fp32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def check_close(d_gpu, d_ref, K: int, what: str = "", dtype: str = "f16", scale: float = 1.0) -> dict:
    """`scale` multiplies the accumulation term (|alpha| of a fused epilogue)."""
    if dtype == "bf16":
        g, r = bf16_bits_to_f64(d_gpu), bf16_bits_to_f64(d_ref)
        rel_tol, fro_tol = BF16_REL_TOL, BF16_FRO_TOL
    else:
        g = np.asarray(d_gpu, dtype=np.float16).astype(np.float64)
        r = np.asarray(d_ref, dtype=np.float16).astype(np.float64)
        rel_tol, fro_tol = REL_TOL, FRO_TOL
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert not np.any(np.isnan(g)), f"{what}: {int(np.isnan(g).sum())} NaN entries (unwritten or bad)"
    diff = np.abs(g - r)
    tol = rel_tol * np.abs(r) + ABS_TOL_PER_SQRT_K * max(scale, 1.0) * math.sqrt(max(K, 1))
    bad = diff > tol
    if np.any(bad):
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} entries out of tolerance, "
                             f"first at {idx.tolist()}: gpu {g[bad][:5]} ref {r[bad][:5]}")
    norm = float(np.linalg.norm(r))
    fro = float(np.linalg.norm(diff)) / norm if norm > 0 else float(np.linalg.norm(diff))
    assert fro <= fro_tol, f"{what}: relative Frobenius error {fro:.3e} > {fro_tol}"
    return {"max_abs": float(diff.max()) if diff.size else 0.0, "rel_fro": fro}
