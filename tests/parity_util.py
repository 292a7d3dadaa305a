"""Comparison of the CUDA path's outputs with the fp64 oracle's.

Tolerances: |dLSE| <= 1e-3 and |dO| <= 1e-2 (bf16 inputs, fp32 accumulation).
O leaves the kernel as bf16, and even the best bf16 value -- the exact result
rounded to nearest -- sits up to half a bf16 spacing from the exact result
(2^-8 for |O| in [2, 4), 2^-7 in [4, 8): more than 1e-2 there).  So the O
bound is applied to the error *in excess of that unavoidable rounding*:

    |O_gpu - O_ref| <= |bf16(O_ref) - O_ref| + 1e-2      for every element,

i.e. the kernel's output is never more than 1e-2 worse than the best possible
bf16 output.  The plain max |dO| is reported beside it.
"""
from __future__ import annotations

import numpy as np
import torch

TOL_O = 1e-2
TOL_LSE = 1e-3


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values to the nearest bf16 value (ties to even), exactly, in fp64."""
    x = np.asarray(x, np.float64)
    out = np.zeros_like(x)
    nz = x != 0
    e = np.floor(np.log2(np.abs(x[nz])))
    spacing = np.exp2(e - 7.0)  # bf16 keeps 8 significant bits
    out[nz] = np.round(x[nz] / spacing) * spacing
    return out


def compare(o_gpu: torch.Tensor, lse_gpu: torch.Tensor, o_ref: np.ndarray, lse_ref: np.ndarray) -> dict:
    """Check element by element; return the statistics (raise AssertionError on a violation)."""
    o = o_gpu.detach().cpu().float().numpy().astype(np.float64).reshape(o_ref.shape)
    lse = lse_gpu.detach().cpu().numpy().astype(np.float64).reshape(lse_ref.shape)
    assert np.all(np.isfinite(o)), "non-finite O"
    d = np.abs(o - o_ref)
    floor = np.abs(round_to_bf16(o_ref) - o_ref)
    excess = d - floor
    stats = {
        "max_abs_dO": float(d.max()) if d.size else 0.0,
        "max_excess_dO": float(excess.max()) if d.size else 0.0,
    }
    bad = excess > TOL_O
    if np.any(bad):
        idx = np.unravel_index(np.argmax(excess), d.shape)
        raise AssertionError(f"O mismatch at {idx}: gpu {o[idx]} ref {o_ref[idx]} (excess {excess[idx]:.4g} over the "
                             f"bf16 rounding floor; {int(bad.sum())} of {bad.size} elements out of bound)")
    dead = np.isneginf(lse_ref)
    assert np.all(np.isneginf(lse[dead])), "rows without keys must have LSE = -inf"
    assert np.all(np.isfinite(lse[~dead])), "non-finite LSE on a row with keys"
    assert np.all(o[dead] == 0.0), "rows without keys must be 0"
    dl = np.abs(lse[~dead] - lse_ref[~dead])
    stats["max_abs_dLSE"] = float(dl.max()) if dl.size else 0.0
    assert stats["max_abs_dLSE"] <= TOL_LSE, f"LSE mismatch: {stats['max_abs_dLSE']}"
    return stats
