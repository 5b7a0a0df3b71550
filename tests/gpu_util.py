"""Helpers shared by the GPU parity tests (not collected by pytest)."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances fixed by the task's parity bar for floating point:
#   LCE:        |Y_gpu - Y_ref| <= 1e-2 * (1 + |Y_ref|)   element-wise
#   attention:  |O_gpu - O_ref| <= 2e-2                    element-wise
LCE_RTOL = 1e-2
ATTN_ATOL = 2e-2


def to_dev(*ts):
    return [None if t is None else t.cuda() for t in ts]


def assert_lce_close(y_gpu: torch.Tensor, y_ref: np.ndarray, what: str = ""):
    g = y_gpu.detach().to(torch.float64).cpu().numpy()
    err = np.abs(g - y_ref)
    bound = LCE_RTOL * (1.0 + np.abs(y_ref))
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"LCE mismatch {what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"max err {err.max():.4g}; first {idx}; gpu {g[tuple(idx[0])]:.6g} "
                             f"ref {y_ref[tuple(idx[0])]:.6g}")
    return float(err.max())


def assert_attn_close(o_gpu: torch.Tensor, o_ref: np.ndarray, what: str = ""):
    g = o_gpu.detach().to(torch.float64).cpu().numpy()
    err = np.abs(g - o_ref)
    if not np.all(np.isfinite(g)) or err.max() > ATTN_ATOL:
        bad = ~(err <= ATTN_ATOL)
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"attention mismatch {what}: {bad.sum()} of {bad.size} out of tolerance; "
                             f"max err {np.nanmax(err):.4g}; first {idx}")
    return float(err.max())


def sample_candidates(map_: torch.Tensor, n: int, seed: int = 0):
    """First and last candidate of every user segment plus random ones."""
    m = map_.numpy()
    picks = set()
    for u in np.unique(m):
        idx = np.nonzero(m == u)[0]
        picks.add(int(idx[0]))
        picks.add(int(idx[-1]))
    rng = np.random.default_rng(seed)
    picks.update(int(x) for x in rng.choice(len(m), size=min(n, len(m)), replace=False))
    return sorted(picks)
