"""Helpers shared by the GPU parity tests (not collected by pytest)."""
from __future__ import annotations

from collections import OrderedDict

import numpy as np
import torch

import oracle

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
    bad = ~(err <= bound)  # NaN counts as out of tolerance
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"LCE mismatch {what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"max err {np.nanmax(err):.4g}; first {idx}; gpu {g[tuple(idx[0])]:.6g} "
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


# ------------------------------------------------------------------ whole-output checks
# Full-size workloads are compared element by element against the oracle,
# which is computed here, in this session, on the host cores (never stored).
# The oracle runs over slices of candidates so that no more than a few
# hundred MB of fp64 reference is alive at a time; a named workload's slices
# may be kept for the next test that runs the same inputs (a small LRU).
_CACHE: "OrderedDict[tuple, object]" = OrderedDict()
_CACHE_ENTRIES = 6


def cached(key, fn):
    """fn() memoised under key (key must identify the inputs exactly)."""
    if key is None:
        return fn()
    if key in _CACHE:
        _CACHE.move_to_end(key)
        return _CACHE[key]
    val = fn()
    _CACHE[key] = val
    while len(_CACHE) > _CACHE_ENTRIES:
        _CACHE.popitem(last=False)
    return val


def _slices(n: int, chunk: int):
    return [(a, min(n, a + chunk)) for a in range(0, n, chunk)]


def check_lce_all(Y: torch.Tensor, x, bias: bool = True, what: str = "", chunk: int = 512,
                  cache_key=None) -> float:
    """Every element of Y [n_cand, N, D] against the oracle's materialised LCE."""
    worst = 0.0
    b = x.b if bias else None
    for a, e in _slices(x.n_cand, chunk):
        key = None if cache_key is None else (cache_key, "lce", bias, a, e)
        ref = cached(key, lambda: oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, b, cands=list(range(a, e))))
        worst = max(worst, assert_lce_close(Y[a:e], ref, f"{what or x.name} candidates {a}..{e - 1}"))
    return worst


def check_attn_all(O: torch.Tensor, x, scale=None, what: str = "", chunk: int = 256, cache_key=None) -> float:
    """Every (candidate, head) of O [n_cand, H, Lq, d] against the oracle's attention."""
    worst = 0.0
    offs = x.kv_offsets if x.jagged else None
    for a, e in _slices(x.n_cand, chunk):
        pairs = [(i, h) for i in range(a, e) for h in range(x.H)]
        key = None if cache_key is None else (cache_key, "attn", scale, a, e)
        ref = cached(key, lambda: oracle.attn(x.map, x.Q, x.K, x.V, kv_offsets=offs, n_users=x.n_users,
                                              scale=scale, pairs=pairs))
        ref = ref.reshape(e - a, x.H, x.Lq, x.d)
        worst = max(worst, assert_attn_close(O[a:e], ref, f"{what or x.name} candidates {a}..{e - 1}"))
    return worst


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
