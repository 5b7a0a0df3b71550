"""Seeded synthetic inputs for the IKBO hot path.

This module only draws random numbers and arranges them into the tensor
shapes of the workloads; it holds none of the method's arithmetic, so both
the CUDA path and the CPU oracle can consume what it produces.

Workloads follow the candidate/user request shapes that the IKBO write-ups
describe (about 15 users broadcast ~70x onto 1024 candidates; candidate
batches 256-4096 and candidate:user ratios 10:1 to 10000:1, see "Meta
Optimizes Inference for Recommendation Systems" and the zubnet.ai IKBO news
item).  The exact sizes (K_u=381, K_c=243, D=256, N=192; H=8, Lq=32,
Lkv=2048, d=128) are this project's synthetic choice.

Recipe (every config):
  * numpy PCG64 generator seeded with ``1000 + config_index`` (sweep points
    add ``10 * sweep_index``);
  * draw order: the candidate->user map first, then (attention) the jagged
    key/value lengths, then the tensors in the order they are listed;
  * values are drawn in float32 and rounded to bfloat16 (round to nearest
    even, via torch) once; those bf16 values are the single source for both
    the GPU and the oracle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np
import torch


def _bf16(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _normal(rng: np.random.Generator, shape, var: float) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if var != 1.0:
        x *= np.float32(math.sqrt(var))
    return _bf16(x)


def sorted_multinomial_map(rng: np.random.Generator, n_cand: int, n_users: int) -> np.ndarray:
    """Segment sizes ~ Multinomial(n_cand, uniform over users); map sorted ascending."""
    counts = rng.multinomial(n_cand, np.full(n_users, 1.0 / n_users))
    return np.repeat(np.arange(n_users, dtype=np.int32), counts).astype(np.int32)


def permuted_multinomial_map(rng: np.random.Generator, n_cand: int, n_users: int) -> np.ndarray:
    m = sorted_multinomial_map(rng, n_cand, n_users)
    return m[rng.permutation(n_cand)].astype(np.int32)


def zipf_permuted_map(rng: np.random.Generator, n_cand: int, n_users: int, s: float) -> np.ndarray:
    """Counts ~ Multinomial(n_cand, p_r ~ r^-s), user u has rank u+1; then permuted."""
    r = np.arange(1, n_users + 1, dtype=np.float64)
    p = r ** (-s)
    p /= p.sum()
    counts = rng.multinomial(n_cand, p)
    m = np.repeat(np.arange(n_users, dtype=np.int32), counts)
    return m[rng.permutation(n_cand)].astype(np.int32)


@dataclass
class LCEInputs:
    name: str
    n_cand: int
    n_users: int
    K_u: int
    K_c: int
    D: int
    N: int
    map: torch.Tensor          # int32 [n_cand]
    U: torch.Tensor            # bf16 [n_users, K_u, D]
    C: torch.Tensor            # bf16 [n_cand, K_c, D]
    Wu: torch.Tensor           # bf16 [K_u, N]
    Wc: torch.Tensor           # bf16 [K_c, N]
    b: Optional[torch.Tensor]  # bf16 [N]

    def tensors(self) -> Dict[str, torch.Tensor]:
        d = dict(map=self.map, U=self.U, C=self.C, Wu=self.Wu, Wc=self.Wc)
        if self.b is not None:
            d["b"] = self.b
        return d


@dataclass
class AttnInputs:
    name: str
    n_cand: int
    n_users: int
    H: int
    Lq: int
    Lkv: int                          # dense per-user length, or total packed rows if jagged
    d: int
    map: torch.Tensor                 # int32 [n_cand]
    Q: torch.Tensor                   # bf16 [n_cand, H, Lq, d]
    K: torch.Tensor                   # bf16 [n_users, H, Lkv, d] or [sum L, H, d]
    V: torch.Tensor
    kv_offsets: Optional[torch.Tensor] = None   # int32 [n_users + 1] when jagged

    @property
    def jagged(self) -> bool:
        return self.kv_offsets is not None

    def kv_len(self, u: int) -> int:
        if self.kv_offsets is None:
            return self.Lkv
        return int(self.kv_offsets[u + 1] - self.kv_offsets[u])


def make_lce(name: str, seed: int, n_cand: int, n_users: int, K_u: int, K_c: int, D: int, N: int,
             map_kind: str = "sorted", explicit_map: Optional[List[int]] = None,
             bias: bool = True, w_var: Optional[float] = None) -> LCEInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    if explicit_map is not None:
        m = np.asarray(explicit_map, dtype=np.int32)
    elif map_kind == "sorted":
        m = sorted_multinomial_map(rng, n_cand, n_users)
    elif map_kind == "permuted":
        m = permuted_multinomial_map(rng, n_cand, n_users)
    else:
        raise ValueError(map_kind)
    if w_var is None:
        w_var = 1.0 / max(1, K_u + K_c)
    U = _normal(rng, (n_users, K_u, D), 1.0)
    C = _normal(rng, (n_cand, K_c, D), 1.0)
    Wu = _normal(rng, (K_u, N), w_var)
    Wc = _normal(rng, (K_c, N), w_var)
    b = _normal(rng, (N,), 0.01) if bias else None
    return LCEInputs(name, n_cand, n_users, K_u, K_c, D, N, torch.from_numpy(m), U, C, Wu, Wc, b)


def make_attn(name: str, seed: int, n_cand: int, n_users: int, H: int, Lq: int, d: int,
              Lkv: Optional[int] = None, jagged_range: Optional[tuple] = None,
              map_kind: str = "sorted", zipf_s: float = 1.1,
              explicit_map: Optional[List[int]] = None,
              explicit_lengths: Optional[List[int]] = None) -> AttnInputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    if explicit_map is not None:
        m = np.asarray(explicit_map, dtype=np.int32)
    elif map_kind == "sorted":
        m = sorted_multinomial_map(rng, n_cand, n_users)
    elif map_kind == "permuted":
        m = permuted_multinomial_map(rng, n_cand, n_users)
    elif map_kind == "zipf":
        m = zipf_permuted_map(rng, n_cand, n_users, zipf_s)
    else:
        raise ValueError(map_kind)
    kv_offsets = None
    if explicit_lengths is not None or jagged_range is not None:
        if explicit_lengths is not None:
            L = np.asarray(explicit_lengths, dtype=np.int64)
        else:
            lo, hi = jagged_range
            L = rng.integers(lo, hi + 1, size=n_users)
        offs = np.zeros(n_users + 1, dtype=np.int64)
        offs[1:] = np.cumsum(L)
        total = int(offs[-1])
        kv_offsets = torch.from_numpy(offs.astype(np.int32))
        Q = _normal(rng, (n_cand, H, Lq, d), 1.0)
        K = _normal(rng, (total, H, d), 1.0)
        V = _normal(rng, (total, H, d), 1.0)
        Lkv_out = total
    else:
        assert Lkv is not None
        Q = _normal(rng, (n_cand, H, Lq, d), 1.0)
        K = _normal(rng, (n_users, H, Lkv, d), 1.0)
        V = _normal(rng, (n_users, H, Lkv, d), 1.0)
        Lkv_out = Lkv
    return AttnInputs(name, n_cand, n_users, H, Lq, Lkv_out, d, torch.from_numpy(m), Q, K, V, kv_offsets)


def make_user_queries(seed: int, n_users: int, H: int, Lq_u: int, d: int) -> torch.Tensor:
    """The users' own query set Q_user [n_users, H, Lq_u, d], bf16 N(0, 1), for
    self + target attention (its own seed, drawn after nothing else)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _normal(rng, (n_users, H, Lq_u, d), 1.0)


# --------------------------------------------------------------------------
# The named workloads.
# --------------------------------------------------------------------------

LCE_TINY = dict(n_cand=16, n_users=2, K_u=24, K_c=16, D=32, N=8)
LCE_70 = dict(n_cand=1024, n_users=15, K_u=381, K_c=243, D=256, N=192)
ATTN_70 = dict(n_cand=1024, n_users=15, H=8, Lq=32, d=128, Lkv=2048)
ATTN_STRESS = dict(n_cand=4096, n_users=64, H=8, Lq=16, d=128)
SWEEP_N_CAND = (256, 1024, 4096)
SWEEP_RATIO = (10, 70, 1000, 10000)


def lce_tiny() -> LCEInputs:
    """LCE tiny: 16 candidates, 2 users, map [0]*8 + [1]*8."""
    return make_lce("lce_tiny", 1000, explicit_map=[0] * 8 + [1] * 8, **LCE_TINY)


def lce_70to1() -> LCEInputs:
    """LCE at the 70:1 request shape (1024 candidates, 15 users)."""
    return make_lce("lce_70to1", 1001, **LCE_70)


def sweep_users(n_cand: int, ratio: int) -> int:
    return max(1, int(round(n_cand / ratio)))


def lce_sweep_points():
    """(n_cand, ratio, seed) for the LCE shape sweep."""
    pts = []
    k = 0
    for n in SWEEP_N_CAND:
        for r in SWEEP_RATIO:
            pts.append((n, r, 1002 + 10 * k))
            k += 1
    return pts


def lce_sweep(n_cand: int, ratio: int, seed: int) -> LCEInputs:
    return make_lce(f"lce_sweep_{n_cand}_{ratio}", seed, n_cand=n_cand,
                    n_users=sweep_users(n_cand, ratio), K_u=381, K_c=243, D=256, N=192)


def lce_70to1_map() -> torch.Tensor:
    """The 70:1 candidate->user map alone (the first draw of the LCE 70:1 seed)."""
    rng = np.random.Generator(np.random.PCG64(1001))
    return torch.from_numpy(sorted_multinomial_map(rng, LCE_70["n_cand"], LCE_70["n_users"]))


def attn_70to1() -> AttnInputs:
    """Broadcast attention at 70:1; it shares the LCE 70:1 request's map."""
    return make_attn("attn_70to1", 1003, explicit_map=lce_70to1_map().tolist(), **ATTN_70)


def attn_stress() -> AttnInputs:
    """4096 candidates, 64 users, Zipf(1.1) counts, permuted map, jagged Lkv ~ U[256, 4096]."""
    return make_attn("attn_stress", 1004, map_kind="zipf", zipf_s=1.1,
                     jagged_range=(256, 4096), **ATTN_STRESS)


def attn_ratio_sweep_points():
    return [(4096, r, 1004 + 10 * (k + 1)) for k, r in enumerate(SWEEP_RATIO)]


def attn_ratio_sweep(n_cand: int, ratio: int, seed: int) -> AttnInputs:
    return make_attn(f"attn_sweep_{n_cand}_{ratio}", seed, n_cand=n_cand,
                     n_users=sweep_users(n_cand, ratio), H=8, Lq=16, d=128, Lkv=2048,
                     map_kind="permuted")


def make_lce_grad(seed: int, n_cand: int, N: int, D: int) -> torch.Tensor:
    """Upstream gradient dY = dL/dY for the LCE backward: bf16 [n_cand, N, D]
    ~ N(0, 1), from its own PCG64 stream (seed + 500, so it never repeats the
    forward inputs' draws)."""
    rng = np.random.Generator(np.random.PCG64(seed + 500))
    return _normal(rng, (n_cand, N, D), 1.0)


def make_attn_grad(seed: int, shape) -> torch.Tensor:
    """Upstream gradient dO = dL/dO for the attention backward: bf16 of the
    given shape ~ N(0, 1), from its own PCG64 stream (seed + 700)."""
    rng = np.random.Generator(np.random.PCG64(seed + 700))
    return _normal(rng, tuple(shape), 1.0)
