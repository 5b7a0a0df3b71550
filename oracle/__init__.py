"""CPU oracle for the IKBO hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product (``broadcast_gemm_attention_gb300``)
never imports it and has no CPU fallback.

The arithmetic lives in ``ikbo_oracle.c`` (plain C, double precision, the
materialised-broadcast definition); this module compiles it with gcc and
marshals numpy/torch arrays to it.  It shares no code with the CUDA path.

Parity status per function (the pins are in ``tests/test_oracle_*.py``):
  * ``segments``  -- pinned: brute force against numpy's stable argsort,
    invariants, special cases (sorted map, single user);
  * ``lce``       -- pinned: the K-axis decomposition identity, exact
    rational brute force on tiny inputs, special cases that reduce to a
    library matmul, permutation and zero-padding invariance;
  * ``lce_backward`` -- pinned: the adjoint identity <dY, Y(x + dx) - Y(x)>
    = <grad, dx> against the (separately pinned) forward for each input,
    torch fp64 autograd on small cases, closed forms (dY = 0, dY = 1, one
    user), and invariance under candidate permutation;
  * ``attn_backward`` -- pinned: torch fp64 autograd through softmax
    attention on K/V gathered by the map (the gather's own backward sums
    over each user's candidates), closed forms (dO = 0; one key; constant V;
    sum over keys of dV), candidate permutation, selections, jagged slices;
  * ``attn``      -- pinned: identity map equals torch fp64 SDPA, one user
    equals multi-query SDPA, closed forms (Q=0, constant V, one key, one
    dominant score, empty key range), permutation invariance, jagged slices
    equal per-user SDPA.
``tests/test_oracle_mutations.py`` plants mistakes in copies of the C source
and checks that the pins catch each one.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from typing import Optional, Sequence

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ikbo_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libikbo_oracle.so")

STATUS = {0: "ok", 1: "bad argument", 2: "map value out of range", 3: "out of memory",
          4: "work list overflow"}


class OracleError(RuntimeError):
    pass


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -fopenmp (no fast-math: IEEE double semantics are kept)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/libikbo_oracle.so``."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> its uint16 bit patterns (no arithmetic)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _i32(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """One loaded build of the C oracle."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        p, i = ctypes.c_void_p, ctypes.c_int
        lib.ikbo_oracle_segments.argtypes = [p, i, i, i, i, p, p, p, p, ctypes.c_int64, p]
        lib.ikbo_oracle_lce.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, p, i, p, i]
        lib.ikbo_oracle_attn.argtypes = [p, p, p, p, p, i, i, i, i, i, i, ctypes.c_double, p, i, p, i]
        lib.ikbo_oracle_lce_backward.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, p, i, p, i, i,
                                                 p, p, p, p, p, i]
        lib.ikbo_oracle_attn_backward.argtypes = [p, p, p, p, p, p, i, i, i, i, i, i, ctypes.c_double, p, i, p, i,
                                                  p, p, p, i]
        lib.ikbo_oracle_attn_lse.argtypes = [p, p, p, p, i, i, i, i, i, i, ctypes.c_double, p, i, p, i]
        lib.ikbo_oracle_max_threads.argtypes = []
        for f in (lib.ikbo_oracle_segments, lib.ikbo_oracle_lce, lib.ikbo_oracle_attn,
                  lib.ikbo_oracle_lce_backward, lib.ikbo_oracle_attn_backward, lib.ikbo_oracle_attn_lse,
                  lib.ikbo_oracle_max_threads):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    @staticmethod
    def _check(rc: int, what: str):
        if rc != 0:
            raise OracleError(f"{what}: {STATUS.get(rc, rc)}")

    def max_threads(self) -> int:
        return int(self.lib.ikbo_oracle_max_threads())

    def segments(self, map_, n_users: int, H: int = 1, cands_per_unit: int = 1):
        """Stable grouping of candidates by user plus the attention work list.

        Returns (counts[n_users], offsets[n_users+1], perm[n_cand], work[n_units, 4]).
        """
        m = _i32(map_)
        n_cand = m.shape[0]
        counts = np.zeros(n_users, np.int32)
        offsets = np.zeros(n_users + 1, np.int32)
        perm = np.zeros(max(n_cand, 1), np.int32)
        max_units = H * (n_users + n_cand) + 1
        work = np.zeros((max_units, 4), np.int32)
        n_units = ctypes.c_int64(0)
        rc = self.lib.ikbo_oracle_segments(_ptr(m), n_cand, n_users, H, cands_per_unit,
                                           _ptr(counts), _ptr(offsets), _ptr(perm), _ptr(work),
                                           max_units, ctypes.byref(n_units))
        self._check(rc, "segments")
        return counts, offsets, perm[:n_cand], work[: n_units.value].copy()

    def lce(self, map_, U, C, Wu, Wc, b=None, cands: Optional[Sequence[int]] = None,
            n_threads: int = 0) -> np.ndarray:
        """Materialised LCE in fp64: Y[s] = b + [Wu;Wc]^T [U[map[i]]; C[i]], i = cands[s].

        Returns float64 [n_sel, N, D].
        """
        m = _i32(map_)
        n_users, K_u, D = U.shape
        n_cand, K_c, D2 = C.shape
        N = Wu.shape[1]
        assert D2 == D and tuple(Wc.shape) == (K_c, N) and tuple(Wu.shape) == (K_u, N)
        Ub, Cb, Wub, Wcb = _bits(U), _bits(C), _bits(Wu), _bits(Wc)
        bb = _bits(b) if b is not None else None
        sel = None if cands is None else _i32(cands)
        n_sel = n_cand if sel is None else sel.shape[0]
        Y = np.zeros((n_sel, N, D), np.float64)
        rc = self.lib.ikbo_oracle_lce(_ptr(m), _ptr(Ub), _ptr(Cb), _ptr(Wub), _ptr(Wcb), _ptr(bb),
                                      n_cand, n_users, K_u, K_c, D, N, _ptr(sel), n_sel, _ptr(Y),
                                      n_threads)
        self._check(rc, "lce")
        return Y

    def lce_backward(self, map_, U, C, Wu, Wc, dY, cands: Optional[Sequence[int]] = None,
                     users: Optional[Sequence[int]] = None, weights: bool = True, n_threads: int = 0) -> dict:
        """Gradients of the materialised LCE in fp64 for upstream gradient dY [n_cand, N, D]:
        dC [n_csel, K_c, D] for ``cands`` (all when None), dU [n_usel, K_u, D] for
        ``users`` (all when None), and, when ``weights``, dWu [K_u, N], dWc [K_c, N],
        db [N].  Returns a dict of float64 arrays.
        """
        m = _i32(map_)
        n_users, K_u, D = U.shape
        n_cand, K_c, D2 = C.shape
        N = Wu.shape[1]
        assert D2 == D and tuple(Wc.shape) == (K_c, N) and tuple(Wu.shape) == (K_u, N)
        assert tuple(dY.shape) == (n_cand, N, D)
        csel = None if cands is None else _i32(cands)
        usel = None if users is None else _i32(users)
        n_csel = n_cand if csel is None else csel.shape[0]
        n_usel = n_users if usel is None else usel.shape[0]
        out = {"dC": np.zeros((n_csel, K_c, D), np.float64), "dU": np.zeros((n_usel, K_u, D), np.float64),
               "dWu": np.zeros((K_u, N), np.float64), "dWc": np.zeros((K_c, N), np.float64),
               "db": np.zeros((N,), np.float64)}
        rc = self.lib.ikbo_oracle_lce_backward(
            _ptr(m), _ptr(_bits(U)), _ptr(_bits(C)), _ptr(_bits(Wu)), _ptr(_bits(Wc)), _ptr(_bits(dY)),
            n_cand, n_users, K_u, K_c, D, N, _ptr(csel), n_csel, _ptr(usel), n_usel, 1 if weights else 0,
            _ptr(out["dC"]), _ptr(out["dU"]), _ptr(out["dWu"]), _ptr(out["dWc"]), _ptr(out["db"]), n_threads)
        self._check(rc, "lce_backward")
        if not weights:
            for k in ("dWu", "dWc", "db"):
                out.pop(k)
        return out

    def attn_backward(self, map_, Q, K, V, dO, kv_offsets=None, n_users: Optional[int] = None,
                      scale: Optional[float] = None, qpairs: Optional[Sequence] = None,
                      kvpairs: Optional[Sequence] = None, n_threads: int = 0) -> dict:
        """Gradients of broadcast attention in fp64 for upstream dO [n_cand, H, Lq, d]:
        dQ [n_qsel, Lq, d] for the (i, h) ``qpairs`` (all when None); dK, dV
        [n_kvsel, max_len, d] for the (u, h) ``kvpairs`` (all when None), summed
        over every candidate of u; rows past a user's key count are 0."""
        m = _i32(map_)
        n_cand, H, Lq, d = Q.shape
        assert tuple(dO.shape) == tuple(Q.shape)
        if kv_offsets is None:
            n_users_k, H2, Lkv, d2 = K.shape
            if n_users is None:
                n_users = n_users_k
            offs = None
            max_len = Lkv
        else:
            offs = _i32(kv_offsets)
            Lkv, H2, d2 = K.shape
            if n_users is None:
                n_users = offs.shape[0] - 1
            max_len = int(np.max(np.diff(offs))) if n_users > 0 else 0
        assert H2 == H and d2 == d and V.shape == K.shape
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        qs = None if qpairs is None else _i32(qpairs).reshape(-1, 2)
        ks = None if kvpairs is None else _i32(kvpairs).reshape(-1, 2)
        n_q = n_cand * H if qs is None else qs.shape[0]
        n_kv = n_users * H if ks is None else ks.shape[0]
        out = {"dQ": np.zeros((n_q, Lq, d), np.float64), "dK": np.zeros((n_kv, max(max_len, 0), d), np.float64),
               "dV": np.zeros((n_kv, max(max_len, 0), d), np.float64)}
        rc = self.lib.ikbo_oracle_attn_backward(
            _ptr(m), _ptr(_bits(Q)), _ptr(_bits(K)), _ptr(_bits(V)), _ptr(_bits(dO)), _ptr(offs), n_cand, n_users,
            H, Lq, Lkv, d, float(scale), _ptr(qs), n_q, _ptr(ks), n_kv, _ptr(out["dQ"]), _ptr(out["dK"]),
            _ptr(out["dV"]), n_threads)
        self._check(rc, "attn_backward")
        return out

    def attn(self, map_, Q, K, V, kv_offsets=None, n_users: Optional[int] = None,
             scale: Optional[float] = None, pairs: Optional[Sequence] = None,
             n_threads: int = 0) -> np.ndarray:
        """Softmax attention in fp64 with K/V taken from each candidate's user.

        Dense: K, V [n_users, H, Lkv, d]; jagged: K, V [total, H, d] with
        kv_offsets int32 [n_users+1].  Returns float64 [n_sel, Lq, d] for the
        (i, h) pairs (all pairs in (i, h) order when ``pairs`` is None).
        """
        m = _i32(map_)
        n_cand, H, Lq, d = Q.shape
        if kv_offsets is None:
            n_users_k, H2, Lkv, d2 = K.shape
            if n_users is None:
                n_users = n_users_k
            offs = None
        else:
            offs = _i32(kv_offsets)
            Lkv, H2, d2 = K.shape
            if n_users is None:
                n_users = offs.shape[0] - 1
        assert H2 == H and d2 == d and V.shape == K.shape
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        sel = None if pairs is None else _i32(pairs).reshape(-1, 2)
        n_sel = n_cand * H if sel is None else sel.shape[0]
        O = np.zeros((n_sel, Lq, d), np.float64)
        rc = self.lib.ikbo_oracle_attn(_ptr(m), _ptr(_bits(Q)), _ptr(_bits(K)), _ptr(_bits(V)),
                                       _ptr(offs), n_cand, n_users, H, Lq, Lkv, d, float(scale),
                                       _ptr(sel), n_sel, _ptr(O), n_threads)
        self._check(rc, "attn")
        return O

    def attn_lse(self, map_, Q, K, kv_offsets=None, n_users: Optional[int] = None,
                 scale: Optional[float] = None, pairs: Optional[Sequence] = None,
                 n_threads: int = 0) -> np.ndarray:
        """Natural-log log-sum-exp of each query row's scores against its user's
        keys, float64 [n_sel, Lq] for the (i, h) pairs (all when None); -inf
        for an empty key range."""
        m = _i32(map_)
        n_cand, H, Lq, d = Q.shape
        if kv_offsets is None:
            n_users_k, H2, Lkv, d2 = K.shape
            if n_users is None:
                n_users = n_users_k
            offs = None
        else:
            offs = _i32(kv_offsets)
            Lkv, H2, d2 = K.shape
            if n_users is None:
                n_users = offs.shape[0] - 1
        assert H2 == H and d2 == d
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        sel = None if pairs is None else _i32(pairs).reshape(-1, 2)
        n_sel = n_cand * H if sel is None else sel.shape[0]
        out = np.zeros((n_sel, Lq), np.float64)
        rc = self.lib.ikbo_oracle_attn_lse(_ptr(m), _ptr(_bits(Q)), _ptr(_bits(K)), _ptr(offs), n_cand, n_users,
                                           H, Lq, Lkv, d, float(scale), _ptr(sel), n_sel, _ptr(out), n_threads)
        self._check(rc, "attn_lse")
        return out


_default: Optional[Oracle] = None
_lock = threading.Lock()


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def segments(*a, **k):
    return default().segments(*a, **k)


def lce(*a, **k):
    return default().lce(*a, **k)


def attn(*a, **k):
    return default().attn(*a, **k)


def lce_backward(*a, **k):
    return default().lce_backward(*a, **k)


def attn_backward(*a, **k):
    return default().attn_backward(*a, **k)


def attn_lse(*a, **k):
    return default().attn_lse(*a, **k)


def max_threads() -> int:
    return default().max_threads()
