"""ctypes binding of libikbo.so (include/ikbo.h), same names as the C ABI.

Argument marshalling only: torch tensors are checked for device, dtype and
contiguity, their shapes become the C size arguments and their data
pointers the C pointers.  Every step of the hot path runs in the library's
CUDA kernels.  If the library is missing this module raises; there is no
fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libikbo.so")

STATUS_NAMES = {0: "IKBO_OK", 1: "IKBO_ERR_INVALID_ARG", 2: "IKBO_ERR_UNSUPPORTED", 3: "IKBO_ERR_CUDA",
                4: "IKBO_ERR_MAP_OUT_OF_RANGE", 5: "IKBO_ERR_TIMEOUT", 6: "IKBO_ERR_NOT_PLANNED",
                7: "IKBO_ERR_INTERNAL"}
IKBO_OK = 0
IKBO_ERR_INVALID_ARG = 1
IKBO_ERR_UNSUPPORTED = 2
IKBO_ERR_CUDA = 3
IKBO_ERR_MAP_OUT_OF_RANGE = 4
IKBO_ERR_TIMEOUT = 5
IKBO_ERR_NOT_PLANNED = 6
IKBO_ERR_INTERNAL = 7
DEBUG_WITHHOLD_USER_PARTIAL = 1
DEBUG_NO_COOPERATIVE = 2

# every function the header declares: name -> (restype, argtypes)
_vp, _i, _u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
SIGNATURES = {
    "ikbo_plan_create": (_i, [ctypes.POINTER(_vp), _i, _i, _i]),
    "ikbo_plan": (_i, [_vp, _vp, _i, _i, _i, _i, _vp]),
    "ikbo_plan_segments": (_i, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_vp)]),
    "ikbo_plan_worklist": (_i, [_vp, ctypes.POINTER(_vp), ctypes.POINTER(_vp), ctypes.POINTER(_i),
                                ctypes.POINTER(_i)]),
    "ikbo_lce_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "ikbo_lce_forward_staged": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "ikbo_lce_forward_noalloc": (_i, [_vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "ikbo_lce_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "ikbo_attn_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, ctypes.c_float, _vp]),
    "ikbo_attn_forward_lse": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, ctypes.c_float, _vp]),
    "ikbo_attn_backward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, ctypes.c_float,
                                _vp]),
    "ikbo_attn_self_target_forward": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, ctypes.c_float, _vp]),
    "ikbo_plan_get_status": (_i, [_vp, _vp]),
    "ikbo_plan_set_debug": (_i, [_vp, ctypes.c_uint]),
    "ikbo_plan_set_timeout_ns": (_i, [_vp, _u64]),
    "ikbo_plan_set_lce_schedule": (_i, [_vp, _i]),
    "ikbo_plan_launch_count": (_u64, [_vp]),
    "ikbo_status_string": (ctypes.c_char_p, [_i]),
    "ikbo_plan_destroy": (None, [_vp]),
    "ikbo_version": (_i, []),
}

_lib = None


class IkboError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")


def load(path: str = LIB_PATH):
    """Load libikbo.so (raises OSError / RuntimeError if it is absent)."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(f"libikbo.so not built ({path}); run "
                               "`python -m broadcast_gemm_attention_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _check(rc: int, what: str):
    if rc != IKBO_OK:
        raise IkboError(rc, what)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


# ---------------------------------------------------------------- the ABI
def ikbo_version() -> int:
    return int(load().ikbo_version())


def ikbo_status_string(code: int) -> str:
    return load().ikbo_status_string(code).decode()


def ikbo_plan_create(max_cand: int, max_users: int, max_heads: int = 1) -> int:
    h = ctypes.c_void_p()
    _check(load().ikbo_plan_create(ctypes.byref(h), max_cand, max_users, max_heads), "ikbo_plan_create")
    return h.value


def ikbo_plan_destroy(plan: int) -> None:
    load().ikbo_plan_destroy(plan)


def ikbo_plan(plan: int, map_: torch.Tensor, n_users: int, H: int = 1, Lq: int = 8, stream=None) -> None:
    ptr = _dev(map_, torch.int32, "map")
    _check(load().ikbo_plan(plan, ptr, map_.numel(), n_users, H, Lq, _stream(stream)), "ikbo_plan")


def ikbo_plan_segments(plan: int):
    """(counts_ptr, offsets_ptr, perm_ptr) device addresses (borrowed)."""
    c, o, p = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
    _check(load().ikbo_plan_segments(plan, ctypes.byref(c), ctypes.byref(o), ctypes.byref(p)), "ikbo_plan_segments")
    return c.value, o.value, p.value


def ikbo_plan_worklist(plan: int):
    """(work_ptr, n_units_ptr, cands_per_unit, max_units)."""
    w, n = ctypes.c_void_p(), ctypes.c_void_p()
    cpu, mu = ctypes.c_int(), ctypes.c_int()
    _check(load().ikbo_plan_worklist(plan, ctypes.byref(w), ctypes.byref(n), ctypes.byref(cpu), ctypes.byref(mu)),
           "ikbo_plan_worklist")
    return w.value, n.value, cpu.value, mu.value


def ikbo_lce_forward(plan: int, U: torch.Tensor, C: torch.Tensor, Wu: torch.Tensor, Wc: torch.Tensor,
                     b: Optional[torch.Tensor], Y: torch.Tensor, stream=None) -> None:
    """Y[i] = Wu^T U[map[i]] + Wc^T C[i] + b for the planned request."""
    bf = torch.bfloat16
    n_users, K_u, D = U.shape
    n_cand, K_c, D2 = C.shape
    N = Wu.shape[1]
    if D2 != D or tuple(Wu.shape) != (K_u, N) or tuple(Wc.shape) != (K_c, N) or tuple(Y.shape) != (n_cand, N, D):
        raise ValueError("inconsistent LCE shapes")
    bptr = None
    if b is not None:
        if tuple(b.shape) != (N,):
            raise ValueError("b must be [N]")
        bptr = _dev(b, bf, "b")
    _check(load().ikbo_lce_forward(plan, _dev(U, bf, "U"), _dev(C, bf, "C"), _dev(Wu, bf, "Wu"), _dev(Wc, bf, "Wc"),
                                   bptr, _dev(Y, bf, "Y"), K_u, K_c, D, N, _stream(stream)), "ikbo_lce_forward")


def ikbo_lce_backward(plan: int, U: torch.Tensor, C: torch.Tensor, Wu: torch.Tensor, Wc: torch.Tensor,
                      dY: torch.Tensor, dU: Optional[torch.Tensor], dC: Optional[torch.Tensor],
                      dWu: Optional[torch.Tensor], dWc: Optional[torch.Tensor], db: Optional[torch.Tensor],
                      stream=None) -> None:
    """Gradients of the LCE for upstream dY (any output may be None to skip it):
    dU/dC bf16, dWu/dWc/db fp32, all overwritten."""
    bf, f32 = torch.bfloat16, torch.float32
    n_users, K_u, D = U.shape
    n_cand, K_c, D2 = C.shape
    N = Wu.shape[1]
    if D2 != D or tuple(Wu.shape) != (K_u, N) or tuple(Wc.shape) != (K_c, N) or tuple(dY.shape) != (n_cand, N, D):
        raise ValueError("inconsistent LCE shapes")
    want = {"dU": (dU, (n_users, K_u, D), bf), "dC": (dC, (n_cand, K_c, D), bf), "dWu": (dWu, (K_u, N), f32),
            "dWc": (dWc, (K_c, N), f32), "db": (db, (N,), f32)}
    ptrs = {}
    for name, (t, shape, dt) in want.items():
        if t is None:
            ptrs[name] = None
            continue
        if tuple(t.shape) != shape:
            raise ValueError(f"{name} must be {list(shape)}")
        ptrs[name] = _dev(t, dt, name)
    _check(load().ikbo_lce_backward(plan, _dev(U, bf, "U"), _dev(C, bf, "C"), _dev(Wu, bf, "Wu"), _dev(Wc, bf, "Wc"),
                                    _dev(dY, bf, "dY"), ptrs["dU"], ptrs["dC"], ptrs["dWu"], ptrs["dWc"], ptrs["db"],
                                    K_u, K_c, D, N, _stream(stream)), "ikbo_lce_backward")


def ikbo_lce_forward_staged(plan: int, U: torch.Tensor, C: torch.Tensor, Wu: torch.Tensor, Wc: torch.Tensor,
                            b: Optional[torch.Tensor], Y: torch.Tensor, stage: int, stream=None) -> None:
    """The LCE as stage 1 (decomposed, unfused), 3 (fused epilogue, one
    accumulator) or 4 (the full kernel) of the pages' stage ladder."""
    bf = torch.bfloat16
    n_users, K_u, D = U.shape
    n_cand, K_c, D2 = C.shape
    N = Wu.shape[1]
    if D2 != D or tuple(Wu.shape) != (K_u, N) or tuple(Wc.shape) != (K_c, N) or tuple(Y.shape) != (n_cand, N, D):
        raise ValueError("inconsistent LCE shapes")
    bptr = None if b is None else _dev(b, bf, "b")
    _check(load().ikbo_lce_forward_staged(plan, _dev(U, bf, "U"), _dev(C, bf, "C"), _dev(Wu, bf, "Wu"),
                                          _dev(Wc, bf, "Wc"), bptr, _dev(Y, bf, "Y"), K_u, K_c, D, N, int(stage),
                                          _stream(stream)), "ikbo_lce_forward_staged")


def ikbo_lce_forward_noalloc(map_: torch.Tensor, n_users: int, U: torch.Tensor, C: torch.Tensor,
                             Wu: torch.Tensor, Wc: torch.Tensor, b: Optional[torch.Tensor], Y: torch.Tensor,
                             stream=None) -> None:
    """The fused LCE without a plan: its scratch lives in the library's own
    fixed device array, so the call allocates nothing (for callers whose
    device memory belongs to another allocator).  Calls share that scratch:
    do not overlap them on the GPU."""
    bf = torch.bfloat16
    n_u, K_u, D = U.shape
    n_cand, K_c, D2 = C.shape
    N = Wu.shape[1]
    if n_u != n_users or D2 != D or tuple(Wu.shape) != (K_u, N) or tuple(Wc.shape) != (K_c, N) or \
            tuple(Y.shape) != (n_cand, N, D) or map_.numel() != n_cand:
        raise ValueError("inconsistent LCE shapes")
    bptr = None
    if b is not None:
        if tuple(b.shape) != (N,):
            raise ValueError("b must be [N]")
        bptr = _dev(b, bf, "b")
    _check(load().ikbo_lce_forward_noalloc(_dev(map_, torch.int32, "map"), n_cand, n_users, _dev(U, bf, "U"),
                                           _dev(C, bf, "C"), _dev(Wu, bf, "Wu"), _dev(Wc, bf, "Wc"), bptr,
                                           _dev(Y, bf, "Y"), K_u, K_c, D, N, _stream(stream)),
           "ikbo_lce_forward_noalloc")


def ikbo_attn_forward(plan: int, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                      kv_offsets: Optional[torch.Tensor], O: torch.Tensor, scale: Optional[float] = None,
                      stream=None) -> None:
    """O[i,h] = softmax(Q[i,h] K[map[i],h]^T scale) V[map[i],h] for the planned request."""
    bf = torch.bfloat16
    d = Q.shape[-1]
    if kv_offsets is None:
        Lkv = K.shape[2]
        optr = None
    else:
        Lkv = K.shape[0]
        optr = _dev(kv_offsets, torch.int32, "kv_offsets")
    if K.shape != V.shape or O.shape != Q.shape:
        raise ValueError("inconsistent attention shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(load().ikbo_attn_forward(plan, _dev(Q, bf, "Q"), _dev(K, bf, "K"), _dev(V, bf, "V"), optr,
                                    _dev(O, bf, "O"), Lkv, d, float(scale), _stream(stream)), "ikbo_attn_forward")


def ikbo_attn_forward_lse(plan: int, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor,
                          kv_offsets: Optional[torch.Tensor], O: torch.Tensor, lse: torch.Tensor,
                          scale: Optional[float] = None, stream=None) -> None:
    """ikbo_attn_forward that also writes each query row's natural-log
    log-sum-exp into lse (fp32 [n_cand, H, Lq])."""
    bf = torch.bfloat16
    d = Q.shape[-1]
    if kv_offsets is None:
        Lkv = K.shape[2]
        optr = None
    else:
        Lkv = K.shape[0]
        optr = _dev(kv_offsets, torch.int32, "kv_offsets")
    if K.shape != V.shape or O.shape != Q.shape or tuple(lse.shape) != tuple(Q.shape[:3]):
        raise ValueError("inconsistent attention shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _check(load().ikbo_attn_forward_lse(plan, _dev(Q, bf, "Q"), _dev(K, bf, "K"), _dev(V, bf, "V"), optr,
                                        _dev(O, bf, "O"), _dev(lse, torch.float32, "lse"), Lkv, d, float(scale),
                                        _stream(stream)), "ikbo_attn_forward_lse")


def ikbo_attn_backward(plan: int, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor,
                       dO: torch.Tensor, kv_offsets: Optional[torch.Tensor], dQ: torch.Tensor, dK: torch.Tensor,
                       dV: torch.Tensor, scale: Optional[float] = None, stream=None,
                       lse: Optional[torch.Tensor] = None) -> None:
    """Gradients of broadcast attention for upstream dO: dQ (Q's layout), and dK,
    dV (K's layout) summed over each user's candidates; all bf16, overwritten.
    lse: the forward's log-sum-exp (ikbo_attn_forward_lse), or None."""
    bf = torch.bfloat16
    d = Q.shape[-1]
    if kv_offsets is None:
        Lkv = K.shape[2]
        optr = None
    else:
        Lkv = K.shape[0]
        optr = _dev(kv_offsets, torch.int32, "kv_offsets")
    if K.shape != V.shape or O.shape != Q.shape or dO.shape != Q.shape or dQ.shape != Q.shape or \
            dK.shape != K.shape or dV.shape != V.shape:
        raise ValueError("inconsistent attention shapes")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    lptr = None
    if lse is not None:
        if tuple(lse.shape) != tuple(Q.shape[:3]):
            raise ValueError("inconsistent lse shape")
        lptr = _dev(lse, torch.float32, "lse")
    _check(load().ikbo_attn_backward(plan, _dev(Q, bf, "Q"), _dev(K, bf, "K"), _dev(V, bf, "V"), _dev(O, bf, "O"),
                                     _dev(dO, bf, "dO"), lptr, optr, _dev(dQ, bf, "dQ"), _dev(dK, bf, "dK"),
                                     _dev(dV, bf, "dV"), Lkv, d, float(scale), _stream(stream)),
           "ikbo_attn_backward")


def ikbo_attn_self_target_forward(plan: int, Q: torch.Tensor, Q_user: torch.Tensor, K: torch.Tensor,
                                  V: torch.Tensor, kv_offsets: Optional[torch.Tensor], O: torch.Tensor,
                                  O_user: torch.Tensor, scale: Optional[float] = None, stream=None) -> None:
    """Target attention (as ikbo_attn_forward) and the users' own queries
    O_user[u,h] = softmax(Q_user[u,h] K[u,h]^T scale) V[u,h], in one launch.
    Q and O both None: the self part alone."""
    bf = torch.bfloat16
    d = Q_user.shape[-1]
    if kv_offsets is None:
        Lkv = K.shape[2]
        optr = None
    else:
        Lkv = K.shape[0]
        optr = _dev(kv_offsets, torch.int32, "kv_offsets")
    if (Q is None) != (O is None):
        raise ValueError("Q and O are given together or not at all")
    if K.shape != V.shape or (Q is not None and O.shape != Q.shape) or O_user.shape != Q_user.shape \
            or Q_user.dim() != 4:
        raise ValueError("shape mismatch among Q/O, Q_user/O_user, K/V")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qp = None if Q is None else _dev(Q, bf, "Q")
    op = None if O is None else _dev(O, bf, "O")
    _check(load().ikbo_attn_self_target_forward(plan, qp, _dev(Q_user, bf, "Q_user"), _dev(K, bf, "K"),
                                                _dev(V, bf, "V"), optr, op, _dev(O_user, bf, "O_user"),
                                                Q_user.shape[2], Lkv, d, float(scale), _stream(stream)),
           "ikbo_attn_self_target_forward")


def ikbo_plan_get_status(plan: int, stream=None) -> int:
    """Synchronises the stream; returns the device-detected status code (and clears it)."""
    return int(load().ikbo_plan_get_status(plan, _stream(stream)))


def ikbo_plan_set_debug(plan: int, flags: int) -> None:
    _check(load().ikbo_plan_set_debug(plan, flags), "ikbo_plan_set_debug")


def ikbo_plan_set_lce_schedule(plan: int, schedule: int) -> None:
    """0 = chosen from the shape, 1 = two launches, 2 = one launch."""
    _check(load().ikbo_plan_set_lce_schedule(plan, int(schedule)), "ikbo_plan_set_lce_schedule")


def ikbo_plan_set_timeout_ns(plan: int, ns: int) -> None:
    _check(load().ikbo_plan_set_timeout_ns(plan, ns), "ikbo_plan_set_timeout_ns")


def ikbo_plan_launch_count(plan: int) -> int:
    return int(load().ikbo_plan_launch_count(plan))


# ------------------------------------------------------------ convenience
class Plan:
    """Owns one ikbo_plan_t; `with Plan(...) as p:` destroys it on exit."""

    def __init__(self, max_cand: int, max_users: int, max_heads: int = 1):
        self._map = None
        self.handle = ikbo_plan_create(max_cand, max_users, max_heads)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def close(self):
        if self.handle:
            ikbo_plan_destroy(self.handle)
            self.handle = None
        self._map = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def plan(self, map_, n_users, H=1, Lq=8, stream=None):
        ikbo_plan(self.handle, map_, n_users, H, Lq, stream)
        # the plan borrows the map for every later call of this request: hold
        # the tensor so that a temporary passed here stays allocated
        self._map = map_

    def lce_forward(self, U, C, Wu, Wc, b, Y, stream=None):
        ikbo_lce_forward(self.handle, U, C, Wu, Wc, b, Y, stream)

    def lce_backward(self, U, C, Wu, Wc, dY, dU=None, dC=None, dWu=None, dWc=None, db=None, stream=None):
        ikbo_lce_backward(self.handle, U, C, Wu, Wc, dY, dU, dC, dWu, dWc, db, stream)

    def lce_forward_staged(self, U, C, Wu, Wc, b, Y, stage, stream=None):
        ikbo_lce_forward_staged(self.handle, U, C, Wu, Wc, b, Y, stage, stream)

    def attn_forward(self, Q, K, V, kv_offsets, O, scale=None, stream=None):
        ikbo_attn_forward(self.handle, Q, K, V, kv_offsets, O, scale, stream)

    def attn_forward_lse(self, Q, K, V, kv_offsets, O, lse, scale=None, stream=None):
        ikbo_attn_forward_lse(self.handle, Q, K, V, kv_offsets, O, lse, scale, stream)

    def attn_backward(self, Q, K, V, O, dO, kv_offsets, dQ, dK, dV, scale=None, stream=None, lse=None):
        ikbo_attn_backward(self.handle, Q, K, V, O, dO, kv_offsets, dQ, dK, dV, scale, stream, lse)

    def attn_self_target_forward(self, Q, Q_user, K, V, kv_offsets, O, O_user, scale=None, stream=None):
        ikbo_attn_self_target_forward(self.handle, Q, Q_user, K, V, kv_offsets, O, O_user, scale, stream)

    def status(self, stream=None) -> int:
        return ikbo_plan_get_status(self.handle, stream)

    def set_lce_schedule(self, schedule: int) -> None:
        ikbo_plan_set_lce_schedule(self.handle, schedule)

    def launches(self) -> int:
        return ikbo_plan_launch_count(self.handle)

    def segments(self, n_cand: int, n_users: int):
        """Copies of (counts, offsets, perm) as CPU int32 tensors (synchronises)."""
        c, o, p = ikbo_plan_segments(self.handle)
        return (_copy_i32(c, n_users), _copy_i32(o, n_users + 1), _copy_i32(p, n_cand))

    def worklist(self):
        """Copy of the work list as a CPU int32 tensor [n_units, 4] (synchronises)."""
        w, n, cpu, mu = ikbo_plan_worklist(self.handle)
        n_units = int(_copy_i32(n, 1)[0])
        return _copy_i32(w, 4 * n_units).view(n_units, 4), cpu


class _DeviceArray:
    """Exposes a borrowed device int32 array through __cuda_array_interface__."""

    def __init__(self, ptr: int, count: int):
        self.__cuda_array_interface__ = {"shape": (count,), "typestr": "<i4", "data": (ptr, False),
                                         "version": 3, "strides": None}


def _copy_i32(dev_ptr: int, count: int) -> torch.Tensor:
    """Device int32 array at a borrowed address -> CPU tensor (synchronises)."""
    if count == 0:
        return torch.empty(0, dtype=torch.int32)
    torch.cuda.synchronize()
    return torch.as_tensor(_DeviceArray(dev_ptr, count), device="cuda").cpu().clone()
