"""Broadcast attention backward (ikbo_attn_backward) against the fp64
oracle's backward.

Tolerance, from the arithmetic: P and dS are rounded to bf16 before the
tensor cores (2^-9 relative per product term), the outputs are bf16 (2^-9
relative), and the forward O that D = rowsum(dO * O) reads is the GPU's own
bf16 output; so errors scale with the size of the gradient tensor itself:
|g - ref| <= 2e-2 * (rms(ref) + |ref|) element-wise (about 5x the expected
error).  The forward's absolute 2e-2 bar would say nothing for dK and dV,
whose entries are small sums of P-weighted terms.
"""
import numpy as np
import pytest
import torch

import oracle
from broadcast_gemm_attention_gb300 import binding as B
from broadcast_gemm_attention_gb300 import inputs as gen
from gpu_util import cached

pytestmark = pytest.mark.gpu
GRAD_RTOL = 2e-2


def assert_grad_close(g_gpu: torch.Tensor, ref: np.ndarray, what: str):
    g = g_gpu.detach().to(torch.float64).cpu().numpy().reshape(ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    err = np.abs(g - ref)
    bound = GRAD_RTOL * (rms + np.abs(ref))
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:4].tolist()
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of tolerance (rms {rms:.4g}); max err "
                             f"{np.nanmax(err):.4g}; first {idx}: gpu {g[tuple(idx[0])]:.6g} ref "
                             f"{ref[tuple(idx[0])]:.6g}")


def run_backward(x, dO, plan=None, use_lse=False):
    """Forward (with its log-sum-exp when use_lse), then the backward, which
    then skips its own log-sum-exp pass."""
    Q, K, V, m, g = (t.cuda() for t in (x.Q, x.K, x.V, x.map, dO))
    offs = x.kv_offsets.cuda() if x.jagged else None
    O = torch.empty_like(Q)
    lse = torch.full(tuple(Q.shape[:3]), float("nan"), dtype=torch.float32, device=Q.device) if use_lse else None
    dQ = torch.full_like(Q, float("nan"))
    dK = torch.full_like(K, float("nan"))
    dV = torch.full_like(V, float("nan"))
    own = plan is None
    p = plan or B.Plan(x.n_cand, x.n_users, x.H)
    try:
        p.plan(m, x.n_users, x.H, x.Lq)
        if use_lse:
            p.attn_forward_lse(Q, K, V, offs, O, lse)
        else:
            p.attn_forward(Q, K, V, offs, O)
        l0 = p.launches()
        p.attn_backward(Q, K, V, O, g, offs, dQ, dK, dV, lse=lse)
        launched = p.launches() - l0
        st = p.status()
    finally:
        if own:
            p.close()
    return dQ, dK, dV, st, launched


def kv_rows(x, dK, dV, u, h):
    """User u, head h rows of dK / dV as [L_u, d] arrays."""
    if x.jagged:
        a, b = int(x.kv_offsets[u]), int(x.kv_offsets[u + 1])
        return dK[a:b, h], dV[a:b, h]
    return dK[u, h], dV[u, h]


def check(x, dO, dQ, dK, dV, qpairs=None, kvpairs=None, what="", cache_key=None):
    offs = x.kv_offsets if x.jagged else None
    ref = cached(cache_key, lambda: oracle.attn_backward(x.map, x.Q, x.K, x.V, dO, kv_offsets=offs,
                                                         n_users=x.n_users, qpairs=qpairs, kvpairs=kvpairs))
    if qpairs is None:
        assert_grad_close(dQ, ref["dQ"].reshape(dQ.shape), f"{what} dQ")
    else:
        got = torch.stack([dQ[i, h] for i, h in qpairs])
        assert_grad_close(got, ref["dQ"], f"{what} dQ")
    pairs = kvpairs if kvpairs is not None else [(u, h) for u in range(x.n_users) for h in range(x.H)]
    for s, (u, h) in enumerate(pairs):
        gk, gv = kv_rows(x, dK, dV, u, h)
        L = gk.shape[0]
        assert_grad_close(gk, ref["dK"][s, :L], f"{what} dK[{u},{h}]")
        assert_grad_close(gv, ref["dV"][s, :L], f"{what} dV[{u},{h}]")


@pytest.mark.parametrize("case", [
    dict(n_cand=7, n_users=3, H=2, Lq=32, d=128, Lkv=200),      # two key tiles, ragged 72
    dict(n_cand=40, n_users=4, H=1, Lq=8, d=128, Lkv=130),      # 16 candidates per tile
    dict(n_cand=9, n_users=2, H=2, Lq=48, d=128, Lkv=64),       # 96 of 128 tile rows used
    dict(n_cand=13, n_users=2, H=1, Lq=24, d=128, Lkv=140),     # 5 candidates per tile: halves of 2, 2, 1
    dict(n_cand=5, n_users=2, H=2, Lq=72, d=128, Lkv=150),      # one candidate split over two halves
    dict(n_cand=3, n_users=2, H=1, Lq=128, d=128, Lkv=129),     # a full 128-row candidate
])
@pytest.mark.parametrize("use_lse", [False, True], ids=["recompute_lse", "forward_lse"])
def test_attn_backward_dense(case, use_lse):
    x = gen.make_attn("abwd", 61, map_kind="permuted", **case)
    dO = gen.make_attn_grad(61, x.Q.shape)
    dQ, dK, dV, st, launched = run_backward(x, dO, use_lse=use_lse)
    assert st == B.IKBO_OK
    assert launched == 3
    check(x, dO, dQ, dK, dV, what=str(case))


@pytest.mark.parametrize("use_lse", [False, True], ids=["recompute_lse", "forward_lse"])
def test_attn_backward_user_without_candidates(use_lse):
    """User 1 has keys but no candidates: its dK, dV are 0; the others sum over
    their candidates."""
    x = gen.make_attn("abwd_empty", 62, n_cand=6, n_users=3, H=2, Lq=16, d=128, Lkv=150,
                      explicit_map=[0, 2, 2, 0, 2, 0])
    dO = gen.make_attn_grad(62, x.Q.shape)
    dQ, dK, dV, st, _ = run_backward(x, dO, use_lse=use_lse)
    assert st == B.IKBO_OK
    assert torch.count_nonzero(dK[1]) == 0 and torch.count_nonzero(dV[1]) == 0
    check(x, dO, dQ, dK, dV, what="empty user")


@pytest.mark.parametrize("use_lse", [False, True], ids=["recompute_lse", "forward_lse"])
def test_attn_backward_jagged(use_lse):
    """Jagged K/V with a user without keys (its candidates get dQ = 0) and a
    user whose keys span three tiles."""
    lens = [40, 0, 300, 129]
    x = gen.make_attn("abwd_jag", 63, n_cand=10, n_users=4, H=2, Lq=16, d=128,
                      explicit_map=[2, 0, 1, 3, 2, 0, 1, 3, 2, 2], explicit_lengths=lens)
    dO = gen.make_attn_grad(63, x.Q.shape)
    dQ, dK, dV, st, _ = run_backward(x, dO, use_lse=use_lse)
    assert st == B.IKBO_OK
    assert torch.count_nonzero(dQ[2]) == 0 and torch.count_nonzero(dQ[6]) == 0
    check(x, dO, dQ, dK, dV, what="jagged")


@pytest.mark.parametrize("use_lse", [False, True], ids=["recompute_lse", "forward_lse"])
def test_attn_backward_70to1_full(use_lse):
    """The 70:1 attention shape: every element of dQ, and of dK and dV for all
    120 (user, head) pairs (each the sum over that user's ~70 candidates)."""
    x = gen.attn_70to1()
    dO = gen.make_attn_grad(1003, x.Q.shape)
    dQ, dK, dV, st, launched = run_backward(x, dO, use_lse=use_lse)
    assert st == B.IKBO_OK
    assert launched == 3
    check(x, dO, dQ, dK, dV, what="70:1", cache_key="attn_70to1_backward")


# fp32 scores from 128-term products of bf16 values and fp32 sums over at most
# a few thousand keys: the log-sum-exp is good to ~1e-5 absolute at |LSE| ~ 10
LSE_TOL = 1e-3


@pytest.mark.parametrize("kind", ["dense", "jagged", "70to1"])
def test_attn_forward_lse(kind):
    """ikbo_attn_forward_lse: O bit-identical to ikbo_attn_forward's, and every
    row's log-sum-exp against the oracle within LSE_TOL * (1 + |ref|); -inf
    for the rows of a user without keys."""
    if kind == "dense":
        x = gen.make_attn("alse", 65, n_cand=11, n_users=3, H=2, Lq=32, d=128, Lkv=300, map_kind="permuted")
    elif kind == "jagged":
        x = gen.make_attn("alse_jag", 66, n_cand=8, n_users=4, H=2, Lq=16, d=128,
                          explicit_map=[3, 1, 0, 2, 3, 1, 0, 3], explicit_lengths=[100, 0, 257, 128])
    else:
        x = gen.attn_70to1()
    Q, K, V, m = (t.cuda() for t in (x.Q, x.K, x.V, x.map))
    offs = x.kv_offsets.cuda() if x.jagged else None
    O, O2 = torch.empty_like(Q), torch.empty_like(Q)
    lse = torch.full(tuple(Q.shape[:3]), float("nan"), dtype=torch.float32, device=Q.device)
    with B.Plan(x.n_cand, x.n_users, x.H) as p:
        p.plan(m, x.n_users, x.H, x.Lq)
        p.attn_forward(Q, K, V, offs, O)
        p.attn_forward_lse(Q, K, V, offs, O2, lse)
        assert p.status() == B.IKBO_OK
    assert torch.equal(O, O2)
    ref = oracle.attn_lse(x.map, x.Q, x.K, kv_offsets=x.kv_offsets if x.jagged else None, n_users=x.n_users)
    got = lse.cpu().numpy().astype(np.float64).reshape(-1, x.Lq)
    inf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf)
    err = np.abs(got[~inf] - ref[~inf])
    assert np.all(err <= LSE_TOL * (1 + np.abs(ref[~inf]))), float(err.max())


def test_attn_backward_errors():
    x = gen.make_attn("abwd_err", 64, n_cand=4, n_users=2, H=1, Lq=8, d=128, Lkv=16)
    Q, K, V = x.Q.cuda(), x.K.cuda(), x.V.cuda()
    O, dO = torch.zeros_like(Q), torch.zeros_like(Q)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    L = B.load()
    with B.Plan(4, 2, 1) as p:
        with pytest.raises(B.IkboError) as e:
            p.attn_backward(Q, K, V, O, dO, None, dQ, dK, dV)
        assert e.value.code == B.IKBO_ERR_NOT_PLANNED
        m = x.map.cuda()  # borrowed by the plan for the calls below
        p.plan(m, 2, 1, 8)
        lse = torch.zeros(4, 1, 8, dtype=torch.float32, device=Q.device)
        args = [Q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), dO.data_ptr(), None, None, dQ.data_ptr(),
                dK.data_ptr(), dV.data_ptr(), 16, 128, 0.1, None]
        bad = list(args)
        bad[4] = None
        assert L.ikbo_attn_backward(p.handle, *bad) == B.IKBO_ERR_INVALID_ARG
        bad = list(args)
        bad[7] = dQ.data_ptr() + 2
        assert L.ikbo_attn_backward(p.handle, *bad) == B.IKBO_ERR_INVALID_ARG
        bad = list(args)
        bad[5] = lse.data_ptr() + 2
        assert L.ikbo_attn_backward(p.handle, *bad) == B.IKBO_ERR_INVALID_ARG
        bad = list(args)
        bad[11] = 64
        assert L.ikbo_attn_backward(p.handle, *bad) == B.IKBO_ERR_UNSUPPORTED
        assert L.ikbo_attn_forward_lse(p.handle, Q.data_ptr(), K.data_ptr(), V.data_ptr(), None, O.data_ptr(),
                                       None, 16, 128, 0.1, None) == B.IKBO_ERR_INVALID_ARG
        assert L.ikbo_attn_backward(p.handle, *args) == B.IKBO_OK
        assert p.status() == B.IKBO_OK
