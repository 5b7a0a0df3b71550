"""Pins for the CPU oracle: checks against what the IKBO pages and plain
mathematics fix, never against the oracle's own formula retyped.

Each ``pin_*`` takes a loaded oracle build and raises AssertionError when the
oracle disagrees with the pin.  ``test_oracle_*.py`` run them on the real
oracle; ``test_oracle_mutations.py`` runs them on copies of the oracle with a
planted mistake and expects at least one pin to fail.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np
import torch
import torch.nn.functional as F

from broadcast_gemm_attention_gb300 import inputs as gen


def f64(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.float64).numpy()


# ====================================================================== LCE
def _small_lce(seed=7, n_cand=9, n_users=3, K_u=5, K_c=7, D=8, N=4, map_kind="permuted", bias=True):
    return gen.make_lce("pin", seed, n_cand, n_users, K_u, K_c, D, N, map_kind=map_kind, bias=bias,
                        w_var=0.3)


def pin_lce_decomposition(orc):
    """Type I decomposition (aibriefing, "Type I"; aixai.ru, LCE stage 1): the
    materialised GEMM equals U[map[i]]-part + C[i]-part + b, each a separate
    library matmul at its own batch size."""
    x = _small_lce()
    Y = orc.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    m = x.map.numpy()
    user = np.einsum("kn,ukd->und", f64(x.Wu), f64(x.U))          # at n_users
    cand = np.matmul(f64(x.Wc).T[None], f64(x.C))                  # at n_cand
    ref = user[m] + cand + f64(x.b)[None, :, None]
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def pin_lce_exact_rational(orc):
    """Brute force in exact rational arithmetic on the tiny workload: bf16
    inputs are dyadic rationals, so the exact value of every output is known;
    fp64 accumulation of <= 40 products must land within 1e-13 of it."""
    x = gen.lce_tiny()
    Y = orc.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    U, C, Wu, Wc, b = (t.to(torch.float64).tolist() for t in (x.U, x.C, x.Wu, x.Wc, x.b))
    m = x.map.tolist()
    picks = [(0, 0, 0), (3, 7, 31), (8, 2, 5), (15, 5, 17), (11, 0, 30)]
    for i, n, d in picks:
        u = m[i]
        acc = Fraction(b[n])
        for k in range(x.K_u):
            acc += Fraction(Wu[k][n]) * Fraction(U[u][k][d])
        for k in range(x.K_c):
            acc += Fraction(Wc[k][n]) * Fraction(C[i][k][d])
        assert abs(Y[i, n, d] - float(acc)) <= 1e-13 * (1 + abs(float(acc))), (i, n, d)


def pin_lce_single_user_no_candidate_part(orc):
    """n_users = 1 and W_c = 0: every candidate gets W_u^T U[0] + b (one matmul)."""
    x = _small_lce(n_users=1, map_kind="sorted")
    Wc0 = torch.zeros_like(x.Wc)
    Y = orc.lce(x.map, x.U, x.C, x.Wu, Wc0, x.b)
    ref = np.matmul(f64(x.Wu).T, f64(x.U)[0]) + f64(x.b)[:, None]
    for i in range(x.n_cand):
        np.testing.assert_allclose(Y[i], ref, rtol=1e-12, atol=1e-12)


def pin_lce_identity_map_is_batched_gemm(orc):
    """map = identity with no user rows (K_u = 0): a plain batched GEMM."""
    x = gen.make_lce("pin", 11, 6, 6, 0, 9, 8, 4, explicit_map=list(range(6)), bias=False, w_var=0.3)
    Y = orc.lce(x.map, x.U, x.C, x.Wu, x.Wc, None)
    ref = np.matmul(f64(x.Wc).T[None], f64(x.C))
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def pin_lce_one_sided(orc):
    """U = 0 leaves the candidate GEMM + b; C = 0 leaves the user GEMM + b."""
    x = _small_lce(seed=9)
    m = x.map.numpy()
    Y = orc.lce(x.map, torch.zeros_like(x.U), x.C, x.Wu, x.Wc, x.b)
    np.testing.assert_allclose(Y, np.matmul(f64(x.Wc).T[None], f64(x.C)) + f64(x.b)[None, :, None],
                               rtol=1e-12, atol=1e-12)
    Y = orc.lce(x.map, x.U, torch.zeros_like(x.C), x.Wu, x.Wc, x.b)
    ref = np.matmul(f64(x.Wu).T[None], f64(x.U)[m]) + f64(x.b)[None, :, None]
    np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def pin_lce_permutation(orc):
    """Permuting candidates (map and C together) permutes Y, exactly."""
    x = _small_lce(seed=13, n_cand=12, n_users=4)
    Y = orc.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    p = torch.from_numpy(np.random.default_rng(5).permutation(x.n_cand))
    Yp = orc.lce(x.map[p], x.U, x.C[p], x.Wu, x.Wc, x.b)
    assert np.array_equal(Yp, Y[p.numpy()])


def pin_lce_zero_padding(orc):
    """Zero-padding K (the pages' stage 2 trick, stated mathematically
    equivalent) leaves Y unchanged."""
    x = _small_lce(seed=17)
    Y = orc.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    pu, pc = 3, 5
    U2 = torch.cat([x.U, torch.zeros(x.n_users, pu, x.D, dtype=torch.bfloat16)], 1)
    Wu2 = torch.cat([x.Wu, torch.zeros(pu, x.N, dtype=torch.bfloat16)], 0)
    C2 = torch.cat([x.C, torch.zeros(x.n_cand, pc, x.D, dtype=torch.bfloat16)], 1)
    Wc2 = torch.cat([x.Wc, torch.zeros(pc, x.N, dtype=torch.bfloat16)], 0)
    Y2 = orc.lce(x.map, U2, C2, Wu2, Wc2, x.b)
    np.testing.assert_allclose(Y2, Y, rtol=0, atol=1e-15)


def pin_lce_selection(orc):
    """Evaluating a subset of candidates returns exactly those rows."""
    x = _small_lce(seed=19)
    Y = orc.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    sel = [4, 0, 8, 4]
    Ys = orc.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b, cands=sel)
    assert np.array_equal(Ys, Y[sel])


LCE_PINS = [pin_lce_decomposition, pin_lce_exact_rational, pin_lce_single_user_no_candidate_part,
            pin_lce_identity_map_is_batched_gemm, pin_lce_one_sided, pin_lce_permutation,
            pin_lce_zero_padding, pin_lce_selection]


# ============================================================ LCE backward
def _dot(a, b) -> float:
    return float(np.sum(np.asarray(a, np.float64) * np.asarray(b, np.float64)))


def _bwd_case(seed=23, **kw):
    x = _small_lce(seed=seed, **kw)
    return x, gen.make_lce_grad(seed, x.n_cand, x.N, x.D)


def pin_lce_bwd_adjoint(orc):
    """The adjoint identity of a linear map: for each input t, with the others
    fixed, Y is affine in t, so <dY, Y(t = dt) - Y(t = 0)> = <dL/dt, dt>.  The
    right-hand side uses the backward; the left-hand side only the forward
    (pinned on its own), evaluated with every other contribution zeroed."""
    x, dY = _bwd_case()
    g = orc.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY)
    rng = np.random.default_rng(3)
    bf = lambda shape: torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    zU, zC = torch.zeros_like(x.U), torch.zeros_like(x.C)
    dU, dC, dWu, dWc, db = bf(tuple(x.U.shape)), bf(tuple(x.C.shape)), bf(tuple(x.Wu.shape)), bf(tuple(x.Wc.shape)), bf((x.N,))
    lhs = {
        "dU": _dot(f64(dY), orc.lce(x.map, dU, zC, x.Wu, x.Wc, None)),
        "dC": _dot(f64(dY), orc.lce(x.map, zU, dC, x.Wu, x.Wc, None)),
        "dWu": _dot(f64(dY), orc.lce(x.map, x.U, zC, dWu, x.Wc, None)),
        "dWc": _dot(f64(dY), orc.lce(x.map, zU, x.C, x.Wu, dWc, None)),
        "db": _dot(f64(dY), orc.lce(x.map, zU, zC, x.Wu, x.Wc, db)),
    }
    rhs = {"dU": _dot(g["dU"], f64(dU)), "dC": _dot(g["dC"], f64(dC)), "dWu": _dot(g["dWu"], f64(dWu)),
           "dWc": _dot(g["dWc"], f64(dWc)), "db": _dot(g["db"], f64(db))}
    for k in lhs:
        assert abs(lhs[k] - rhs[k]) <= 1e-10 * (1 + abs(lhs[k])), (k, lhs[k], rhs[k])


def pin_lce_bwd_autograd(orc):
    """torch fp64 autograd through the materialised forward (U[map] gathered,
    concatenated with C, one batched matmul, + b) gives every gradient."""
    x, dY = _bwd_case(seed=29, n_cand=11, n_users=4)
    g = orc.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY)
    t = {k: torch.tensor(f64(v), requires_grad=True) for k, v in
         dict(U=x.U, C=x.C, Wu=x.Wu, Wc=x.Wc, b=x.b).items()}
    Xrep = torch.cat([t["U"][x.map.long()], t["C"]], dim=1)
    W = torch.cat([t["Wu"], t["Wc"]], dim=0)
    Y = torch.matmul(W.t().unsqueeze(0), Xrep) + t["b"][None, :, None]
    (Y * torch.tensor(f64(dY))).sum().backward()
    for mine, ref in (("dU", "U"), ("dC", "C"), ("dWu", "Wu"), ("dWc", "Wc"), ("db", "b")):
        np.testing.assert_allclose(g[mine], t[ref].grad.numpy(), rtol=1e-11, atol=1e-11, err_msg=mine)


def pin_lce_bwd_closed_forms(orc):
    """dY = 0 gives zero gradients.  dY = 1 gives db[n] = n_cand * D,
    dWc[k][n] = sum_{i,d} C[i][k][d] (the same for every n),
    dU[u][k][d] = count_u * sum_n Wu[k][n] (0 for a user with no candidates),
    dC[i][k][d] = sum_n Wc[k][n]."""
    x = gen.make_lce("pin", 31, 7, 4, 3, 5, 6, 4, explicit_map=[0, 2, 2, 0, 2, 0, 0], w_var=0.3)
    z = orc.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, torch.zeros(x.n_cand, x.N, x.D, dtype=torch.bfloat16))
    for k, v in z.items():
        assert not np.any(v), k
    g = orc.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, torch.ones(x.n_cand, x.N, x.D, dtype=torch.bfloat16))
    np.testing.assert_allclose(g["db"], np.full(x.N, x.n_cand * x.D, np.float64), rtol=0, atol=0)
    csum = f64(x.C).sum(axis=(0, 2))
    np.testing.assert_allclose(g["dWc"], np.repeat(csum[:, None], x.N, 1), rtol=1e-13, atol=1e-13)
    counts = np.bincount(x.map.numpy(), minlength=x.n_users)
    wsum = f64(x.Wu).sum(axis=1)
    for u in range(x.n_users):
        np.testing.assert_allclose(g["dU"][u], counts[u] * np.repeat(wsum[:, None], x.D, 1), rtol=1e-13, atol=1e-13)
    wcs = f64(x.Wc).sum(axis=1)
    for i in range(x.n_cand):
        np.testing.assert_allclose(g["dC"][i], np.repeat(wcs[:, None], x.D, 1), rtol=1e-13, atol=1e-13)


def pin_lce_bwd_permutation(orc):
    """Permuting candidates (map, C and dY together) permutes dC and leaves
    dU, dWu, dWc and db unchanged."""
    x, dY = _bwd_case(seed=37, n_cand=12, n_users=4)
    g = orc.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY)
    p = torch.from_numpy(np.random.default_rng(8).permutation(x.n_cand))
    gp = orc.lce_backward(x.map[p], x.U, x.C[p], x.Wu, x.Wc, dY[p])
    assert np.array_equal(gp["dC"], g["dC"][p.numpy()])
    for k in ("dU", "dWu", "dWc", "db"):
        np.testing.assert_allclose(gp[k], g[k], rtol=1e-12, atol=1e-12, err_msg=k)


def pin_lce_bwd_selection(orc):
    """Selected candidates and users return exactly those rows."""
    x, dY = _bwd_case(seed=41)
    g = orc.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY)
    s = orc.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY, cands=[5, 0, 5], users=[2, 0], weights=False)
    assert np.array_equal(s["dC"], g["dC"][[5, 0, 5]])
    assert np.array_equal(s["dU"], g["dU"][[2, 0]])
    assert set(s) == {"dC", "dU"}


LCE_BWD_PINS = [pin_lce_bwd_adjoint, pin_lce_bwd_autograd, pin_lce_bwd_closed_forms, pin_lce_bwd_permutation,
                pin_lce_bwd_selection]


# ================================================================ attention
def _sdpa64(q, k, v, scale=None):
    return F.scaled_dot_product_attention(q.to(torch.float64), k.to(torch.float64),
                                          v.to(torch.float64), scale=scale).numpy()


def pin_attn_identity_map_is_sdpa(orc):
    """map = identity (one candidate per user) is ordinary batched attention:
    torch's fp64 scaled_dot_product_attention on the CPU."""
    x = gen.make_attn("pin", 21, n_cand=5, n_users=5, H=3, Lq=4, d=16, Lkv=11,
                      explicit_map=list(range(5)))
    O = orc.attn(x.map, x.Q, x.K, x.V).reshape(5, 3, 4, 16)
    ref = _sdpa64(x.Q, x.K, x.V)
    np.testing.assert_allclose(O, ref, rtol=1e-10, atol=1e-12)


def pin_attn_single_user_is_mqa(orc):
    """One user serving every candidate: multi-query attention of all
    candidates' queries against the one K/V (SDPA on the expanded K/V)."""
    x = gen.make_attn("pin", 23, n_cand=6, n_users=1, H=2, Lq=3, d=16, Lkv=9, explicit_map=[0] * 6)
    O = orc.attn(x.map, x.Q, x.K, x.V).reshape(6, 2, 3, 16)
    ref = _sdpa64(x.Q, x.K.expand(6, -1, -1, -1), x.V.expand(6, -1, -1, -1))
    np.testing.assert_allclose(O, ref, rtol=1e-10, atol=1e-12)


def pin_attn_broadcast_is_sdpa_on_gathered_kv(orc):
    """General map: equal to SDPA on the materialised K[map], V[map]."""
    x = gen.make_attn("pin", 25, n_cand=10, n_users=3, H=2, Lq=5, d=16, Lkv=13, map_kind="permuted")
    O = orc.attn(x.map, x.Q, x.K, x.V).reshape(10, 2, 5, 16)
    idx = x.map.long()
    ref = _sdpa64(x.Q, x.K[idx], x.V[idx])
    np.testing.assert_allclose(O, ref, rtol=1e-10, atol=1e-12)


def pin_attn_closed_forms(orc):
    """Q = 0 gives the mean of the user's V rows; a constant V gives that
    constant; a single key gives its V row; one dominant score picks its row."""
    d, L = 16, 7
    x = gen.make_attn("pin", 27, n_cand=4, n_users=2, H=1, Lq=2, d=d, Lkv=L, explicit_map=[1, 0, 1, 0])
    O = orc.attn(x.map, torch.zeros_like(x.Q), x.K, x.V).reshape(4, 2, d)
    for i, u in enumerate(x.map.tolist()):
        mean = f64(x.V[u, 0]).mean(0)
        np.testing.assert_allclose(O[i], np.broadcast_to(mean, (2, d)), rtol=1e-12, atol=1e-13)
    Vc = torch.full_like(x.V, 0.375)
    O = orc.attn(x.map, x.Q, x.K, Vc)
    np.testing.assert_allclose(O, 0.375, rtol=0, atol=1e-14)
    x1 = gen.make_attn("pin", 29, n_cand=3, n_users=2, H=2, Lq=2, d=d, Lkv=1, explicit_map=[1, 1, 0])
    O = orc.attn(x1.map, x1.Q, x1.K, x1.V).reshape(3, 2, 2, d)
    for i, u in enumerate(x1.map.tolist()):
        for h in range(2):
            np.testing.assert_allclose(O[i, h], np.broadcast_to(f64(x1.V[u, h, 0]), (2, d)), rtol=0, atol=0)
    # one dominant score: key j* = 3 aligned with the query, the rest orthogonal
    K = torch.zeros(1, 1, 6, d, dtype=torch.bfloat16)
    K[0, 0, 3, 0] = 8.0
    K[0, 0, :, 1] = 1.0
    Q = torch.zeros(1, 1, 1, d, dtype=torch.bfloat16)
    Q[0, 0, 0, 0] = 8.0
    V = gen.make_attn("pin", 31, 1, 1, 1, 1, d, Lkv=6, explicit_map=[0]).V
    O = orc.attn(torch.tensor([0], dtype=torch.int32), Q, K, V)
    # score gap 64/sqrt(16) = 16 -> the other 5 rows weigh 5 e^-16 ~ 5.6e-7 in total
    np.testing.assert_allclose(O[0, 0], f64(V[0, 0, 3]), rtol=0, atol=5e-6)


def pin_attn_permutation(orc):
    """Permuting candidates (map and Q together) permutes O, exactly."""
    x = gen.make_attn("pin", 33, n_cand=8, n_users=3, H=2, Lq=3, d=16, Lkv=10, map_kind="permuted")
    O = orc.attn(x.map, x.Q, x.K, x.V).reshape(8, 2, 3, 16)
    p = torch.from_numpy(np.random.default_rng(3).permutation(8))
    Op = orc.attn(x.map[p], x.Q[p], x.K, x.V).reshape(8, 2, 3, 16)
    assert np.array_equal(Op, O[p.numpy()])


def pin_attn_jagged(orc):
    """Jagged K/V [sum L, H, d] with int32 offsets: each candidate attends to
    exactly its user's slice (SDPA per slice); an empty slice gives 0."""
    lens = [5, 0, 12, 3]
    x = gen.make_attn("pin", 35, n_cand=7, n_users=4, H=2, Lq=3, d=16,
                      explicit_map=[2, 0, 1, 3, 2, 0, 1], explicit_lengths=lens)
    O = orc.attn(x.map, x.Q, x.K, x.V, kv_offsets=x.kv_offsets).reshape(7, 2, 3, 16)
    offs = x.kv_offsets.tolist()
    for i, u in enumerate(x.map.tolist()):
        a, b = offs[u], offs[u + 1]
        if b == a:
            assert np.all(O[i] == 0)
            continue
        k = x.K[a:b].permute(1, 0, 2).unsqueeze(0)
        v = x.V[a:b].permute(1, 0, 2).unsqueeze(0)
        ref = _sdpa64(x.Q[i:i + 1], k, v)[0]
        np.testing.assert_allclose(O[i], ref, rtol=1e-10, atol=1e-12)


def pin_attn_scale(orc):
    """An explicit scale is honoured: scale s on Q.K equals default scale on (s*sqrt(d)) Q."""
    x = gen.make_attn("pin", 37, n_cand=3, n_users=2, H=1, Lq=2, d=16, Lkv=6, explicit_map=[0, 1, 1])
    O = orc.attn(x.map, x.Q, x.K, x.V, scale=0.5).reshape(3, 1, 2, 16)
    ref = _sdpa64(x.Q, x.K[x.map.long()], x.V[x.map.long()], scale=0.5)
    np.testing.assert_allclose(O, ref, rtol=1e-10, atol=1e-12)


ATTN_PINS = [pin_attn_identity_map_is_sdpa, pin_attn_single_user_is_mqa,
             pin_attn_broadcast_is_sdpa_on_gathered_kv, pin_attn_closed_forms,
             pin_attn_permutation, pin_attn_jagged, pin_attn_scale]

# ------------------------------------------------------- softmax log-sum-exp
def pin_attn_lse_is_logsumexp(orc):
    """General map and an explicit scale: torch's fp64 logsumexp of the scores
    against the gathered K[map] (a library routine on a separately formed
    score matrix)."""
    x = gen.make_attn("pin", 41, n_cand=9, n_users=3, H=2, Lq=3, d=16, Lkv=14, map_kind="permuted")
    for scale in (None, 0.3):
        got = orc.attn_lse(x.map, x.Q, x.K, scale=scale).reshape(9, 2, 3)
        sc = 0.25 if scale is None else scale
        s = torch.einsum("ihqc,ihjc->ihqj", x.Q.to(torch.float64), x.K[x.map.long()].to(torch.float64)) * sc
        np.testing.assert_allclose(got, torch.logsumexp(s, -1).numpy(), rtol=1e-12, atol=1e-12)


def pin_attn_lse_closed_forms(orc):
    """Q = 0: every score is 0, LSE = log L; one key: LSE is its score; an
    empty jagged slice: -inf; and the forward's output is the softmax that
    this normaliser defines: O = sum_j exp(s_j - LSE) V_j."""
    x = gen.make_attn("pin", 43, n_cand=4, n_users=2, H=1, Lq=2, d=16, Lkv=7, explicit_map=[1, 0, 1, 0])
    got = orc.attn_lse(x.map, torch.zeros_like(x.Q), x.K)
    np.testing.assert_allclose(got, np.log(7.0), rtol=0, atol=1e-15)
    x1 = gen.make_attn("pin", 45, n_cand=3, n_users=2, H=2, Lq=2, d=16, Lkv=1, explicit_map=[1, 1, 0])
    got = orc.attn_lse(x1.map, x1.Q, x1.K).reshape(3, 2, 2)
    for i, u in enumerate(x1.map.tolist()):
        for h in range(2):
            np.testing.assert_allclose(got[i, h], f64(x1.Q[i, h]) @ f64(x1.K[u, h, 0]) * 0.25, rtol=1e-14, atol=1e-14)
    lens = [5, 0, 9]
    xj = gen.make_attn("pin", 47, n_cand=5, n_users=3, H=2, Lq=2, d=16,
                       explicit_map=[2, 1, 0, 1, 2], explicit_lengths=lens)
    got = orc.attn_lse(xj.map, xj.Q, xj.K, kv_offsets=xj.kv_offsets).reshape(5, 2, 2)
    assert np.all(np.isneginf(got[1])) and np.all(np.isneginf(got[3]))
    assert np.all(np.isfinite(got[[0, 2, 4]]))
    x2 = gen.make_attn("pin", 49, n_cand=5, n_users=2, H=2, Lq=3, d=16, Lkv=10, map_kind="permuted")
    lse = orc.attn_lse(x2.map, x2.Q, x2.K).reshape(5, 2, 3)
    O = orc.attn(x2.map, x2.Q, x2.K, x2.V).reshape(5, 2, 3, 16)
    for i, u in enumerate(x2.map.tolist()):
        for h in range(2):
            s = f64(x2.Q[i, h]) @ f64(x2.K[u, h]).T * 0.25
            w = np.exp(s - lse[i, h][:, None])
            np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-13)
            np.testing.assert_allclose(O[i, h], w @ f64(x2.V[u, h]), rtol=1e-11, atol=1e-12)


ATTN_LSE_PINS = [pin_attn_lse_is_logsumexp, pin_attn_lse_closed_forms]


# ================================================================ segments
def _check_segments_against_brute_force(orc, m: np.ndarray, n_users: int, H: int, cpu: int):
    counts, offsets, perm, work = orc.segments(m, n_users, H, cpu)
    # brute force with library routines
    assert np.array_equal(counts, np.bincount(m, minlength=n_users))
    assert np.array_equal(perm, np.argsort(m, kind="stable"))
    assert offsets[0] == 0 and offsets[-1] == len(m)
    assert np.array_equal(np.diff(offsets), counts)
    # invariants
    assert sorted(perm.tolist()) == list(range(len(m)))
    for u in range(n_users):
        seg = perm[offsets[u]:offsets[u + 1]]
        assert np.all(m[seg] == u)
        assert np.all(np.diff(seg) > 0)
    # work list: units cover every (u, h) segment exactly, in (u, h, start) order
    covered = {}
    prev = None
    for u, h, s, c in work.tolist():
        assert 1 <= c <= cpu
        key = (u, h, s)
        assert prev is None or key > prev
        prev = key
        covered.setdefault((u, h), []).append((s, c))
    for u in range(n_users):
        for h in range(H):
            runs = covered.get((u, h), [])
            if counts[u] == 0:
                assert runs == []
                continue
            pos = offsets[u]
            for s, c in runs:
                assert s == pos
                pos += c
            assert pos == offsets[u + 1]
            assert all(c == cpu for _, c in runs[:-1])
    assert len(work) == H * sum(-(-int(c) // cpu) for c in counts)


def pin_segments_brute_force(orc):
    rng = np.random.default_rng(41)
    for n, U in [(1, 1), (17, 4), (300, 7), (1024, 15), (513, 600)]:
        m = rng.integers(0, U, size=n).astype(np.int32)
        _check_segments_against_brute_force(orc, m, U, 3, 4)
    m = gen.zipf_permuted_map(np.random.default_rng(2), 4096, 64, 1.1)
    _check_segments_against_brute_force(orc, m, 64, 8, 16)


def pin_segments_special_cases(orc):
    m = np.repeat(np.arange(5, dtype=np.int32), [3, 0, 4, 1, 2])
    counts, offsets, perm, work = orc.segments(m, 5, 2, 2)
    assert np.array_equal(perm, np.arange(len(m)))           # sorted map: identity
    assert offsets.tolist() == [0, 3, 3, 7, 8, 10]
    counts, offsets, perm, work = orc.segments(np.zeros(9, np.int32), 1, 1, 4)
    assert offsets.tolist() == [0, 9] and work.tolist() == [[0, 0, 0, 4], [0, 0, 4, 4], [0, 0, 8, 1]]
    counts, offsets, perm, work = orc.segments(np.array([2, 0, 2, 0, 1], np.int32), 4, 1, 8)
    assert perm.tolist() == [1, 3, 4, 0, 2] and counts.tolist() == [2, 1, 2, 0]
    assert work.tolist() == [[0, 0, 0, 2], [1, 0, 2, 1], [2, 0, 3, 2]]


SEG_PINS = [pin_segments_brute_force, pin_segments_special_cases]
ALL_PINS = LCE_PINS + ATTN_PINS + SEG_PINS


# ===================================================== attention backward
def _attn_autograd(Q, K, V, dO, m, scale):
    """torch fp64 autograd through softmax(scale Q K[m]^T) V[m]: the gather's
    own backward sums the K/V gradients over each user's candidates."""
    q, k, v = (torch.tensor(f64(t), requires_grad=True) for t in (Q, K, V))
    idx = m.long()
    kg, vg = k[idx], v[idx]                       # [n_cand, H, L, d]
    p = torch.softmax(scale * torch.matmul(q, kg.transpose(-1, -2)), dim=-1)
    o = torch.matmul(p, vg)
    (o * torch.tensor(f64(dO))).sum().backward()
    return q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


def pin_attn_bwd_autograd(orc):
    """Dense K/V, permuted map with a user that has no candidates (its dK, dV
    must be 0): every gradient equals torch fp64 autograd."""
    x = gen.make_attn("pin", 41, n_cand=9, n_users=4, H=2, Lq=3, d=16, Lkv=7,
                      explicit_map=[2, 0, 2, 1, 0, 2, 1, 0, 2])
    dO = gen.make_attn_grad(41, x.Q.shape)
    g = orc.attn_backward(x.map, x.Q, x.K, x.V, dO)
    dq, dk, dv = _attn_autograd(x.Q, x.K, x.V, dO, x.map, 1.0 / math.sqrt(16))
    np.testing.assert_allclose(g["dQ"].reshape(dq.shape), dq, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dK"].reshape(dk.shape), dk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dV"].reshape(dv.shape), dv, rtol=1e-10, atol=1e-12)
    assert not np.any(g["dK"].reshape(dk.shape)[3]) and not np.any(g["dV"].reshape(dv.shape)[3])


def pin_attn_bwd_closed_forms(orc):
    """dO = 0: zero gradients.  One key: p = 1, so dQ = dK = 0 and dV[u] = sum
    of dO over u's candidates and queries.  Constant V rows: dP is constant
    along keys, dS = 0, so dQ = dK = 0.  Always: sum_j dV[u,h,j] = sum of dO
    over u's candidates and queries (each row of P sums to 1)."""
    x = gen.make_attn("pin", 43, n_cand=6, n_users=2, H=2, Lq=4, d=8, Lkv=5, explicit_map=[0, 1, 1, 0, 1, 1])
    dO = gen.make_attn_grad(43, x.Q.shape)
    z = orc.attn_backward(x.map, x.Q, x.K, x.V, torch.zeros_like(dO))
    for k, v in z.items():
        assert not np.any(v), k
    g = orc.attn_backward(x.map, x.Q, x.K, x.V, dO)
    m = x.map.numpy()
    dOs = np.stack([f64(dO)[m == u].sum(axis=(0, 2)) for u in range(2)])       # [u, H, d]
    np.testing.assert_allclose(g["dV"].reshape(2, 2, 5, 8).sum(axis=2), dOs, rtol=1e-12, atol=1e-12)
    one = orc.attn_backward(x.map, x.Q, x.K[:, :, :1].contiguous(), x.V[:, :, :1].contiguous(), dO)
    assert np.allclose(one["dQ"], 0, atol=1e-13) and np.allclose(one["dK"], 0, atol=1e-13)
    np.testing.assert_allclose(one["dV"].reshape(2, 2, 8), dOs, rtol=1e-12, atol=1e-12)
    Vc = x.V[:, :, :1].expand(-1, -1, 5, -1).contiguous()
    c = orc.attn_backward(x.map, x.Q, x.K, Vc, dO)
    assert np.allclose(c["dQ"], 0, atol=1e-12) and np.allclose(c["dK"], 0, atol=1e-12)


def pin_attn_bwd_permutation(orc):
    """Permuting candidates (map, Q and dO together) permutes dQ and leaves dK
    and dV unchanged."""
    x = gen.make_attn("pin", 47, n_cand=8, n_users=3, H=2, Lq=2, d=8, Lkv=6, map_kind="permuted")
    dO = gen.make_attn_grad(47, x.Q.shape)
    g = orc.attn_backward(x.map, x.Q, x.K, x.V, dO)
    p = torch.from_numpy(np.random.default_rng(4).permutation(8))
    gp = orc.attn_backward(x.map[p], x.Q[p], x.K, x.V, dO[p])
    np.testing.assert_array_equal(gp["dQ"].reshape(8, 2, 2, 8), g["dQ"].reshape(8, 2, 2, 8)[p.numpy()])
    for k in ("dK", "dV"):
        np.testing.assert_allclose(gp[k], g[k], rtol=1e-12, atol=1e-13, err_msg=k)


def pin_attn_bwd_jagged_and_selection(orc):
    """Jagged K/V: each user's dK/dV slice equals a dense single-user case
    (its candidates only); selections return exactly those rows."""
    lens = [4, 0, 7]
    x = gen.make_attn("pin", 53, n_cand=6, n_users=3, H=2, Lq=2, d=8, explicit_map=[2, 0, 1, 2, 0, 2],
                      explicit_lengths=lens)
    dO = gen.make_attn_grad(53, x.Q.shape)
    g = orc.attn_backward(x.map, x.Q, x.K, x.V, dO, kv_offsets=x.kv_offsets)
    offs = x.kv_offsets.tolist()
    m = x.map.numpy()
    for u in range(3):
        a, b = offs[u], offs[u + 1]
        sel = np.nonzero(m == u)[0]
        gk = g["dK"].reshape(3, 2, 7, 8)[u]
        gv = g["dV"].reshape(3, 2, 7, 8)[u]
        if b == a or len(sel) == 0:
            assert not np.any(gk) and not np.any(gv)
            continue
        Kd = x.K[a:b].permute(1, 0, 2).unsqueeze(0).contiguous()
        Vd = x.V[a:b].permute(1, 0, 2).unsqueeze(0).contiguous()
        s = orc.attn_backward(torch.zeros(len(sel), dtype=torch.int32), x.Q[sel], Kd, Vd, dO[sel])
        np.testing.assert_allclose(gk[:, :b - a], s["dK"].reshape(2, b - a, 8), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(gv[:, :b - a], s["dV"].reshape(2, b - a, 8), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(g["dQ"].reshape(6, 2, 2, 8)[sel], s["dQ"].reshape(len(sel), 2, 2, 8),
                                   rtol=1e-12, atol=1e-13)
        assert not np.any(gk[:, b - a:]) and not np.any(gv[:, b - a:])
    part = orc.attn_backward(x.map, x.Q, x.K, x.V, dO, kv_offsets=x.kv_offsets, qpairs=[[4, 1], [0, 0]],
                             kvpairs=[[2, 1]])
    assert np.array_equal(part["dQ"], g["dQ"][[4 * 2 + 1, 0]])
    assert np.array_equal(part["dK"][0], g["dK"][2 * 2 + 1])


ATTN_BWD_PINS = [pin_attn_bwd_autograd, pin_attn_bwd_closed_forms, pin_attn_bwd_permutation,
                 pin_attn_bwd_jagged_and_selection]
