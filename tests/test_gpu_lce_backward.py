"""LCE backward (ikbo_lce_backward) against the fp64 oracle's materialised
backward.

Tolerance: the LCE bar |g_gpu - g_ref| <= 1e-2 (1 + |g_ref|) element-wise for
every gradient.  What it has to absorb: bf16 rounding of the dU / dC outputs
(2^-9 relative), and S = sum of dY rounded to bf16 before the two products
that read it (dU, dWu: 2^-9 relative per term, averaging down over the sum).
The weight gradients are fp32 sums of exact bf16 products.
"""
import numpy as np
import pytest
import torch

import oracle
from broadcast_gemm_attention_gb300 import binding as B
from broadcast_gemm_attention_gb300 import inputs as gen
from gpu_util import assert_lce_close, to_dev

pytestmark = pytest.mark.gpu


def run_backward(x, dY, plan=None, want=("dU", "dC", "dWu", "dWc", "db"), debug=0):
    U, C, Wu, Wc, m, g = to_dev(x.U, x.C, x.Wu, x.Wc, x.map, dY)
    bf, f32 = torch.bfloat16, torch.float32
    shapes = {"dU": ((x.n_users, x.K_u, x.D), bf), "dC": ((x.n_cand, x.K_c, x.D), bf),
              "dWu": ((x.K_u, x.N), f32), "dWc": ((x.K_c, x.N), f32), "db": ((x.N,), f32)}
    out = {k: torch.full(s, float("nan"), dtype=dt, device="cuda") for k, (s, dt) in shapes.items() if k in want}
    own = plan is None
    p = plan or B.Plan(x.n_cand, x.n_users, 1)
    try:
        if debug:
            B.ikbo_plan_set_debug(p.handle, debug)
        p.plan(m, x.n_users)
        l0 = p.launches()
        p.lce_backward(U, C, Wu, Wc, g, **out)
        launched = p.launches() - l0
        st = p.status()
    finally:
        if debug:
            B.ikbo_plan_set_debug(p.handle, 0)
        if own:
            p.close()
    return out, st, launched


def check_all(x, dY, out, cands=None, users=None, what=""):
    ref = oracle.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY, cands=cands, users=users,
                              weights=any(k in out for k in ("dWu", "dWc", "db")))
    sel_c = slice(None) if cands is None else cands
    sel_u = slice(None) if users is None else users
    if "dC" in out:
        assert_lce_close(out["dC"][sel_c], ref["dC"], f"{what} dC")
    if "dU" in out:
        assert_lce_close(out["dU"][sel_u], ref["dU"], f"{what} dU")
    for k in ("dWu", "dWc", "db"):
        if k in out:
            assert_lce_close(out[k], ref[k], f"{what} {k}")


@pytest.mark.parametrize("shape", [
    dict(n_cand=16, n_users=2, K_u=24, K_c=16, D=32, N=8),
    dict(n_cand=37, n_users=3, K_u=37, K_c=29, D=136, N=40),
    dict(n_cand=300, n_users=7, K_u=381, K_c=243, D=384, N=200),   # K_u > 256: one accumulator; N -> 208 columns
    dict(n_cand=90, n_users=30, K_u=130, K_c=260, D=200, N=128),   # K_c > 256, ragged D block
    dict(n_cand=40, n_users=6, K_u=100, K_c=60, D=64, N=256),      # N = 256: the widest weight-gradient tile
    dict(n_cand=500, n_users=40, K_u=50, K_c=100, D=200, N=192),   # one K_c block, many short runs, ragged D block
    dict(n_cand=64, n_users=5, K_u=70, K_c=256, D=64, N=176),      # K_c = 256 exactly, N = 176 (3 n chunks)
])
def test_lce_backward_full(shape):
    x = gen.make_lce("bwd", 91, map_kind="permuted", **shape)
    dY = gen.make_lce_grad(91, x.n_cand, x.N, x.D)
    out, st, launched = run_backward(x, dY)
    assert st == B.IKBO_OK
    if shape["K_c"] <= 256 and shape["N"] <= 192:
        # candidate pass (dC, dW_c, S, db: one cooperative launch), dU, dW_u (one
        # launch as a cluster per K_u block, or split-K partials + reduce)
        assert launched in (3, 4)
    else:
        assert launched >= 7  # segment sum, db, dC, dW_c + reduce, dU, dW_u + reduce
    check_all(x, dY, out, what=str(shape))


def test_lce_backward_few_users_many_candidates():
    """One or two users with many candidates: each user's segment sum is
    spread over many CTAs of the candidate pass, whose partial sums the finish
    kernel adds in CTA order."""
    for n_users in (1, 2):
        x = gen.make_lce("bwd_chunks", 92, 2048, n_users, 64, 48, 128, 64, map_kind="permuted")
        dY = gen.make_lce_grad(92, x.n_cand, x.N, x.D)
        out, st, launched = run_backward(x, dY)
        assert st == B.IKBO_OK
        assert launched in (3, 4)  # candidate pass, dU, dW_u (cluster, or partials + reduce)
        check_all(x, dY, out, what=f"{n_users} users")


@pytest.mark.parametrize("shape", [
    dict(n_cand=300, n_users=7, K_u=100, K_c=243, D=256, N=192, map_kind="permuted"),
    # users 1 and 3 without candidates, ragged D block
    dict(n_cand=37, n_users=5, K_u=37, K_c=29, D=136, N=40, explicit_map=[(0, 2, 4)[i % 3] for i in range(37)]),
])
def test_lce_backward_finish_kernel(shape):
    """The path taken where a cooperative launch is refused: the candidate
    pass, then the finish (dW_c reduce, db, zero S of users without
    candidates) as a second kernel.  Same bits as the one-launch path."""
    x = gen.make_lce("bwd_fin", 96, **shape)
    dY = gen.make_lce_grad(96, x.n_cand, x.N, x.D)
    with B.Plan(x.n_cand, x.n_users, 1) as p:
        two, st, launched = run_backward(x, dY, plan=p, debug=B.DEBUG_NO_COOPERATIVE)
        assert st == B.IKBO_OK
        assert launched in (4, 5)
        one, st, launched = run_backward(x, dY, plan=p)
        assert st == B.IKBO_OK and launched in (3, 4)
    for k in one:
        assert torch.equal(one[k], two[k]), k
    check_all(x, dY, two, what=str(shape))


def test_lce_backward_70to1_full():
    """The 70:1 request shape: every element of dC, dU, dWu, dWc and db."""
    x = gen.lce_70to1()
    dY = gen.make_lce_grad(1001, x.n_cand, x.N, x.D)
    out, st, _ = run_backward(x, dY)
    assert st == B.IKBO_OK
    check_all(x, dY, out, what="70:1")


def test_lce_backward_subsets_and_repeatability():
    """Outputs left out are not written; the others equal the full call's bit
    for bit, and two calls give identical bits (fixed summation order)."""
    x = gen.make_lce("bwd_sub", 93, 120, 5, 100, 70, 256, 96, map_kind="permuted")
    dY = gen.make_lce_grad(93, x.n_cand, x.N, x.D)
    with B.Plan(x.n_cand, x.n_users, 1) as p:
        full, st, _ = run_backward(x, dY, plan=p)
        again, _, _ = run_backward(x, dY, plan=p)
        for want in (("dC",), ("dU", "db"), ("dWc",), ("dWu",)):
            part, st2, _ = run_backward(x, dY, plan=p, want=want)
            assert st2 == B.IKBO_OK
            for k in want:
                assert torch.equal(part[k], full[k]), k
    assert st == B.IKBO_OK
    for k in full:
        assert torch.equal(full[k], again[k]), k


def test_lce_backward_errors():
    x = gen.make_lce("bwd_err", 94, 24, 3, 40, 30, 64, 16)
    dY = gen.make_lce_grad(94, x.n_cand, x.N, x.D)
    U, C, Wu, Wc, m, g = to_dev(x.U, x.C, x.Wu, x.Wc, x.map, dY)
    dC = torch.empty(x.n_cand, x.K_c, x.D, dtype=torch.bfloat16, device="cuda")
    L = B.load()
    with B.Plan(x.n_cand, x.n_users, 1) as p:
        with pytest.raises(B.IkboError) as e:
            p.lce_backward(U, C, Wu, Wc, g, dC=dC)
        assert e.value.code == B.IKBO_ERR_NOT_PLANNED
        p.plan(m, x.n_users)
        # dC needs Wc; dY is required
        rc = L.ikbo_lce_backward(p.handle, None, None, None, None, g.data_ptr(), None, dC.data_ptr(), None, None,
                                 None, x.K_u, x.K_c, x.D, x.N, None)
        assert rc == B.IKBO_ERR_INVALID_ARG
        rc = L.ikbo_lce_backward(p.handle, None, None, None, Wc.data_ptr(), None, None, dC.data_ptr(), None, None,
                                 None, x.K_u, x.K_c, x.D, x.N, None)
        assert rc == B.IKBO_ERR_INVALID_ARG
        # misaligned output, unsupported N
        rc = L.ikbo_lce_backward(p.handle, None, None, None, Wc.data_ptr(), g.data_ptr(), None, dC.data_ptr() + 2,
                                 None, None, None, x.K_u, x.K_c, x.D, x.N, None)
        assert rc == B.IKBO_ERR_INVALID_ARG
        rc = L.ikbo_lce_backward(p.handle, None, None, None, Wc.data_ptr(), g.data_ptr(), None, dC.data_ptr(),
                                 None, None, None, x.K_u, x.K_c, x.D, 264, None)
        assert rc == B.IKBO_ERR_UNSUPPORTED
        # only dC (Wc and dY given): fine
        rc = L.ikbo_lce_backward(p.handle, None, None, None, Wc.data_ptr(), g.data_ptr(), None, dC.data_ptr(),
                                 None, None, None, x.K_u, x.K_c, x.D, x.N, None)
        assert rc == B.IKBO_OK
        assert p.status() == B.IKBO_OK
    ref = oracle.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY, weights=False)
    assert_lce_close(dC, ref["dC"], "dC alone")


def test_lce_backward_map_out_of_range():
    """A candidate with a map value out of range is reported and left out of S
    (dU, dWu, db); dC and dWc still include it."""
    x = gen.make_lce("bwd_oor", 95, 40, 4, 50, 30, 64, 24, map_kind="permuted")
    dY = gen.make_lce_grad(95, x.n_cand, x.N, x.D)
    bad = x.map.clone()
    bad[7] = 9
    y = gen.LCEInputs("oor", x.n_cand, x.n_users, x.K_u, x.K_c, x.D, x.N, bad, x.U, x.C, x.Wu, x.Wc, x.b)
    out, st, _ = run_backward(y, dY)
    assert st == B.IKBO_ERR_MAP_OUT_OF_RANGE
    ref = oracle.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY)
    assert_lce_close(out["dC"], ref["dC"], "dC")
    assert_lce_close(out["dWc"], ref["dWc"], "dWc")
    # the user side equals the oracle on a map without candidate 7 (its dY zeroed)
    dY0 = dY.clone()
    dY0[7] = 0
    ref0 = oracle.lce_backward(x.map, x.U, x.C, x.Wu, x.Wc, dY0)
    for k in ("dU", "dWu", "db"):
        assert_lce_close(out[k], ref0[k], k)
