"""Fused LCE on the GPU against the fp64 oracle (materialised definition).

Tolerance: |Y_gpu - Y_ref| <= 1e-2 (1 + |Y_ref|) element-wise.
"""
import numpy as np
import pytest
import torch

import oracle
from broadcast_gemm_attention_gb300 import binding as B
from broadcast_gemm_attention_gb300 import inputs as gen
from gpu_util import assert_lce_close, check_lce_all, to_dev

pytestmark = pytest.mark.gpu


def run_lce(x, plan=None, bias=True):
    U, C, Wu, Wc, b, m = to_dev(x.U, x.C, x.Wu, x.Wc, x.b if bias else None, x.map)
    Y = torch.full((x.n_cand, x.N, x.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    own = plan is None
    p = plan or B.Plan(x.n_cand, x.n_users, 1)
    try:
        p.plan(m, x.n_users)
        p.lce_forward(U, C, Wu, Wc, b, Y)
        st = p.status()
    finally:
        if own:
            p.close()
    return Y, st


def full_check(x, bias=True):
    Y, st = run_lce(x, bias=bias)
    assert st == B.IKBO_OK
    ref = oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b if bias else None)
    return assert_lce_close(Y, ref, x.name)


def test_lce_tiny():
    """16 candidates, 2 users, K_u 24, K_c 16, D 32, N 8 (every output checked)."""
    full_check(gen.lce_tiny())


@pytest.mark.parametrize("shape", [
    dict(n_cand=37, n_users=3, K_u=37, K_c=29, D=136, N=40),     # ragged K, D and N
    dict(n_cand=5, n_users=5, K_u=8, K_c=8, D=8, N=16),          # minimum sizes, identity-like
    dict(n_cand=64, n_users=1, K_u=700, K_c=100, D=256, N=192),  # long user K (11 chunks > 8 W slots)
    dict(n_cand=20, n_users=4, K_u=64, K_c=256, D=128, N=256),   # Wc region at its limit (16 boxes)
    dict(n_cand=300, n_users=7, K_u=381, K_c=243, D=384, N=200),  # 3 D blocks, N_mma 208
])
@pytest.mark.parametrize("map_kind", ["sorted", "permuted"])
def test_lce_shapes(shape, map_kind):
    x = gen.make_lce("shape", 77, map_kind=map_kind, **shape)
    full_check(x)


def test_lce_no_bias():
    x = gen.make_lce("nobias", 5, 40, 6, 50, 70, 64, 24, map_kind="permuted", bias=False)
    full_check(x, bias=False)


def test_lce_70to1_full():
    """The 70:1 request shape, in the launch configuration the benchmark uses;
    every element of Y against the oracle."""
    x = gen.lce_70to1()
    Y, st = run_lce(x)
    assert st == B.IKBO_OK
    check_lce_all(Y, x, what="70:1", cache_key="lce_70to1")


def test_lce_many_empty_users():
    """3 000 users of which ~20 have candidates (runs of very different
    lengths, most users empty): the candidate-tile ranges are weighted by the
    non-empty runs, found by a search over all users in several rounds."""
    rng = np.random.default_rng(31)
    active = np.sort(rng.choice(3000, size=20, replace=False))
    counts = rng.multinomial(700, rng.dirichlet(np.full(20, 0.5)))
    m = np.repeat(active, counts)
    rng.shuffle(m)
    x = gen.make_lce("empties", 32, 700, 3000, 40, 30, 136, 40, explicit_map=m.tolist())
    Y, st = run_lce(x)
    assert st == B.IKBO_OK
    ref = oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    assert_lce_close(Y, ref, "many empty users")


def test_lce_users_past_1024():
    """1 500 users with one candidate each: every candidate tile starts a
    run, and the range search takes two rounds of 32 probes."""
    m = np.random.default_rng(33).permutation(1500)
    x = gen.make_lce("runs", 34, 1500, 1500, 24, 40, 128, 32, explicit_map=m.tolist())
    Y, st = run_lce(x)
    assert st == B.IKBO_OK
    ref = oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    assert_lce_close(Y, ref, "users past 1024")


def test_lce_at_the_user_limit():
    """8 192 users (the segment builder's limit), 12 000 candidates in a
    permuted map: most users have one or two candidates, some none."""
    m = np.random.default_rng(35).integers(0, 8192, size=12000)
    x = gen.make_lce("umax", 36, 12000, 8192, 24, 40, 64, 16, explicit_map=m.tolist())
    Y, st = run_lce(x)
    assert st == B.IKBO_OK
    ref = oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    assert_lce_close(Y, ref, "8192 users")


@pytest.mark.parametrize("n_cand,ratio", [(n, r) for n, r, _ in gen.lce_sweep_points()])
def test_lce_sweep_point_full(n_cand, ratio):
    """Every point of the shape sweep (256 / 1024 / 4096 candidates x ratio
    10 / 70 / 1000 / 10000), every element of Y."""
    pts = {(n, r): s for n, r, s in gen.lce_sweep_points()}
    x = gen.lce_sweep(n_cand, ratio, pts[(n_cand, ratio)])
    Y, st = run_lce(x)
    assert st == B.IKBO_OK
    check_lce_all(Y, x)


def test_materialised_ablation_matches():
    """Our kernel fed the replicated user tensor (identity map, n_users = n_cand)
    gives the same Y as the broadcast form, up to rounding."""
    x = gen.make_lce("abl", 9, 96, 5, 40, 30, 128, 64, map_kind="permuted")
    Y1, st1 = run_lce(x)
    rep = gen.LCEInputs("rep", x.n_cand, x.n_cand, x.K_u, x.K_c, x.D, x.N,
                        torch.arange(x.n_cand, dtype=torch.int32), x.U[x.map.long()].contiguous(), x.C, x.Wu, x.Wc, x.b)
    Y2, st2 = run_lce(rep)
    assert st1 == st2 == B.IKBO_OK
    ref = oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    assert_lce_close(Y1, ref)
    assert_lce_close(Y2, ref)


def test_repeated_calls_and_replans_are_identical():
    x = gen.make_lce("rep", 13, 200, 9, 100, 80, 256, 96, map_kind="permuted")
    with B.Plan(400, 20, 1) as p:
        Y1, _ = run_lce(x, p)
        Y2, _ = run_lce(x, p)
        assert torch.equal(Y1, Y2)
        y = gen.make_lce("rep2", 14, 300, 20, 100, 80, 256, 96, map_kind="permuted")
        Y3, st = run_lce(y, p)
        assert st == B.IKBO_OK
        assert_lce_close(Y3, oracle.lce(y.map, y.U, y.C, y.Wu, y.Wc, y.b))


def test_map_out_of_range_skips_only_bad_candidates():
    x = gen.make_lce("oor", 21, 24, 3, 40, 30, 64, 16, map_kind="permuted")
    bad = x.map.clone()
    bad[5] = 3
    y = gen.LCEInputs("oor", x.n_cand, x.n_users, x.K_u, x.K_c, x.D, x.N, bad, x.U, x.C, x.Wu, x.Wc, x.b)
    Y, st = run_lce(y)
    assert st == B.IKBO_ERR_MAP_OUT_OF_RANGE
    good = [i for i in range(x.n_cand) if i != 5]
    assert_lce_close(Y[good], oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b, cands=good))
    assert torch.isnan(Y[5].float()).all()  # untouched


@pytest.mark.parametrize("schedule", [1, 2], ids=["two_launches", "one_launch"])
def test_forced_flag_timeout_still_gives_right_y(schedule):
    """Candidate epilogues wait on user partials that are never published
    (debug switch): the bounded wait gives up, the waiting tiles form the
    partial on the CUDA cores, Y is still right, the status says TIMEOUT, and
    the next normal call on the same context is right too (the flags were
    returned to zero)."""
    x = gen.make_lce("to", 31, 64, 4, 40, 30, 128, 32, map_kind="permuted")
    ref = oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    with B.Plan(64, 4, 1) as p:
        p.set_lce_schedule(schedule)  # the schedules that hand partials between CTAs
        B.ikbo_plan_set_timeout_ns(p.handle, 20_000_000)  # 20 ms
        B.ikbo_plan_set_debug(p.handle, B.DEBUG_WITHHOLD_USER_PARTIAL)
        Y, st = run_lce(x, p)
        assert st == B.IKBO_ERR_TIMEOUT
        assert_lce_close(Y, ref, "after the wait ran out")
        B.ikbo_plan_set_debug(p.handle, 0)
        for _ in range(2):
            Y, st = run_lce(x, p)
            assert st == B.IKBO_OK
            assert_lce_close(Y, ref, "next calls")


def test_argument_validation():
    x = gen.lce_tiny()
    U, C, Wu, Wc, b, m = to_dev(x.U, x.C, x.Wu, x.Wc, x.b, x.map)
    Y = torch.empty(16, 8, 32, dtype=torch.bfloat16, device="cuda")
    with B.Plan(16, 2, 1) as p:
        with pytest.raises(B.IkboError) as e:
            p.lce_forward(U, C, Wu, Wc, b, Y)
        assert e.value.code == B.IKBO_ERR_NOT_PLANNED
        p.plan(m, 2)
        L = B.load()
        # misaligned pointer
        rc = L.ikbo_lce_forward(p.handle, U.data_ptr() + 2, C.data_ptr(), Wu.data_ptr(), Wc.data_ptr(), b.data_ptr(),
                                Y.data_ptr(), 24, 16, 32, 8, None)
        assert rc == B.IKBO_ERR_INVALID_ARG
        # N not a multiple of 8, N > 256, D not a multiple of 8
        for (D, N) in [(32, 12), (32, 264), (30, 8)]:
            rc = L.ikbo_lce_forward(p.handle, U.data_ptr(), C.data_ptr(), Wu.data_ptr(), Wc.data_ptr(), None,
                                    Y.data_ptr(), 24, 16, D, N, None)
            assert rc == B.IKBO_ERR_UNSUPPORTED
        # Wc too large to stay resident (K_c 1024 x N 256)
        rc = L.ikbo_lce_forward(p.handle, U.data_ptr(), C.data_ptr(), Wu.data_ptr(), Wc.data_ptr(), None,
                                Y.data_ptr(), 24, 1024, 32, 256, None)
        assert rc == B.IKBO_ERR_UNSUPPORTED
        assert p.status() == B.IKBO_OK
