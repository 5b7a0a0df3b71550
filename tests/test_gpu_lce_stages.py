"""The pages' LCE stage ladder (ikbo_lce_forward_staged) against the fp64
oracle: stage 1 (decomposed, unfused: separate broadcast-add launch),
stage 3 (fused epilogue, one accumulator), stage 4 (the full kernel).

Tolerance: |Y_gpu - Y_ref| <= 1e-2 (1 + |Y_ref|) element-wise.  Stages 3
and 4 do the same arithmetic in another schedule, so they agree bit for bit.
"""
import pytest
import torch

import oracle
from broadcast_gemm_attention_gb300 import binding as B
from broadcast_gemm_attention_gb300 import inputs as gen
from gpu_util import assert_lce_close, check_lce_all, sample_candidates, to_dev

pytestmark = pytest.mark.gpu


def run_stages(x, stages=(1, 3, 4), schedule=1):
    U, C, Wu, Wc, b, m = to_dev(x.U, x.C, x.Wu, x.Wc, x.b, x.map)
    out, launches = {}, {}
    with B.Plan(x.n_cand, x.n_users, 1) as p:
        p.set_lce_schedule(schedule)
        p.plan(m, x.n_users)
        for st in stages:
            Y = torch.full((x.n_cand, x.N, x.D), float("nan"), dtype=torch.bfloat16, device="cuda")
            l0 = p.launches()
            p.lce_forward_staged(U, C, Wu, Wc, b, Y, st)
            launches[st] = p.launches() - l0
            assert p.status() == B.IKBO_OK
            out[st] = Y
    return out, launches


@pytest.mark.parametrize("shape", [
    dict(n_cand=16, n_users=2, K_u=24, K_c=16, D=32, N=8),
    dict(n_cand=37, n_users=3, K_u=37, K_c=29, D=136, N=40),
    dict(n_cand=300, n_users=7, K_u=381, K_c=243, D=384, N=200),
])
@pytest.mark.parametrize("schedule", [1, 2])
def test_lce_stages_full(shape, schedule):
    x = gen.make_lce("stages", 81, map_kind="permuted", **shape)
    out, launches = run_stages(x, schedule=schedule)
    assert launches == ({1: 3, 3: 2, 4: 2} if schedule == 1 else {1: 2, 3: 1, 4: 1})
    ref = oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    for st, Y in out.items():
        assert_lce_close(Y, ref, f"stage {st}")
    assert torch.equal(out[3], out[4])


def test_lce_stages_70to1_full():
    """Every stage at the 70:1 request shape, every element of Y."""
    x = gen.lce_70to1()
    out, _ = run_stages(x)
    for st, Y in out.items():
        check_lce_all(Y, x, what=f"70:1 stage {st}", cache_key="lce_70to1")
    assert torch.equal(out[3], out[4])


def test_lce_stage_argument_and_map_errors():
    x = gen.make_lce("stage_err", 82, 12, 3, 16, 16, 32, 16)
    U, C, Wu, Wc, b = to_dev(x.U, x.C, x.Wu, x.Wc, x.b)
    Y = torch.empty((x.n_cand, x.N, x.D), dtype=torch.bfloat16, device="cuda")
    bad = x.map.clone()
    bad[5] = 7
    with B.Plan(x.n_cand, x.n_users, 1) as p:
        m = bad.cuda()  # borrowed by the plan for the calls below
        p.plan(m, x.n_users)
        for st in (0, 2, 5):
            with pytest.raises(B.IkboError) as e:
                p.lce_forward_staged(U, C, Wu, Wc, b, Y, st)
            assert e.value.code == B.IKBO_ERR_INVALID_ARG
        p.lce_forward_staged(U, C, Wu, Wc, b, Y, 1)
        assert p.status() == B.IKBO_ERR_MAP_OUT_OF_RANGE


@pytest.mark.parametrize("shape", [
    dict(n_cand=256, n_users=26, K_u=381, K_c=243, D=256, N=192),
    dict(n_cand=1024, n_users=15, K_u=381, K_c=243, D=256, N=192),
    dict(n_cand=64, n_users=1, K_u=700, K_c=100, D=256, N=192),
    dict(n_cand=200, n_users=9, K_u=100, K_c=60, D=200, N=104),
    dict(n_cand=120, n_users=5, K_u=381, K_c=243, D=256, N=200),  # N > 192: no local partials
])
def test_lce_schedules_agree(shape):
    """Two launches, one launch and local partials do the same arithmetic per
    element: identical Y; the automatic choice is one of them.  A request
    for local partials where they do not apply runs as the automatic one."""
    x = gen.make_lce("sched", 83, map_kind="permuted", **shape)
    U, C, Wu, Wc, b, m = to_dev(x.U, x.C, x.Wu, x.Wc, x.b, x.map)
    ys, launched = {}, {}
    with B.Plan(x.n_cand, x.n_users, 1) as p:
        p.plan(m, x.n_users)
        for sch in (0, 1, 2, 3):
            p.set_lce_schedule(sch)
            Y = torch.full((x.n_cand, x.N, x.D), float("nan"), dtype=torch.bfloat16, device="cuda")
            l0 = p.launches()
            p.lce_forward(U, C, Wu, Wc, b, Y)
            launched[sch] = p.launches() - l0
            assert p.status() == B.IKBO_OK
            ys[sch] = Y
        for bad in (-1, 4):
            with pytest.raises(B.IkboError):
                p.set_lce_schedule(bad)
    assert launched[1] == 2 and launched[2] == 1 and launched[3] in (1, launched[0])
    assert torch.equal(ys[1], ys[2])
    assert torch.equal(ys[3], ys[1])
    assert torch.equal(ys[0], ys[1])
    assert_lce_close(ys[3], oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b), "local partials")


@pytest.mark.parametrize("schedule", [1, 2, 3])
def test_lce_schedules_map_out_of_range(schedule):
    """A map value out of range: that candidate's rows stay untouched, the
    status says so, and the candidates around it (same user before and after)
    are still right -- in the local-partial schedule the bad candidate must
    not disturb the partial its neighbours share."""
    x = gen.make_lce("sched_oor", 84, 300, 4, 381, 243, 256, 192)
    bad = x.map.clone()
    order = torch.argsort(x.map, stable=True)
    hits = [int(order[k]) for k in (0, 37, 150, 299)]
    for i in hits:
        bad[i] = 4 if i % 2 else -3
    U, C, Wu, Wc, b, m = to_dev(x.U, x.C, x.Wu, x.Wc, x.b, bad)
    Y = torch.full((x.n_cand, x.N, x.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    with B.Plan(x.n_cand, x.n_users, 1) as p:
        p.set_lce_schedule(schedule)
        p.plan(m, x.n_users)
        p.lce_forward(U, C, Wu, Wc, b, Y)
        assert p.status() == B.IKBO_ERR_MAP_OUT_OF_RANGE
    for i in hits:
        assert torch.isnan(Y[i].float()).all()
    good = [i for i in range(x.n_cand) if i not in hits]
    sel = sorted(set(good[:8] + good[-8:] + [int(order[k]) for k in (1, 36, 38, 149, 151, 298)]))
    assert_lce_close(Y[sel], oracle.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b, cands=sel), f"schedule {schedule}")
