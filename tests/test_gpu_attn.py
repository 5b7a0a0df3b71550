"""Broadcast attention on the GPU against the fp64 oracle.

Tolerance: |O_gpu - O_ref| <= 2e-2 element-wise.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from broadcast_gemm_attention_gb300 import binding as B
from broadcast_gemm_attention_gb300 import inputs as gen
from gpu_util import assert_attn_close, check_attn_all, to_dev

pytestmark = pytest.mark.gpu


def run_attn(x, plan=None, scale=None):
    Q, K, V, m = to_dev(x.Q, x.K, x.V, x.map)
    offs = None if x.kv_offsets is None else x.kv_offsets.cuda()
    O = torch.full_like(Q, float("nan"))
    own = plan is None
    p = plan or B.Plan(x.n_cand, x.n_users, x.H)
    try:
        p.plan(m, x.n_users, x.H, x.Lq)
        p.attn_forward(Q, K, V, offs, O, scale)
        st = p.status()
    finally:
        if own:
            p.close()
    return O, st


def full_check(x, scale=None):
    O, st = run_attn(x, scale=scale)
    assert st == B.IKBO_OK
    ref = oracle.attn(x.map, x.Q, x.K, x.V, kv_offsets=x.kv_offsets, n_users=x.n_users, scale=scale)
    ref = ref.reshape(x.n_cand, x.H, x.Lq, x.d)
    return assert_attn_close(O, ref, x.name)


@pytest.mark.parametrize("Lq", [8, 16, 32, 48, 128])
@pytest.mark.parametrize("map_kind", ["sorted", "permuted"])
def test_attn_dense_small(Lq, map_kind):
    """Ragged key tail (300 = 2 x 128 + 44), several users, partial units."""
    x = gen.make_attn("dense", 41 + Lq, n_cand=37, n_users=5, H=2, Lq=Lq, d=128, Lkv=300, map_kind=map_kind)
    full_check(x)


@pytest.mark.parametrize("Lkv", [1, 127, 128, 129, 1000])
def test_attn_key_lengths(Lkv):
    x = gen.make_attn("len", 50, n_cand=12, n_users=3, H=1, Lq=16, d=128, Lkv=Lkv, map_kind="permuted")
    full_check(x)


def test_attn_jagged_with_empty_and_tiny_users():
    lens = [200, 0, 1, 129, 384, 77]
    x = gen.make_attn("jag", 60, n_cand=50, n_users=6, H=2, Lq=16, d=128, map_kind="permuted",
                      explicit_lengths=lens)
    full_check(x)


def test_attn_identity_map_and_single_user():
    x = gen.make_attn("id", 61, n_cand=9, n_users=9, H=2, Lq=32, d=128, Lkv=256,
                      explicit_map=list(range(9)))
    full_check(x)
    y = gen.make_attn("mqa", 62, n_cand=40, n_users=1, H=3, Lq=32, d=128, Lkv=520, explicit_map=[0] * 40)
    full_check(y)


def test_attn_large_scores_exercise_rescaling():
    """Scores spread over tens of units and the max growing across key tiles:
    the lazy rescale of O must still give the exact softmax."""
    x = gen.make_attn("big", 63, n_cand=20, n_users=2, H=1, Lq=16, d=128, Lkv=1024, map_kind="permuted")
    ramp = torch.linspace(0.2, 3.0, 1024).view(1, 1, 1024, 1)
    K = (x.K.float() * ramp).to(torch.bfloat16)
    Q = (x.Q.float() * 2.0).to(torch.bfloat16)
    y = gen.AttnInputs("big", x.n_cand, x.n_users, x.H, x.Lq, x.Lkv, x.d, x.map, Q, K, x.V)
    full_check(y)
    full_check(y, scale=0.5)


def test_attn_70to1_full():
    """The 70:1 workload in the benchmark's launch configuration; every
    (candidate, head) of O against the oracle."""
    x = gen.attn_70to1()
    O, st = run_attn(x)
    assert st == B.IKBO_OK
    check_attn_all(O, x, what="70:1", cache_key="attn_70to1")


def test_attn_stress_jagged_zipf_full():
    """4096 candidates of 64 users (Zipf counts, permuted map) over jagged
    histories of 256-4096 keys; every (candidate, head)."""
    x = gen.attn_stress()
    O, st = run_attn(x)
    assert st == B.IKBO_OK
    check_attn_all(O, x, what="stress")


@pytest.mark.parametrize("ratio", list(gen.SWEEP_RATIO))
def test_attn_ratio_sweep_full(ratio):
    """The ratio sweep at 4096 candidates (410 / 59 / 4 / 1 users), every (candidate, head)."""
    n, r, seed = [t for t in gen.attn_ratio_sweep_points() if t[1] == ratio][0]
    x = gen.attn_ratio_sweep(n, r, seed)
    O, st = run_attn(x)
    assert st == B.IKBO_OK
    check_attn_all(O, x)


def test_attn_runs_of_every_length_per_user():
    """Users whose runs of candidates end in a partial unit, fill units
    exactly, or have a single candidate (Lq 32: 4 candidates per unit;
    counts 1, 5, 8, 13, 20), over three heads."""
    m = [0] * 1 + [1] * 5 + [2] * 8 + [3] * 13 + [4] * 20
    x = gen.make_attn("runs", 67, n_cand=len(m), n_users=5, H=3, Lq=32, d=128, Lkv=260, explicit_map=m)
    full_check(x)


def test_attn_at_the_user_limit():
    """8 192 users (the segment builder's limit) with 1-3 candidates each over
    short dense histories (Lkv 130: a full and a 2-key tile), Lq 16."""
    rng = np.random.default_rng(68)
    m = rng.integers(0, 8192, size=12000).tolist()
    x = gen.make_attn("umax", 69, n_cand=len(m), n_users=8192, H=1, Lq=16, d=128, Lkv=130, explicit_map=m)
    full_check(x)


def test_attn_materialised_ablation_matches():
    x = gen.make_attn("abl", 64, n_cand=24, n_users=3, H=2, Lq=32, d=128, Lkv=256, map_kind="permuted")
    idx = x.map.long()
    rep = gen.AttnInputs("rep", x.n_cand, x.n_cand, x.H, x.Lq, x.Lkv, x.d, torch.arange(x.n_cand, dtype=torch.int32),
                         x.Q, x.K[idx].contiguous(), x.V[idx].contiguous())
    O1, s1 = run_attn(x)
    O2, s2 = run_attn(rep)
    assert s1 == s2 == B.IKBO_OK
    ref = oracle.attn(x.map, x.Q, x.K, x.V).reshape(x.n_cand, x.H, x.Lq, x.d)
    assert_attn_close(O1, ref)
    assert_attn_close(O2, ref)


def test_attn_argument_validation():
    x = gen.make_attn("v", 65, n_cand=4, n_users=2, H=1, Lq=16, d=128, Lkv=64, map_kind="sorted")
    Q, K, V, m = to_dev(x.Q, x.K, x.V, x.map)
    O = torch.empty_like(Q)
    with B.Plan(4, 2, 1) as p:
        with pytest.raises(B.IkboError) as e:
            p.attn_forward(Q, K, V, None, O)
        assert e.value.code == B.IKBO_ERR_NOT_PLANNED
        p.plan(m, 2, 1, 16)
        L = B.load()
        rc = L.ikbo_attn_forward(p.handle, Q.data_ptr(), K.data_ptr(), V.data_ptr(), None, O.data_ptr(), 64, 64,
                                 0.125, None)
        assert rc == B.IKBO_ERR_UNSUPPORTED  # d != 128
        rc = L.ikbo_attn_forward(p.handle, Q.data_ptr() + 8, K.data_ptr(), V.data_ptr(), None, O.data_ptr(), 64, 128,
                                 0.125, None)
        assert rc == B.IKBO_ERR_INVALID_ARG  # misaligned
        rc = L.ikbo_attn_forward(p.handle, Q.data_ptr(), K.data_ptr(), V.data_ptr(), None, O.data_ptr(), 64, 128,
                                 -1.0, None)
        assert rc == B.IKBO_ERR_INVALID_ARG  # bad scale
        assert p.status() == B.IKBO_OK
