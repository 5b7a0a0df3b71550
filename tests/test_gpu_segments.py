"""Segment builder on the GPU: bit-exact against the oracle's counting sort."""
import numpy as np
import pytest
import torch

import oracle
from broadcast_gemm_attention_gb300 import binding as B
from broadcast_gemm_attention_gb300 import inputs as gen

pytestmark = pytest.mark.gpu


def _maps():
    rng = np.random.default_rng(123)
    yield "random", rng.integers(0, 7, size=300).astype(np.int32), 7
    yield "sorted_70to1", gen.lce_70to1_map().numpy(), 15
    yield "permuted", gen.permuted_multinomial_map(rng, 1024, 15), 15
    yield "zipf_stress", gen.zipf_permuted_map(np.random.default_rng(1004), 4096, 64, 1.1), 64
    yield "empty_users", np.array([5, 5, 0, 5, 2, 0], np.int32), 9
    yield "single_user", np.zeros(777, np.int32), 1
    yield "one_candidate", np.array([3], np.int32), 4
    yield "identity_4096", np.arange(4096, dtype=np.int32), 4096
    yield "many_users", rng.integers(0, 5000, size=2049).astype(np.int32), 5000
    # the few-user scatter's limit (32 users, several blocks of 1024) and one past it
    yield "users_32_blocks", gen.permuted_multinomial_map(rng, 3000, 32), 32
    yield "users_33_blocks", gen.permuted_multinomial_map(rng, 3000, 33), 33
    # the builder's user limit (8192, its counts and cursors in shared memory):
    # ~2.4 candidates per user, about 9 % of the users empty
    yield "max_users_8192", rng.integers(0, 8192, size=20000).astype(np.int32), 8192


@pytest.mark.parametrize("name,m,n_users", list(_maps()), ids=[x[0] for x in _maps()])
@pytest.mark.parametrize("H,Lq", [(8, 32), (3, 16), (1, 128), (2, 48)])
def test_segments_bit_exact(name, m, n_users, H, Lq):
    n = len(m)
    with B.Plan(n, n_users, H) as p:
        dmap = torch.from_numpy(m).cuda()
        p.plan(dmap, n_users, H, Lq)
        assert p.status() == B.IKBO_OK
        counts, offsets, perm = p.segments(n, n_users)
        work, cpu = p.worklist()
        assert cpu == 128 // Lq
        c, o, pm, w = oracle.segments(m, n_users, H, cpu)
        assert np.array_equal(counts.numpy(), c)
        assert np.array_equal(offsets.numpy(), o)
        assert np.array_equal(perm.numpy(), pm)
        assert np.array_equal(work.numpy(), w)


def test_replan_reuses_the_plan():
    with B.Plan(2000, 100, 8) as p:
        for seed in range(3):
            m = np.random.default_rng(seed).integers(0, 100, size=1500 + seed).astype(np.int32)
            p.plan(torch.from_numpy(m).cuda(), 100, 8, 32)
            counts, offsets, perm = p.segments(len(m), 100)
            c, o, pm, _ = oracle.segments(m, 100, 8, 8)
            assert np.array_equal(perm.numpy(), pm) and np.array_equal(offsets.numpy(), o)


def test_map_out_of_range_is_reported_not_trapped():
    m = np.array([0, 1, 7, 1, -2, 0], np.int32)
    with B.Plan(16, 4, 1) as p:
        p.plan(torch.from_numpy(m).cuda(), 4, 1, 8)
        assert p.status() == B.IKBO_ERR_MAP_OUT_OF_RANGE
        assert p.status() == B.IKBO_OK  # cleared by the read
        counts, offsets, perm = p.segments(len(m), 4)
        assert counts.tolist() == [2, 2, 0, 0] and offsets.tolist()[-1] == 4
        assert perm[:4].tolist() == [0, 5, 1, 3]


def test_plan_argument_errors():
    with B.Plan(8, 2, 2) as p:
        dmap = torch.zeros(16, dtype=torch.int32, device="cuda")
        with pytest.raises(B.IkboError) as e:
            p.plan(dmap, 2, 1, 8)  # n_cand above max_cand
        assert e.value.code == B.IKBO_ERR_INVALID_ARG
        with pytest.raises(B.IkboError) as e:
            p.plan(dmap[:4], 2, 1, 12)  # Lq not a multiple of 8
        assert e.value.code == B.IKBO_ERR_UNSUPPORTED
        with pytest.raises(B.IkboError) as e:
            p.plan(dmap[:4], 2, 3, 8)  # H above max_heads
        assert e.value.code == B.IKBO_ERR_INVALID_ARG


def test_plan_user_limit():
    """A plan for more users than the segment builder holds is refused
    before any allocation; one at the limit is accepted."""
    with pytest.raises(B.IkboError) as e:
        B.ikbo_plan_create(16, 8193, 1)
    assert e.value.code == B.IKBO_ERR_UNSUPPORTED
    h = B.ikbo_plan_create(16, 8192, 1)
    B.ikbo_plan_destroy(h)
