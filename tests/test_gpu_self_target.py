"""Self + target attention in one launch (ikbo_attn_self_target_forward)
against the fp64 oracle.

The target rows must equal ikbo_attn_forward's bit for bit (same kernel
path and the same order of units per CTA); the users' own rows, fused or
alone, are ordinary attention of Q_user[u]
against K[u], V[u], i.e. the oracle with the identity map over users.
Tolerance: |O_gpu - O_ref| <= 2e-2 element-wise.
"""
import pytest
import torch

import oracle
from broadcast_gemm_attention_gb300 import binding as B
from broadcast_gemm_attention_gb300 import inputs as gen
from gpu_util import assert_attn_close, check_attn_all, to_dev

pytestmark = pytest.mark.gpu


def run_both(x, Q_user, scale=None):
    Q, K, V, m, Qu = to_dev(x.Q, x.K, x.V, x.map, Q_user)
    offs = None if x.kv_offsets is None else x.kv_offsets.cuda()
    O_sep = torch.full_like(Q, float("nan"))
    O = torch.full_like(Q, float("nan"))
    O_user = torch.full_like(Qu, float("nan"))
    O_user_alone = torch.full_like(Qu, float("nan"))
    with B.Plan(x.n_cand, x.n_users, x.H) as p:
        p.plan(m, x.n_users, x.H, x.Lq)
        p.attn_forward(Q, K, V, offs, O_sep, scale)
        l0 = p.launches()
        p.attn_self_target_forward(Q, Qu, K, V, offs, O, O_user, scale)
        launched = p.launches() - l0
        p.attn_self_target_forward(None, Qu, K, V, offs, None, O_user_alone, scale)  # the self part alone
        st = p.status()
    return O, O_user, O_sep, st, launched, O_user_alone


def check(x, Lq_u, seed, scale=None):
    Q_user = gen.make_user_queries(seed, x.n_users, x.H, Lq_u, x.d)
    O, O_user, O_sep, st, launched, O_alone = run_both(x, Q_user, scale)
    assert st == B.IKBO_OK
    assert launched == 1
    assert torch.equal(O, O_sep), "target rows differ from ikbo_attn_forward"
    ref = oracle.attn(x.map, x.Q, x.K, x.V, kv_offsets=x.kv_offsets, n_users=x.n_users, scale=scale)
    assert_attn_close(O, ref.reshape(O.shape), x.name + " target")
    ident = torch.arange(x.n_users, dtype=torch.int32)
    ref_u = oracle.attn(ident, Q_user, x.K, x.V, kv_offsets=x.kv_offsets, n_users=x.n_users, scale=scale)
    assert_attn_close(O_user, ref_u.reshape(O_user.shape), x.name + " self")
    assert_attn_close(O_alone, ref_u.reshape(O_user.shape), x.name + " self part alone")


@pytest.mark.parametrize("Lq_u", [8, 40, 128, 200])
def test_self_target_dense(Lq_u):
    """One self tile (8, 40, 128 rows) and two (200 = 128 + 72, ragged)."""
    x = gen.make_attn("st_dense", 71, n_cand=37, n_users=5, H=2, Lq=16, d=128, Lkv=300, map_kind="permuted")
    check(x, Lq_u, 80 + Lq_u)


def test_self_target_jagged_with_empty_user():
    lens = [200, 0, 129, 1, 384]
    x = gen.make_attn("st_jag", 72, n_cand=30, n_users=5, H=2, Lq=32, d=128, map_kind="permuted",
                      explicit_lengths=lens)
    check(x, 48, 90)
    check(x, 48, 91, scale=0.3)


def test_self_target_70to1_full():
    """The 70:1 request plus 64 user queries per (user, head); every row."""
    x = gen.attn_70to1()
    Q_user = gen.make_user_queries(92, x.n_users, x.H, 64, x.d)
    O, O_user, O_sep, st, launched, O_alone = run_both(x, Q_user)
    assert st == B.IKBO_OK and launched == 1
    assert torch.equal(O, O_sep)
    check_attn_all(O, x, what="70:1 target", cache_key="attn_70to1")
    ident = torch.arange(x.n_users, dtype=torch.int32)
    ref_u = oracle.attn(ident, Q_user, x.K, x.V).reshape(O_user.shape)
    assert_attn_close(O_user, ref_u, "70:1 self")
    assert_attn_close(O_alone, ref_u, "70:1 self part alone")


def test_self_target_argument_validation():
    x = gen.make_attn("st_val", 73, n_cand=8, n_users=2, H=1, Lq=8, d=128, Lkv=64)
    Q, K, V, m = to_dev(x.Q, x.K, x.V, x.map)
    O = torch.empty_like(Q)
    with B.Plan(x.n_cand, x.n_users, x.H) as p:
        p.plan(m, x.n_users, x.H, x.Lq)
        Qu = torch.zeros(2, 1, 12, 128, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(B.IkboError) as e:
            p.attn_self_target_forward(Q, Qu, K, V, None, O, torch.empty_like(Qu))
        assert e.value.code == B.IKBO_ERR_UNSUPPORTED
        rc = B.load().ikbo_attn_self_target_forward(p.handle, Q.data_ptr(), None, K.data_ptr(), V.data_ptr(), None,
                                                    O.data_ptr(), None, 16, 64, 128, 0.1, None)
        assert rc == B.IKBO_ERR_INVALID_ARG
        Qu = torch.zeros(2, 1, 16, 128, dtype=torch.bfloat16, device="cuda")
        Ou = torch.empty_like(Qu)
        # Q without O (or O without Q) is an error; neither is the self part alone
        rc = B.load().ikbo_attn_self_target_forward(p.handle, Q.data_ptr(), Qu.data_ptr(), K.data_ptr(), V.data_ptr(),
                                                    None, None, Ou.data_ptr(), 16, 64, 128, 0.1, None)
        assert rc == B.IKBO_ERR_INVALID_ARG
        rc = B.load().ikbo_attn_self_target_forward(p.handle, None, Qu.data_ptr(), K.data_ptr(), V.data_ptr(),
                                                    None, O.data_ptr(), Ou.data_ptr(), 16, 64, 128, 0.1, None)
        assert rc == B.IKBO_ERR_INVALID_ARG
        assert p.status() == B.IKBO_OK
