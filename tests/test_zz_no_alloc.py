"""ikbo_lce_forward_noalloc: the fused LCE for callers that must not allocate
device memory (their memory belongs to another allocator, or their request
path may not call cudaMalloc / cudaFree, which can synchronise the device).
It keeps its scratch in a fixed array inside the library.

Checked through the C ABI against ikbo_lce_forward (the plan-based entry
point) on two calls in a row, with the LCE tolerance used everywhere else:
|Y_noalloc - Y_plan| <= 1e-2 (1 + |Y_plan|); and both calls against the
fp64 oracle, every element.  The file is named so that pytest collects it
last; it also passes on its own in a fresh process (its first call then
performs the per-device set-up).
"""
import numpy as np
import pytest
import torch

from broadcast_gemm_attention_gb300 import binding as B
from broadcast_gemm_attention_gb300 import inputs as gen
from gpu_util import check_lce_all

pytestmark = pytest.mark.gpu

RTOL = 1e-2


def _dev(x):
    return [t.cuda() if t is not None else None for t in (x.map, x.U, x.C, x.Wu, x.Wc, x.b)]


def _plan_path(x):
    m, U, C, Wu, Wc, b = _dev(x)
    Y = torch.full((x.n_cand, x.N, x.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    with B.Plan(x.n_cand, x.n_users, 1) as p:
        p.plan(m, x.n_users)
        p.lce_forward(U, C, Wu, Wc, b, Y)
        assert p.status() == B.IKBO_OK
    return Y


def _noalloc_path(x):
    m, U, C, Wu, Wc, b = _dev(x)
    Y = torch.full((x.n_cand, x.N, x.D), float("nan"), dtype=torch.bfloat16, device="cuda")
    B.ikbo_lce_forward_noalloc(m, x.n_users, U, C, Wu, Wc, b, Y)
    torch.cuda.synchronize()
    return Y


def _close(y, ref, what):
    g = y.double().cpu().numpy()
    r = ref.double().cpu().numpy()
    assert np.all(np.isfinite(g)), what
    bad = np.abs(g - r) > RTOL * (1.0 + np.abs(r))
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance"


def test_noalloc_matches_plan_path_on_two_calls_in_a_row():
    a = gen.lce_70to1()                                                      # the 70:1 request
    b = gen.make_lce("noalloc_b", 4242, n_cand=300, n_users=7, K_u=101, K_c=77, D=136, N=40,
                     map_kind="permuted")                                    # ragged shapes, other map
    ref_a, ref_b = _plan_path(a), _plan_path(b)
    y_a = _noalloc_path(a)   # first call (per-device set-up when run alone); two launches
    y_b = _noalloc_path(b)   # second call reuses the scratch left by the first; one launch
    _close(y_a, ref_a, "first call")
    _close(y_b, ref_b, "second call")
    check_lce_all(y_a, a, what="no-alloc 70:1", cache_key="lce_70to1")
    check_lce_all(y_b, b, what="no-alloc ragged")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    x = gen.lce_tiny()
    m, U, C, Wu, Wc, b = _dev(x)
    Y = torch.empty(x.n_cand, x.N, x.D, dtype=torch.bfloat16, device="cuda")
    L = B.load()
    # 100 users x N 256 x D 256 fp32 partials = 26 MB > 16 MiB: rejected before any launch
    rc = L.ikbo_lce_forward_noalloc(m.data_ptr(), 16, 100, U.data_ptr(), C.data_ptr(), Wu.data_ptr(),
                                    Wc.data_ptr(), None, Y.data_ptr(), 24, 16, 256, 256, None)
    assert rc == B.IKBO_ERR_UNSUPPORTED
    rc = L.ikbo_lce_forward_noalloc(None, 16, 2, U.data_ptr(), C.data_ptr(), Wu.data_ptr(), Wc.data_ptr(),
                                    None, Y.data_ptr(), 24, 16, 32, 8, None)
    assert rc == B.IKBO_ERR_INVALID_ARG
