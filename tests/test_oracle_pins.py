"""The oracle against its pins (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from oracle_pins import ATTN_BWD_PINS, ATTN_LSE_PINS, ATTN_PINS, LCE_BWD_PINS, LCE_PINS, SEG_PINS
from broadcast_gemm_attention_gb300 import inputs as gen


@pytest.mark.parametrize("pin", LCE_PINS, ids=lambda f: f.__name__)
def test_lce_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("pin", LCE_BWD_PINS, ids=lambda f: f.__name__)
def test_lce_backward_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("pin", ATTN_BWD_PINS, ids=lambda f: f.__name__)
def test_attn_backward_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("pin", ATTN_PINS, ids=lambda f: f.__name__)
def test_attn_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("pin", ATTN_LSE_PINS, ids=lambda f: f.__name__)
def test_attn_lse_pin(orc, pin):
    pin(orc)


@pytest.mark.parametrize("pin", SEG_PINS, ids=lambda f: f.__name__)
def test_segments_pin(orc, pin):
    pin(orc)


def test_map_out_of_range_is_an_error(orc):
    x = gen.lce_tiny()
    bad = x.map.clone()
    bad[3] = 2
    with pytest.raises(oracle.OracleError, match="out of range"):
        orc.lce(bad, x.U, x.C, x.Wu, x.Wc, x.b)
    with pytest.raises(oracle.OracleError, match="out of range"):
        orc.segments(np.array([0, -1], np.int32), 2)
    a = gen.make_attn("e", 1, 2, 2, 1, 2, 16, Lkv=3, explicit_map=[0, 1])
    with pytest.raises(oracle.OracleError, match="out of range"):
        orc.attn(torch.tensor([0, 5], dtype=torch.int32), a.Q, a.K, a.V)


def test_tiny_config_shapes_and_scale(orc):
    """The tiny LCE workload: Y is [16, 8, 32] and O(1) (W ~ N(0, 1/40))."""
    x = gen.lce_tiny()
    Y = orc.lce(x.map, x.U, x.C, x.Wu, x.Wc, x.b)
    assert Y.shape == (16, 8, 32)
    assert 0.3 < Y.std() < 3.0
    assert x.map.tolist() == [0] * 8 + [1] * 8
