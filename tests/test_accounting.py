"""FLOP/byte accounting (used for every roofline fraction) against the
figures the IKBO pages print."""
import json
import os

from broadcast_gemm_attention_gb300 import accounting as acc
from broadcast_gemm_attention_gb300 import inputs as gen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_attention_intensity_reproduces_printed_figures():
    g = json.load(open(os.path.join(GOLDEN, "attn_intensity.json")))
    Lq, Lkv, r = g["reading_Lq"], g["printed"]["sequence_length"], g["printed"]["ratio"]
    assert round(acc.attn_intensity_standard(Lq, Lkv)) == g["printed"]["standard_flop_per_byte"]
    assert round(acc.attn_intensity_ikbo(Lq, Lkv, r)) == g["printed"]["ikbo_flop_per_byte"]
    # the closed forms agree with the explicit FLOP and byte counts
    d, H = 128, 1
    fl = acc.attn_flops(H, Lq, d, [Lkv] * r)
    by = acc.attn_bytes(r, H, Lq, d, Lkv) - 4 * r          # drop the map bytes
    assert abs(fl / by - acc.attn_intensity_ikbo(Lq, Lkv, r)) < 1e-9
    fl1 = acc.attn_flops(H, Lq, d, [Lkv])
    by1 = acc.attn_bytes(1, H, Lq, d, Lkv) - 4
    assert abs(fl1 / by1 - acc.attn_intensity_standard(Lq, Lkv)) < 1e-9


def test_lce_stage_figures_are_consistent():
    """The printed per-stage reductions follow from the printed latencies, and
    15 users x ~70 = 1024 candidates (user work cut by > 98%)."""
    g = json.load(open(os.path.join(GOLDEN, "lce_stage_latencies.json")))
    t = g["latency_ms"]
    red = g["printed_reduction_percent"]
    # the pages print one decimal; 0.580/0.798 gives 27.3, printed 27.4
    assert abs(100 * (1 - t["stage1_decomposition"] / t["baseline"]) - red["stage1"]) < 0.1
    assert abs(100 * (1 - t["stage2_pad_k"] / t["stage1_decomposition"]) - red["stage2"]) < 0.1
    assert abs(100 * (1 - t["stage3_epilogue_fusion"] / t["stage2_pad_k"]) - red["stage3"]) < 0.1
    assert round(t["baseline"] / t["stage4_warp_specialised"]) == g["printed_total_speedup"]
    # "about 15 users" replicated "about 70 times" onto 1024 candidates
    assert abs(g["candidates_per_request"] / g["users_per_request"] - g["printed_ratio"]) < 3
    assert 1 - g["users_per_request"] / g["candidates_per_request"] > 0.98


def test_lce_counts_at_70to1():
    c = gen.LCE_70
    f = acc.lce_flops(**c)
    b = acc.lce_bytes(**c)
    assert abs(f - 25.022988288e9) < 1
    # U 2.93 MB + C 127.4 MB + W 0.24 MB + b + map + Y 100.66 MB
    assert abs(b / 1e6 - 231.235456) < 1e-6
    assert acc.lce_materialised_flops(c["n_cand"], c["K_u"], c["K_c"], c["D"], c["N"]) > 2 * f


def test_attention_counts_at_70to1():
    c = gen.ATTN_70
    f = acc.attn_flops(c["H"], c["Lq"], c["d"], [c["Lkv"]] * c["n_cand"])
    assert abs(f - 4 * 1024 * 8 * 32 * 2048 * 128) < 1
    b = acc.attn_bytes(c["n_cand"], c["H"], c["Lq"], c["d"], c["n_users"] * c["Lkv"])
    assert abs(b / 1e6 - 260.05) < 0.1


def test_lce_backward_counts_at_70to1():
    """The backward's products: twice the forward's FLOPs (each forward GEMM has
    a data-gradient and a weight-gradient product); bytes counted by hand."""
    fl = acc.lce_backward_flops(1024, 15, 381, 243, 256, 192)
    assert fl == 2 * acc.lce_flops(1024, 15, 381, 243, 256, 192)
    assert abs(fl - 50.046e9) < 0.01e9
    dY = 1024 * 192 * 256 * 2
    inputs = (15 * 381 * 256 + 1024 * 243 * 256 + 381 * 192 + 243 * 192) * 2 + 1024 * 4
    outputs = (15 * 381 * 256 + 1024 * 243 * 256) * 2 + (381 * 192 + 243 * 192 + 192) * 4
    assert acc.lce_backward_bytes(1024, 15, 381, 243, 256, 192) == dY + inputs + outputs


def test_attention_backward_counts():
    """Five products of 2*Lq*L*d multiply-adds each (S, dP, dV, dK, dQ) per
    (candidate, head), and every tensor of the backward moved once."""
    H, Lq, d, L = 8, 32, 128, 2048
    lens = [L] * 70
    assert acc.attn_backward_flops(H, Lq, d, lens) == 5 * 2 * 2 * Lq * L * d * H * 70 / 2
    assert acc.attn_backward_flops(H, Lq, d, lens) == 2.5 * acc.attn_flops(H, Lq, d, lens)
    # Q, O, dO in and dQ out per candidate; K, V in and dK, dV out per user
    by = acc.attn_backward_bytes(70, H, Lq, d, L)
    assert by == 2 * (4 * 70 * H * Lq * d + 4 * L * H * d) + 4 * 70
    assert by - 4 * 70 == 2 * (acc.attn_bytes(70, H, Lq, d, L) - 4 * 70)
