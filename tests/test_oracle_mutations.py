"""Plant plausible mistakes in copies of the oracle's C source and check that
the pins catch every one (a pin that a planted mistake slips past is a pin
that would not catch that mistake in the real oracle either)."""
import os

import pytest

import oracle
from oracle_pins import ATTN_BWD_PINS, ATTN_LSE_PINS, ATTN_PINS, LCE_BWD_PINS, LCE_PINS, SEG_PINS

MUTATIONS = {
    # LCE
    "lce_drop_bias": ("double bias = b ? bf16_bits_to_double(b[n]) : 0.0;", "double bias = 0.0;", LCE_PINS),
    "lce_user_index_is_candidate": ("int u = map[i];\n            /* the broadcast", "int u = i % n_users;\n            /* the broadcast", LCE_PINS),
    "lce_drop_last_k": ("for (int k = 0; k < K; ++k) acc +=", "for (int k = 0; k < K - 1; ++k) acc +=", LCE_PINS),
    "lce_sign_flip": ("acc += W[(size_t)k * N + n] * X", "acc -= W[(size_t)k * N + n] * X", LCE_PINS),
    "lce_transposed_w": ("W[(size_t)(K_u + k) * N + n] = bf16_bits_to_double(Wc[(size_t)k * N + n]);",
                         "W[(size_t)(K_u + k) * N + n] = bf16_bits_to_double(Wc[((size_t)k * N + n) % ((size_t)K_c * N) / K_c + ((size_t)k * N + n) % K_c * N]);", LCE_PINS),
    "lce_user_rows_from_candidate": ("X[(size_t)k * D + d] = bf16_bits_to_double(U[((size_t)u * K_u + k) * D + d]);",
                                     "X[(size_t)k * D + d] = bf16_bits_to_double(U[((size_t)(u ? 0 : u) * K_u + k) * D + d]);", LCE_PINS),
    # LCE backward
    "bwd_dc_uses_wu": ("acc += bf16_bits_to_double(Wc[(size_t)k * N + n]) *\n                           bf16_bits_to_double(dY[((size_t)i * N + n) * D + d]);\n                dC",
                       "acc += bf16_bits_to_double(Wu[(size_t)k * N + n]) *\n                           bf16_bits_to_double(dY[((size_t)i * N + n) * D + d]);\n                dC", LCE_BWD_PINS),
    "bwd_du_every_candidate": ("if (map[i] != u) continue;", "if (map[i] < 0) continue;", LCE_BWD_PINS),
    "bwd_dw_user_rows_not_broadcast": ("const uint16_t *xrow = k < K_u ? U + ((size_t)map[i] * K_u + k) * D",
                                       "const uint16_t *xrow = k < K_u ? U + ((size_t)(i % n_users) * K_u + k) * D", LCE_BWD_PINS),
    "bwd_db_drop_last_d": ("for (int d = 0; d < D; ++d) acc += bf16_bits_to_double(dY[((size_t)i * N + n) * D + d]);",
                           "for (int d = 0; d < D - 1; ++d) acc += bf16_bits_to_double(dY[((size_t)i * N + n) * D + d]);", LCE_BWD_PINS),
    "bwd_dwc_sign": ("dWc[(size_t)(k - K_u) * N + n] = acc;", "dWc[(size_t)(k - K_u) * N + n] = -acc;", LCE_BWD_PINS),
    "bwd_dc_drop_last_n": ("for (int n = 0; n < N; ++n)\n                    acc += bf16_bits_to_double(Wc",
                           "for (int n = 0; n < N - 1; ++n)\n                    acc += bf16_bits_to_double(Wc", LCE_BWD_PINS),
    # attention backward
    "abwd_no_D": ("for (int j = 0; j < L; ++j) ds[j] = p[j] * (ds[j] - D);", "for (int j = 0; j < L; ++j) ds[j] = p[j] * ds[j];", ATTN_BWD_PINS),
    "abwd_dq_no_scale": ("for (int c = 0; c < d; ++c) out[c] += scale * ds[j] * bf16_bits_to_double(kr[c]);",
                         "for (int c = 0; c < d; ++c) out[c] += ds[j] * bf16_bits_to_double(kr[c]);", ATTN_BWD_PINS),
    "abwd_dk_from_dO": ("gk[(size_t)j * d + c] += scale * ds[j] * bf16_bits_to_double(qr[c]);",
                        "gk[(size_t)j * d + c] += scale * ds[j] * bf16_bits_to_double(gr[c]);", ATTN_BWD_PINS),
    "abwd_dv_uses_ds": ("gv[(size_t)j * d + c] += p[j] * bf16_bits_to_double(gr[c]);",
                        "gv[(size_t)j * d + c] += ds[j] * bf16_bits_to_double(gr[c]);", ATTN_BWD_PINS),
    "abwd_dkdv_every_candidate": ("if (map[i] != u || L == 0) continue;", "if (L == 0) continue;", ATTN_BWD_PINS),
    "abwd_dp_from_k": ("const uint16_t *vr = V + row0 + (size_t)j * row_stride;\n        double dp",
                       "const uint16_t *vr = K + row0 + (size_t)j * row_stride;\n        double dp", ATTN_BWD_PINS),
    # attention
    "attn_no_scale": ("sc[j] = scale * dot;", "sc[j] = dot;", ATTN_PINS),
    "attn_no_normalise": ("for (int c = 0; c < d; ++c) orow[c] /= l;", "", ATTN_PINS),
    "attn_v_from_k": ("const uint16_t *vrow = V + row0", "const uint16_t *vrow = K + row0", ATTN_PINS),
    "attn_user_is_candidate": ("int h = pairs ? pairs[2 * s + 1] : s % H;\n            int u = map[i];\n            int L;",
                               "int h = pairs ? pairs[2 * s + 1] : s % H;\n            int u = i % n_users;\n            int L;", ATTN_PINS),
    "attn_drop_last_key": ("for (int j = 0; j < L; ++j) {\n                    const uint16_t *vrow", "for (int j = 0; j < L - 1; ++j) {\n                    const uint16_t *vrow", ATTN_PINS),
    "attn_jagged_stride": ("row_stride = (size_t)H * d;\n            } else {\n                L = Lkv;\n                row0 = ((size_t)u * H + h) * (size_t)Lkv * d;\n                row_stride = (size_t)d;\n            }\n            for (int q = 0; q < Lq; ++q) {\n                const uint16_t *qrow",
                           "row_stride = (size_t)d;\n            } else {\n                L = Lkv;\n                row0 = ((size_t)u * H + h) * (size_t)Lkv * d;\n                row_stride = (size_t)d;\n            }\n            for (int q = 0; q < Lq; ++q) {\n                const uint16_t *qrow", ATTN_PINS),
    # segments
    "seg_unstable": ("for (int i = 0; i < n_cand; ++i) {       /* ascending i: stable */", "for (int i = n_cand - 1; i >= 0; --i) {", SEG_PINS),
    # every planted mistake keeps its writes inside the caller's buffers
    "seg_perm_stores_user": ("perm[next[u]] = i;", "perm[next[u]] = u;", SEG_PINS),
    "lse_drop_max": ("lse[(size_t)s * Lq + q] = L > 0 ? m + log(sum) : -INFINITY;",
                     "lse[(size_t)s * Lq + q] = L > 0 ? log(sum) : -INFINITY;", ATTN_LSE_PINS),
    "lse_no_scale": ("double sj = scale * dot;", "double sj = dot;", ATTN_LSE_PINS),
    "lse_drop_last_key": ("for (int j = 0; j < L; ++j) {\n                    const uint16_t *krow = kv_offsets ? K",
                          "for (int j = 0; j < L - (pass == 1); ++j) {\n                    const uint16_t *krow = kv_offsets ? K",
                          ATTN_LSE_PINS),
    "seg_chunk_off_by_one": ("if (cnt > cands_per_unit) cnt = cands_per_unit;", "if (cnt >= cands_per_unit) cnt = cands_per_unit - 1 + (cands_per_unit == 1);", SEG_PINS),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new, pins = MUTATIONS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/not found"
    mutated = tmp_path / "mut.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutated), str(tmp_path / "libmut.so"))
    orc = oracle.Oracle(lib)
    caught = []
    for pin in pins:
        try:
            pin(orc)
        except (AssertionError, oracle.OracleError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {name}"
