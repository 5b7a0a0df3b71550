"""Algorithmic FLOP and byte counts for the IKBO hot path (host logic).

These are the counts the roofline is measured against: the method's own
work (the user GEMM at the user batch, not the candidate batch; no padding
FLOPs) and its non-replicated bytes (every input read once, every output
written once; the fp32 user-partial workspace and the segment arrays are
not counted, so they count against the kernels).

The attention intensity formula is the one behind the FLOP/byte figures of
aixai.ru, "Deep Dive: Flash Attention" (about 60 FLOP/B for standard
attention at sequence length 1024, about 833 FLOP/B for IKBO at 70:1).
"""
from __future__ import annotations

BF16 = 2
I32 = 4


# ----------------------------------------------------------------- LCE
def lce_flops(n_cand: int, n_users: int, K_u: int, K_c: int, D: int, N: int) -> float:
    """2*D*N*(n_users*K_u + n_cand*K_c): user GEMM at n_users, candidate GEMM at n_cand."""
    return 2.0 * D * N * (n_users * K_u + n_cand * K_c)


def lce_bytes(n_cand: int, n_users: int, K_u: int, K_c: int, D: int, N: int, bias: bool = True) -> float:
    """U, C, W_u, W_c, b and map read once; Y written once (bf16)."""
    rd = BF16 * (n_users * K_u * D + n_cand * K_c * D + K_u * N + K_c * N + (N if bias else 0))
    rd += I32 * n_cand
    wr = BF16 * n_cand * N * D
    return float(rd + wr)


def lce_backward_flops(n_cand: int, n_users: int, K_u: int, K_c: int, D: int, N: int) -> float:
    """The four products of the LCE backward, each at its own batch: dU and dW_u
    at n_users, dC and dW_c at n_cand (2*D*N*K per batch row each); the segment
    sum's additions are not counted."""
    return 2.0 * lce_flops(n_cand, n_users, K_u, K_c, D, N)


def lce_backward_bytes(n_cand: int, n_users: int, K_u: int, K_c: int, D: int, N: int) -> float:
    """dY, U, C, W_u, W_c and map read once; dU, dC (bf16) and dW_u, dW_c, db
    (fp32) written once."""
    rd = BF16 * (n_cand * N * D + n_users * K_u * D + n_cand * K_c * D + K_u * N + K_c * N) + I32 * n_cand
    wr = BF16 * (n_users * K_u * D + n_cand * K_c * D) + 4 * (K_u * N + K_c * N + N)
    return float(rd + wr)


def lce_materialised_flops(n_cand: int, K_u: int, K_c: int, D: int, N: int) -> float:
    """The replicated baseline: one GEMM over K_u + K_c for every candidate."""
    return 2.0 * D * N * n_cand * (K_u + K_c)


def lce_candidate_bytes(K_c: int, D: int, N: int) -> float:
    """Per-candidate streaming bytes of the candidate GEMM: C[i] read + Y[i] written."""
    return float(BF16 * (K_c * D + N * D))


# ----------------------------------------------------------- attention
def attn_flops(H: int, Lq: int, d: int, kv_len_per_cand) -> float:
    """4*H*Lq*d*sum_i L_{map[i]} (QK^T and PV, 2 FLOPs per multiply-add)."""
    total = sum(int(x) for x in kv_len_per_cand)
    return 4.0 * H * Lq * d * total


def attn_bytes(n_cand: int, H: int, Lq: int, d: int, kv_rows_total: int) -> float:
    """Q read and O written once per candidate; K and V read once per user.

    kv_rows_total: number of (user, key) rows stored, i.e. n_users*Lkv dense or
    sum_u L_u jagged.  The map is read once.
    """
    return float(BF16 * (2 * n_cand * H * Lq * d + 2 * kv_rows_total * H * d) + I32 * n_cand)


def attn_backward_flops(H: int, Lq: int, d: int, kv_len_per_cand) -> float:
    """The five products of the attention backward per (candidate, head): S
    recomputed, dP = dO V^T, dV += P^T dO, dK += dS^T Q, dQ = dS K, each
    2*Lq*L*d multiply-adds -> 10*H*Lq*d*sum_i L_{map[i]} (2.5x the forward).
    The softmax's element-wise work is not counted."""
    return 2.5 * attn_flops(H, Lq, d, kv_len_per_cand)


def attn_backward_bytes(n_cand: int, H: int, Lq: int, d: int, kv_rows_total: int) -> float:
    """Q, O, dO read and dQ written once per candidate (bf16); K, V read and
    dK, dV written once per user; the map read once.  The per-row softmax
    statistics the kernels keep between passes are not counted."""
    return float(BF16 * (4 * n_cand * H * Lq * d + 4 * kv_rows_total * H * d) + I32 * n_cand)


def attn_intensity_standard(Lq: int, Lkv: int) -> float:
    """FLOP/B of attention on materialised K/V, per (candidate, head).

    FLOPs 4*Lq*Lkv*d over bytes 2*d*(2*Lq + 2*Lkv) (Q, O, K, V once) =
    Lq*Lkv/(Lq+Lkv); d cancels.
    """
    return Lq * Lkv / (Lq + Lkv)


def attn_intensity_ikbo(Lq: int, Lkv: int, ratio: float) -> float:
    """FLOP/B when one user's K/V serves `ratio` candidates: r*Lq*Lkv/(r*Lq + Lkv)."""
    return ratio * Lq * Lkv / (ratio * Lq + Lkv)


def roofline_time(flops: float, nbytes: float, peak_flops: float, peak_bytes_per_s: float) -> float:
    """max(FLOPs / compute peak, bytes / HBM peak), in seconds."""
    return max(flops / peak_flops, nbytes / peak_bytes_per_s)
