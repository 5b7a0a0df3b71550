// bwd_internal.h -- parameter blocks of the training (backward) kernels:
// LCE backward (lce_bwd.cu) and attention backward (attn_bwd.cu).  Not part
// of the public ABI.
#pragma once
#include "ikbo_internal.h"

namespace ikbo {

// -------------------------------------------------------- LCE backward
// S[u] = sum of dY over user u's candidates (the broadcast's transpose).
// 128 threads x 8 elements per CTA slice; a user's segment may be split
// into nch chunks whose fp32 partial sums a second pass adds in order.  For
// the tensor-core products S is kept as a bf16 pair, hi = bf16(S) and
// lo = bf16(S - hi) (16 significant bits), in S2[u][hi, lo][NP][D] with
// NP = ceil(N / 64) * 64 rows per half (rows N .. NP-1 are zero).
constexpr int BWD_SEG_THREADS = 128;
constexpr int BWD_SEG_SLICE = BWD_SEG_THREADS * 8;

struct SegSumParams {
  const uint16_t* dY;        // [n_cand][N][D] bf16
  const int32_t* offsets;    // [n_users + 1] (the plan's)
  const int32_t* perm;       // [n_cand] candidates grouped by user (the plan's)
  float* S;                  // [n_users][N][D] fp32
  uint16_t* S2;              // [n_users][2][NP][D] bf16: hi, lo
  float* part;               // [n_users * nch][N][D] fp32 when nch > 1
  int n_cand, n_users, ND, NPD, nch, slices;   // NPD = NP * D
};

// Activation-gradient GEMM: out[b][m][d] = sum_n W[m][n] X[b][n][d] (dC from
// dY and W_c, dU from S and W_u).  Tile = (b, 128-row block of D) over all m:
// M = 128 d rows on TMEM lanes, N = m in ranges of <= 256 columns, K = n.
// X chunks stream (MN-major, as the forward's C); W stays resident (K-major).
// X may hold kcx = 2 * kc chunks per b (the hi and lo halves of S2): X chunk
// j multiplies W chunk j % kc.
constexpr int BWD_THREADS = 384;       // warp 0 TMA, 1 MMA, 2 TMEM, 3 idle, 4-11 epilogue
constexpr int BWD_ACT_MAX_STAGES = 4;  // X ring depth: 4, or fewer (>= 2) when W leaves less room

struct ActParams {
  uint16_t* out;             // [B][M][D] bf16
  uint32_t* status;
  int B, M, D, N;
  int n_dblk;                // ceil(D / 128)
  int kc;                    // ceil(N / 64): resident W chunks
  int kcx;                   // X chunks per b (kc, or 2 * kc for a hi/lo pair)
  int m_pad;                 // accumulator columns: roundup(M, 16), or 128 when M is split
  int m_rows;                // resident W rows per K chunk: roundup(M, 128), or 128 when M is split
  int n_mgrp;                // blocks of m_rows rows M is split into (1: not split)
  int bufs;                  // accumulator buffers (2 when m_pad <= 256)
  int stages;                // X ring depth
  uint64_t timeout_ns;
};

// Weight-gradient GEMM, split along K = (b, d): unit (group of <= 2 m
// blocks, b range) accumulates A[b][m][d] G[b][n][d] over its b range into
// TMEM (M = 128 m rows per block, N = n, both operands K-major) and writes
// fp32 partials; a reduce pass adds the partials of each m block in order.
constexpr int BWD_WG_MAX_STAGES = 4;

struct WgradParams {
  float* part;               // [n_units][128][N] fp32 (split-K partials; not used with clusters)
  float* dW;                 // [M][N] fp32, written by the kernel itself with clusters
  int cluster;               // 0: partials + reduce kernel; else the R CTAs of an m block form a
                             // cluster and add their partials through distributed shared memory
  uint32_t* status;
  int B, M, D, N;            // B = batches of G; A's batch is b >> a_shift
  int a_shift;               // 1 when G holds a hi/lo pair per batch of A
  int n_mblk;                // ceil(M / 128)
  int mg;                    // m blocks per unit (1 or 2)
  int n_mgrp;                // ceil(n_mblk / mg)
  int R;                     // b ranges per m group (n_units = n_mgrp * R)
  int stages;                // ring depth
  int dc;                    // ceil(D / 64)
  int n_mma;                 // roundup(N, 16)
  int nb;                    // ceil(n_mma / 64): 64-row boxes of G per chunk
  uint64_t timeout_ns;
};

// Candidate pass of the LCE backward: one persistent launch that reads each
// candidate's dY (and C) once.  Unit = (candidate b = perm[pos], 64-wide
// block dh of D), numbered dh * n_cand + pos (the plan's user-grouped order
// within each D block); each CTA takes one contiguous range of units.  Per
// unit, from the dY block staged in shared memory:
//   dC[b]  = W_c dY[b]            (W_c resident in shared memory; TMEM)
//   dW_c  += C[b] dY[b]^T         (TMEM, <= 2 blocks of 128 K_c rows, per CTA)
//   S[u]  += dY[b]                (epilogue warps, fp32 registers)
// S of a run (user u, D block dh) that lies inside one CTA's range is
// written by that CTA; a run shared by several CTAs leaves partial slots
// (each CTA's first and last run).  S leaves as the bf16 hi/lo pair the
// user-side products read.  Each CTA also keeps its share of db (per n, its
// runs' sums over d).  The finish -- dW_c as the sum of the per-CTA partials
// in CTA order, S of the shared runs as the sum of their slots in CTA order,
// db as the sum of the CTAs' shares in CTA order -- runs after a grid
// barrier in the same launch (cooperative: all CTAs resident), or, where a
// cooperative launch is refused, as a second kernel.  Applies when
// K_c <= 256 and N <= 192.
constexpr int BWD_CAND_DY_SLOTS = 2;    // dY blocks: <= 3 n chunks of 64 n x 64 d (24 KB)
constexpr int BWD_CAND_C_SLOTS = 5;     // C slots: 128 K_c rows x 64 d (16 KB)
constexpr int BWD_CAND_MAX_N = 192;
constexpr int BWD_CAND_MAX_KC = 256;

struct CandParams {
  const int32_t* perm;       // [n_cand] the plan's user-grouped order (out-of-range candidates last)
  const int32_t* map;        // [n_cand]
  const int32_t* offsets;    // [n_users + 1] the plan's segment offsets
  uint16_t* dC;              // [n_cand][K_c][D] bf16, or null (no dC)
  float* wpart;              // [n_mblk][G][N][128] fp32 dW_c partials (K_c row of the block
                             // innermost), or null (no dW_c)
  float* dWc;                // [K_c][N] fp32 (with wpart)
  uint16_t* S2;              // [n_users][2][NP][D] bf16 hi, lo of S, or null (no S)
  float* spart;              // [G][2][N][64] fp32 S partials of each CTA's first and last run
  float* dbcta;              // [G][N] each CTA's share of db
  float* db;                 // [N] or null
  uint32_t* ctrl;            // [2] grid barrier: arrivals, departures (zero at launch)
  uint32_t* status;
  int n_cand, n_users, K_c, D, N, NPD;  // NPD = NP * D, NP = roundup(N, 64)
  int n_dh;                  // ceil(D / 64)
  int kcn;                   // ceil(N / 64): dY n chunks (<= 3)
  int n_mblk;                // ceil(K_c / 128): K_c blocks (1 or 2)
  int n_mma;                 // roundup(N, 16): dW_c accumulator columns per block
  int G;                     // grid of the candidate pass (the number of dW_c partials)
  int fused_finish;          // 1: the finish runs in the same (cooperative) launch
  uint64_t timeout_ns;
};

// ------------------------------------------------- attention backward
// dQ kernel (per work-list unit = one 128-row query tile): pass 1 over the
// user's key tiles forms each row's log-sum-exp; pass 2 recomputes S, forms
// dP = dO V^T, dS = P (dP - D) scale into TMEM and accumulates dQ += dS K.
// It also stores LSE and D = rowsum(dO * O) for the dK/dV kernel.
// dK/dV kernel (per (user, head, 128-key block)): over every query tile of
// the user's candidates, S^T = K Q^T and dP^T = V dO^T with keys on TMEM
// lanes, then dV += P^T dO and dK += dS^T Q accumulate in TMEM.
constexpr int ABWD_THREADS = 384;  // warp 0 TMA, 1 MMA + TMEM, 2 MMA (dK/dV), 3 idle, 4-11 element-wise

struct AttnBwdParams {
  const int32_t* perm;
  const int32_t* work;       // the plan's work list [n_units][4]
  const int32_t* n_units;
  const int32_t* offsets;    // the plan's user segment offsets [n_users + 1]
  const int32_t* kv_offsets; // jagged K/V or null (dense)
  const int32_t* blk_prefix; // dK/dV kernel: [n_users + 1] prefix of ceil(L_u / 128)
  const int32_t* tile_prefix;// [n_users + 1] prefix of the users' query tiles, ceil(count_u / cands_per_tile)
  const uint16_t* O;         // forward output [n_cand][H][Lq][d]
  const uint16_t* dO;        // [n_cand][H][Lq][d]
  uint16_t* dQ;              // [n_cand][H][Lq][d]
  uint16_t* dK;              // like K
  uint16_t* dV;              // like V
  float* lse;                // [work unit][128 tile rows]: log2-domain LSE (+inf for rows without a query)
  float* Drow;               // [work unit][128 tile rows]: D = rowsum(dO * O) (0 for rows without a query)
  const float* lse_in;       // the forward's natural-log LSE [n_cand][H][Lq], or null (recomputed)
  uint32_t* status;
  int n_cand, n_users, H, Lq, Lkv, cands_per_tile;
  float scale, scale_log2;
  uint64_t timeout_ns;
};

}  // namespace ikbo
