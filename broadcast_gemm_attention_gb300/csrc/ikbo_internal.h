// ikbo_internal.h -- kernel parameter blocks, tile constants and the device
// status word shared by the kernels (seg.cu, lce.cu, attn.cu) and the host
// API (api.cu).  Not part of the public ABI (include/ikbo.h is).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace ikbo {

// ----------------------------------------------------------- status word
// One uint32 in device memory per plan; kernels OR these bits in, the host
// reads and clears it in ikbo_plan_get_status.
enum : uint32_t {
  DEV_ERR_MAP_RANGE = 1u << 0,     // a map entry outside [0, n_users)
  DEV_ERR_FLAG_TIMEOUT = 1u << 1,  // an LCE user partial never became ready
  DEV_ERR_PIPE_TIMEOUT = 1u << 2,  // an mbarrier wait inside a kernel ran out
  DEV_ERR_BAD_WORK = 1u << 3,      // inconsistent attention work unit
  DEV_ERR_SMEM_LAYOUT = 1u << 4,   // dynamic shared memory too misaligned for the tile layout
};

// Debug switches (ikbo_plan_set_debug).
enum : uint32_t {
  DEBUG_WITHHOLD_USER_PARTIAL = 1u << 0,  // LCE: never publish user partials
  DEBUG_NO_COOPERATIVE = 1u << 1,         // LCE backward: the candidate pass and its finish as two launches
};

// ------------------------------------------------------------ segments
constexpr int SEG_THREADS = 1024;
constexpr int SEG_MAX_USERS = 8192;

struct SegParams {
  const int32_t* map;
  int n_cand, n_users, H, cands_per_unit;
  int32_t* counts;    // [n_users]
  int32_t* offsets;   // [n_users + 1]
  int32_t* runs;      // [n_users + 1] users before u with at least one candidate; [n_users] = all such
  int32_t* perm;      // [n_cand]
  int32_t* work;      // [max_units][4]
  int32_t* n_units;   // [1]
  int64_t max_units;
  uint32_t* status;
};

// ----------------------------------------------------------------- LCE
// Tiles: M = 128 rows of D (TMEM lanes), N = N_mma columns (<= 256), K in
// chunks of 64 (one 128-byte swizzle row per k when MN-major).
constexpr int LCE_BM = 128;
constexpr int LCE_BK = 64;
constexpr int LCE_THREADS = 384;            // warp 0 TMA, 1 MMA, 2 TMEM, 3 idle, 4-11 epilogue
constexpr int LCE_EPI_WARP0 = 4;
constexpr int LCE_EPI_THREADS = LCE_THREADS - 32 * LCE_EPI_WARP0;
constexpr int LCE_A_STAGE_BYTES = LCE_BM * LCE_BK * 2;   // 16 KB: two 64(d) x 64(k) boxes
constexpr int LCE_MAX_STAGES = 8;
constexpr int LCE_MAX_W_SLOTS = 8;

struct LceParams {
  const int32_t* map;
  const int32_t* order;   // candidate order for the candidate tiles (a permutation of 0..n_cand-1, grouped
                          // by user) or null for 0..n_cand-1
  const int32_t* seg_offsets;  // [n_users + 1] where each user's run starts in order, or null
  const int32_t* seg_runs;     // [n_users + 1] non-empty runs before each user (and in all), or null
  const uint16_t* bias;   // [N] bf16 or null
  const uint16_t* U;      // [n_users][K_u][D] bf16 (read through tmU; raw for the CUDA-core fallback)
  const uint16_t* Wu;     // [K_u][N] bf16 (likewise)
  uint16_t* Y;            // [n_cand][N][D] bf16
  float* partial;         // [n_users][N][D] fp32 workspace (user GEMM + bias)
  uint32_t* flags;        // [n_users][n_dblk][NB] readiness (one per user tile): `epoch` once published,
                          // 0 between calls (the launch that reads them clears them as it ends)
  uint32_t* status;
  uint32_t* timeout_epoch;  // set to `epoch` by the first flag wait that times out in a launch (cleared
                            // with the flags)
  uint32_t* done;         // CTAs of the flag-reading launch that have finished (0 between calls)
  int n_cand, n_users, K_u, K_c, D, N;
  int N_mma;              // N rounded up to 16
  int NB;                 // 64-wide column blocks of W (ceil(N_mma / 64))
  int n_dblk;             // ceil(D / 128)
  int n_user_units;       // n_users * n_dblk * NB (user tiles are split along N)
  int n_units;            // n_user_units + n_cand * n_dblk
  int kc_u, kc_c;         // 64-wide K chunks (ceil(K / 64))
  int ks_u, ks_c;         // 16-wide MMA k-steps (ceil(K / 16))
  int stages;             // A ring depth
  int stages_local;       // A ring depth of the local-partial schedule (0: that schedule does not fit)
  int w_slots;            // 8 KB W_u slots in the W region used by user tiles (2..8)
  int wu_slots;           // full-width W_u chunk slots after the A ring (local-partial schedule only, else 0)
  uint32_t w_region_bytes;
  uint32_t epoch;         // value written to / awaited in `flags` (LCE_FLAG_READY)
  uint32_t debug;
  uint32_t mode;          // LCE_MODE_* bits: the stage-ladder ablations (0 = the full kernel)
  int schedule;           // LCE_SCHEDULE_*: one launch or two (plan-time choice by default)
  uint64_t timeout_ns;
};

// Ablation modes of the LCE kernel (the pages' stage ladder, rebuilt from
// this kernel): NO_PARTIAL = candidate tiles store bf16(C W_c) without the
// user partial (a separate broadcast-add launch adds it: the decomposed,
// unfused stage); ONE_ACC = a single TMEM accumulator, so a tile's epilogue
// and the next tile's products no longer overlap (fused epilogue without
// the warp-specialised pipelining across tiles).
enum : uint32_t {
  LCE_MODE_NO_PARTIAL = 1u << 0,
  LCE_MODE_ONE_ACC = 1u << 1,
};

// Launch schedule of the LCE: chosen from the shape (AUTO), or forced.
enum : int {
  LCE_SCHEDULE_AUTO = 0,
  LCE_SCHEDULE_TWO = 1,    // user tiles, then candidate tiles
  LCE_SCHEDULE_ONE = 2,    // one launch, user tiles first in every CTA's list
  LCE_SCHEDULE_LOCAL = 3,  // one launch of candidate tiles; each CTA computes the user partials its
                           // own tiles need, into TMEM (N <= 192)
};
// Value of a published readiness flag.  Flags are zero before every call
// (cleared by the last CTA of the launch that reads them), so a fixed value
// serves every call.
constexpr uint32_t LCE_FLAG_READY = 1;
// AUTO takes one launch below this many candidate tiles per SM.
constexpr int LCE_ONE_LAUNCH_TILES_PER_SM = 8;
constexpr int LCE_WU_SLOTS = 2;     // W_u chunk slots of the local-partial schedule
constexpr int LCE_LOCAL_MAX_N = 192;  // the epilogue keeps a partial of at most 6 x 32 columns per row

// Fills the derived fields of an LceParams from its sizes (n_cand, n_users,
// K_u, K_c, D, N); returns false for shapes the kernel does not support.
// Shared by every LCE entry point so they configure the kernel identically.
bool lce_configure(LceParams* lp, size_t max_smem);
// The schedule a launch of lp runs: lp->schedule where it applies to the
// shape and mode, else the plan-time choice.
int lce_resolve_schedule(const LceParams& lp, int num_sms);
size_t lce_flag_count(const LceParams& lp);
size_t lce_smem_bytes(const LceParams& lp);

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

// ----------------------------------------------------------- attention
constexpr int ATT_BM = 128;        // query rows per tile (TMEM lanes)
constexpr int ATT_BN = 128;        // keys per K/V tile
constexpr int ATT_D = 128;         // head dim (the only one supported)
constexpr int ATT_TILES = 1;       // query tiles per work unit
constexpr int ATT_THREADS = 384;   // warp 0 TMA Q+K, 1 S issuer, 2 P.V issuer, 3 TMA V, 4-11 softmax
constexpr int ATT_KV_STAGE_BYTES = ATT_BN * ATT_D * 2;   // 32 KB
constexpr int ATT_Q_TILE_BYTES = ATT_BM * ATT_D * 2;     // 32 KB
constexpr int ATT_Q_BUFS = 2;      // Q tiles (a unit's Q stays in shared memory for all of its S products;
                                   // a finished unit's buffer stages its O on the way out)
constexpr int ATT_K_STAGES = 3;    // K ring
constexpr int ATT_V_STAGES = 2;    // V ring
// shared memory: 2 x 32 KB Q + 5 x 32 KB K/V = 224 KB of 227

struct AttnParams {
  const int32_t* perm;
  const int32_t* work;       // [n_units][4]: user, head, perm start, count
  const int32_t* n_units;    // device scalar written by the segment builder
  const int32_t* kv_offsets; // [n_users+1] or null (dense)
  uint16_t* O;               // [n_cand][H][Lq][d]
  float* lse;                // [n_cand][H][Lq] natural-log row log-sum-exp, or null (not written)
  uint32_t* status;
  int n_cand, n_users, H, Lq, Lkv;  // Lkv: dense length (ignored when jagged)
  int cands_per_tile;        // floor(128 / Lq)
  float scale_log2;          // scale * log2(e)
  uint64_t timeout_ns;
  // self units (users' own queries against the same K/V), after the work
  // list's units: n_self = n_users * H * self_tiles, 0 if none
  uint16_t* O_user;          // [n_users][H][Lq_u][d]
  int n_self, self_tiles, self_rows, Lq_u;  // self_rows = query rows per self tile (<= 128)
  int self_only;             // 1: skip the work list's units (the self part alone)
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
