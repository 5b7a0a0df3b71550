// ikbo_internal.h -- kernel parameter blocks, tile constants and the device
// status word shared by the inference kernels (seg.cu, lce.cu, attn.cu) and
// the host API (api.cu); the training kernels' blocks are in bwd_internal.h.
// Not part of the public ABI (include/ikbo.h is).
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

}  // namespace ikbo
