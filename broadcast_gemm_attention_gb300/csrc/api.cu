// api.cu -- the C ABI declared in include/ikbo.h: plan lifetime, argument
// validation, TMA tensor-map encoding and kernel launches.  No computation
// of the method happens on the host.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "ikbo.h"
#include "bwd_internal.h"

namespace ikbo {
cudaError_t launch_seg_build(const SegParams& p, cudaStream_t s);
size_t lce_smem_bytes(const LceParams& p);
cudaError_t launch_lce(const CUtensorMap& tmU, const CUtensorMap& tmC, const CUtensorMap& tmWu,
                       const CUtensorMap& tmWc, const LceParams& p, int num_sms, cudaStream_t s, int* launches);
cudaError_t launch_lce_stage(const CUtensorMap& tmU, const CUtensorMap& tmC, const CUtensorMap& tmWu,
                             const CUtensorMap& tmWc, LceParams p, int stage, int num_sms, cudaStream_t s,
                             int* launches);
size_t attn_smem_bytes();
cudaError_t launch_attn(const CUtensorMap& tmQ, const CUtensorMap& tmQu, const CUtensorMap& tmK,
                        const CUtensorMap& tmV, const AttnParams& p, int grid, cudaStream_t s);
int bwd_segsum_chunks(int n_cand, int n_users, int ND, int num_sms);
cudaError_t launch_bwd_segsum(const SegSumParams& p, cudaStream_t s, int* launches);
cudaError_t launch_bwd_db(const float* S, float* db, int n_users, int N, int D, cudaStream_t s);
bool bwd_act_configure(ActParams* p, size_t max_smem, bool pair, int num_sms, bool split);
cudaError_t launch_bwd_act(const CUtensorMap& tmX, const CUtensorMap& tmW, const ActParams& p, int num_sms,
                           cudaStream_t s);
bool bwd_wgrad_configure(WgradParams* p, int num_sms, size_t max_smem);
size_t bwd_wgrad_part_elems(const WgradParams& p);
bool bwd_cand_configure(CandParams* p, size_t max_smem);
int bwd_cand_grid(const CandParams& p, int num_sms);
cudaError_t launch_bwd_cand(const CUtensorMap& tmDY, const CUtensorMap& tmC, const CUtensorMap& tmW,
                            const CandParams& p, int num_sms, bool cooperative, cudaStream_t s, int* launches);
cudaError_t launch_bwd_wgrad(const CUtensorMap& tmA, const CUtensorMap& tmG, const WgradParams& p, float* dW,
                             int num_sms, cudaStream_t s, int* launches);
size_t attn_bwd_smem_bytes();
cudaError_t launch_attn_backward(const CUtensorMap& tmQ, const CUtensorMap& tmDO, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const AttnBwdParams& p, int grid, cudaStream_t s,
                                 int* launches);
}  // namespace ikbo

using namespace ikbo;

struct ikbo_plan_s {
  int device = 0;
  int num_sms = 0;
  size_t max_smem = 0;
  int max_cand = 0, max_users = 0, max_heads = 0;
  // the bound request
  bool planned = false;
  const int32_t* d_map = nullptr;
  int n_cand = 0, n_users = 0, H = 0, Lq = 0, cands_per_unit = 0;
  // plan-owned device memory
  int32_t* d_counts = nullptr;
  int32_t* d_offsets = nullptr;
  int32_t* d_runs = nullptr;
  int32_t* d_perm = nullptr;
  int32_t* d_work = nullptr;
  int32_t* d_n_units = nullptr;
  int64_t max_units = 0;
  uint32_t* d_status = nullptr;  // [0] status bits, [1] LCE flag-timeout word, [2] LCE finished-CTA count
  float* d_partial = nullptr;
  size_t partial_elems = 0;
  uint32_t* d_flags = nullptr;
  size_t flags_elems = 0;
  // LCE backward workspaces (grown on first use)
  float* d_bwd_S = nullptr;
  size_t bwd_S_elems = 0;
  uint16_t* d_bwd_Sb = nullptr;
  size_t bwd_Sb_elems = 0;
  float* d_bwd_seg = nullptr;
  size_t bwd_seg_elems = 0;
  float* d_bwd_wpart = nullptr;
  size_t bwd_wpart_elems = 0;
  float* d_bwd_spart = nullptr;  // candidate pass: S partials of each CTA's first and last run
  size_t bwd_spart_elems = 0;
  float* d_bwd_dbcta = nullptr;  // candidate pass: each CTA's share of db
  size_t bwd_dbcta_elems = 0;
  uint32_t* d_bwd_ctrl = nullptr;  // candidate pass: grid barrier counts
  size_t bwd_ctrl_elems = 0;
  // a second stream (created on first use) on which dW_u runs beside dU
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  // attention backward workspaces
  float* d_abwd_lse = nullptr;
  size_t abwd_lse_elems = 0;
  float* d_abwd_drow = nullptr;
  size_t abwd_drow_elems = 0;
  int32_t* d_abwd_blk = nullptr;
  size_t abwd_blk_elems = 0;
  bool lce_flags_dirty = false;  // an LCE launch failed: its flags may still be set
  uint32_t debug = 0;
  uint64_t timeout_ns = 2000000000ull;
  int lce_schedule = LCE_SCHEDULE_AUTO;
  std::atomic<uint64_t> launches{0};
};

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// bf16 tensor map with 128-byte swizzle; out-of-bounds elements read as zero.
bool encode_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                 const uint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gd,
                  gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Grows a plan workspace to `need` elements.  New memory is zeroed on
// `stream`, the stream of the call that will use it, so the clear is ordered
// before that call's kernels.
template <typename T>
cudaError_t grow(T** ptr, size_t* have, size_t need, cudaStream_t stream) {
  if (*have >= need && *ptr) return cudaSuccess;
  if (*ptr) cudaFree(*ptr);
  *ptr = nullptr;
  *have = 0;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(ptr), need * sizeof(T));
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(*ptr, 0, need * sizeof(T), stream);
  if (e != cudaSuccess) return e;
  *have = need;
  return cudaSuccess;
}

void free_plan(ikbo_plan_t p) {
  if (!p) return;
  cudaFree(p->d_counts);
  cudaFree(p->d_offsets);
  cudaFree(p->d_runs);
  cudaFree(p->d_perm);
  cudaFree(p->d_work);
  cudaFree(p->d_n_units);
  cudaFree(p->d_status);
  cudaFree(p->d_partial);
  cudaFree(p->d_flags);
  cudaFree(p->d_bwd_S);
  cudaFree(p->d_bwd_Sb);
  cudaFree(p->d_bwd_seg);
  cudaFree(p->d_bwd_wpart);
  cudaFree(p->d_bwd_spart);
  cudaFree(p->d_bwd_dbcta);
  cudaFree(p->d_bwd_ctrl);
  if (p->ev_fork) cudaEventDestroy(p->ev_fork);
  if (p->ev_join) cudaEventDestroy(p->ev_join);
  if (p->side) cudaStreamDestroy(p->side);
  cudaFree(p->d_abwd_lse);
  cudaFree(p->d_abwd_drow);
  cudaFree(p->d_abwd_blk);
  delete p;
}

}  // namespace

namespace {
// Both LCE entry points: stage 4 is the full kernel, 1 and 3 the ablations.
ikbo_status_t lce_launch(ikbo_plan_t p, const void* U, const void* C, const void* Wu, const void* Wc, const void* b,
                         void* Y, int K_u, int K_c, int D, int N, int stage, cudaStream_t stream) {
  if (!p) return IKBO_ERR_INVALID_ARG;
  if (!p->planned) return IKBO_ERR_NOT_PLANNED;
  if (!U || !C || !Wu || !Wc || !Y) return IKBO_ERR_INVALID_ARG;
  if (K_u < 1 || K_c < 1 || D < 1 || N < 1) return IKBO_ERR_UNSUPPORTED;
  if (!aligned16(U) || !aligned16(C) || !aligned16(Wu) || !aligned16(Wc) || !aligned16(Y) || (b && !aligned16(b)))
    return IKBO_ERR_INVALID_ARG;
  if (D % 8 != 0 || N % 8 != 0 || N > 256) return IKBO_ERR_UNSUPPORTED;

  LceParams lp;
  std::memset(&lp, 0, sizeof(lp));
  lp.n_cand = p->n_cand;
  lp.n_users = p->n_users;
  lp.K_u = K_u;
  lp.K_c = K_c;
  lp.D = D;
  lp.N = N;
  if (!lce_configure(&lp, p->max_smem)) return IKBO_ERR_UNSUPPORTED;
  lp.map = p->d_map;
  lp.order = p->d_perm;  // candidates grouped by user: consecutive tiles of a CTA share the user partial
  lp.seg_offsets = p->d_offsets;
  lp.seg_runs = p->d_runs;
  lp.bias = static_cast<const uint16_t*>(b);
  lp.Y = static_cast<uint16_t*>(Y);

  const size_t part = static_cast<size_t>(p->n_users) * N * D;
  const size_t nflags = lce_flag_count(lp);
  if (grow(&p->d_partial, &p->partial_elems, part, stream) != cudaSuccess) return IKBO_ERR_CUDA;
  if (grow(&p->d_flags, &p->flags_elems, nflags, stream) != cudaSuccess) return IKBO_ERR_CUDA;
  if (p->lce_flags_dirty) {  // a failed launch may have left flags set: clear them, the timeout word and the count
    if (cudaMemsetAsync(p->d_flags, 0, sizeof(uint32_t) * p->flags_elems, stream) != cudaSuccess ||
        cudaMemsetAsync(p->d_status + 1, 0, 2 * sizeof(uint32_t), stream) != cudaSuccess)
      return IKBO_ERR_CUDA;
    p->lce_flags_dirty = false;
  }
  lp.U = static_cast<const uint16_t*>(U);
  lp.Wu = static_cast<const uint16_t*>(Wu);
  lp.partial = p->d_partial;
  lp.flags = p->d_flags;
  lp.status = p->d_status;
  lp.timeout_epoch = p->d_status + 1;
  lp.done = p->d_status + 2;
  lp.epoch = LCE_FLAG_READY;  // the flags are back at zero after every call
  lp.debug = p->debug;
  lp.schedule = p->lce_schedule;
  lp.timeout_ns = p->timeout_ns;

  CUtensorMap tmU, tmC, tmWu, tmWc;
  const uint64_t ud[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(K_u), static_cast<uint64_t>(p->n_users)};
  const uint64_t us[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(K_u) * D * 2};
  const uint64_t cd[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(K_c), static_cast<uint64_t>(p->n_cand)};
  const uint64_t cs[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(K_c) * D * 2};
  const uint32_t abox[3] = {64, LCE_BK, 1};
  const uint64_t wud[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K_u)};
  const uint64_t wcd[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K_c)};
  const uint64_t ws[1] = {static_cast<uint64_t>(N) * 2};
  const uint32_t wbox[2] = {64, LCE_BK};
  if (!encode_bf16(&tmU, U, 3, ud, us, abox) || !encode_bf16(&tmC, C, 3, cd, cs, abox) ||
      !encode_bf16(&tmWu, Wu, 2, wud, ws, wbox) || !encode_bf16(&tmWc, Wc, 2, wcd, ws, wbox))
    return IKBO_ERR_CUDA;

  int launches = 0;
  const cudaError_t e = launch_lce_stage(tmU, tmC, tmWu, tmWc, lp, stage, p->num_sms, stream, &launches);
  p->launches += static_cast<uint64_t>(launches);
  if (e != cudaSuccess) p->lce_flags_dirty = true;
  return e == cudaSuccess ? IKBO_OK : IKBO_ERR_CUDA;
}
}  // namespace

namespace {
// Both attention entry points: the work list's (target) units, plus, when
// Q_user is given, n_users * H * ceil(Lq_u / 128) self units in the same launch.
ikbo_status_t attn_launch(ikbo_plan_t p, const void* Q, const void* Q_user, const void* K, const void* V,
                          const int32_t* d_kv_offsets, void* O, void* O_user, float* lse, int Lq_u, int Lkv, int d,
                          float scale, cudaStream_t stream) {
  if (!p) return IKBO_ERR_INVALID_ARG;
  if (!p->planned) return IKBO_ERR_NOT_PLANNED;
  const bool self = Q_user != nullptr;
  const bool self_only = self && !Q && !O && !lse;  // the users' own queries alone
  if (!K || !V || (!self_only && (!Q || !O))) return IKBO_ERR_INVALID_ARG;
  if (!aligned16(K) || !aligned16(V) || (!self_only && (!aligned16(Q) || !aligned16(O))))
    return IKBO_ERR_INVALID_ARG;
  if (d != ATT_D) return IKBO_ERR_UNSUPPORTED;
  if (Lkv < 1 || !(scale > 0.f) || !std::isfinite(scale)) return IKBO_ERR_INVALID_ARG;
  if (self) {
    if (!O_user || !aligned16(Q_user) || !aligned16(O_user) || Lq_u < 1) return IKBO_ERR_INVALID_ARG;
    if (Lq_u % 8 != 0) return IKBO_ERR_UNSUPPORTED;
  }
  if (attn_smem_bytes() > p->max_smem) return IKBO_ERR_UNSUPPORTED;

  AttnParams ap;
  std::memset(&ap, 0, sizeof(ap));
  ap.perm = p->d_perm;
  ap.work = p->d_work;
  ap.n_units = p->d_n_units;
  ap.kv_offsets = d_kv_offsets;
  ap.O = static_cast<uint16_t*>(O);
  ap.lse = lse;
  ap.status = p->d_status;
  ap.n_cand = p->n_cand;
  ap.n_users = p->n_users;
  ap.H = p->H;
  ap.Lq = p->Lq;
  ap.Lkv = Lkv;
  ap.cands_per_tile = ATT_BM / p->Lq;
  ap.scale_log2 = scale * 1.4426950408889634f;
  ap.timeout_ns = p->timeout_ns;

  const uint64_t H = static_cast<uint64_t>(p->H), Lq = static_cast<uint64_t>(p->Lq);
  CUtensorMap tmQ, tmQu, tmK, tmV;
  const uint64_t qd[4] = {ATT_D, Lq, H, static_cast<uint64_t>(p->n_cand)};
  const uint64_t qs[3] = {ATT_D * 2, Lq * ATT_D * 2, H * Lq * ATT_D * 2};
  const uint32_t qbox[4] = {64, static_cast<uint32_t>(p->Lq), 1, 1};
  ap.self_only = self_only ? 1 : 0;
  if (!self_only && !encode_bf16(&tmQ, Q, 4, qd, qs, qbox)) return IKBO_ERR_CUDA;
  if (self) {
    ap.O_user = static_cast<uint16_t*>(O_user);
    ap.Lq_u = Lq_u;
    ap.self_rows = Lq_u < ATT_BM ? Lq_u : ATT_BM;
    ap.self_tiles = (Lq_u + ap.self_rows - 1) / ap.self_rows;
    ap.n_self = p->n_users * p->H * ap.self_tiles;
    const uint64_t Lu = static_cast<uint64_t>(Lq_u);
    const uint64_t ud[4] = {ATT_D, Lu, H, static_cast<uint64_t>(p->n_users)};
    const uint64_t us[3] = {ATT_D * 2, Lu * ATT_D * 2, H * Lu * ATT_D * 2};
    const uint32_t ubox[4] = {64, static_cast<uint32_t>(ap.self_rows), 1, 1};
    if (!encode_bf16(&tmQu, Q_user, 4, ud, us, ubox)) return IKBO_ERR_CUDA;
    if (self_only) tmQ = tmQu;  // no target units read it
  } else {
    tmQu = tmQ;  // not read without self units
  }
  if (d_kv_offsets) {
    const uint64_t kd[3] = {ATT_D, H, static_cast<uint64_t>(Lkv)};
    const uint64_t ks[2] = {ATT_D * 2, H * ATT_D * 2};
    const uint32_t kbox[3] = {64, 1, ATT_BN};
    if (!encode_bf16(&tmK, K, 3, kd, ks, kbox) || !encode_bf16(&tmV, V, 3, kd, ks, kbox)) return IKBO_ERR_CUDA;
  } else {
    const uint64_t L = static_cast<uint64_t>(Lkv);
    const uint64_t kd[4] = {ATT_D, L, H, static_cast<uint64_t>(p->n_users)};
    const uint64_t ks[3] = {ATT_D * 2, L * ATT_D * 2, H * L * ATT_D * 2};
    const uint32_t kbox[4] = {64, ATT_BN, 1, 1};
    if (!encode_bf16(&tmK, K, 4, kd, ks, kbox) || !encode_bf16(&tmV, V, 4, kd, ks, kbox)) return IKBO_ERR_CUDA;
  }
  if (launch_attn(tmQ, tmQu, tmK, tmV, ap, p->num_sms, stream) != cudaSuccess) return IKBO_ERR_CUDA;
  p->launches++;
  return IKBO_OK;
}
}  // namespace

namespace {
ikbo_status_t attn_backward_launch(ikbo_plan_t p, const void* Q, const void* K, const void* V, const void* O,
                                   const void* dO, const float* lse, const int32_t* d_kv_offsets, void* dQ, void* dK,
                                   void* dV, int Lkv, int d, float scale, cudaStream_t stream) {
  if (!p) return IKBO_ERR_INVALID_ARG;
  if (!p->planned) return IKBO_ERR_NOT_PLANNED;
  const void* ptrs[] = {Q, K, V, O, dO, dQ, dK, dV};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return IKBO_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return IKBO_ERR_INVALID_ARG;
  if (d != ATT_D) return IKBO_ERR_UNSUPPORTED;
  if (Lkv < 1 || !(scale > 0.f) || !std::isfinite(scale)) return IKBO_ERR_INVALID_ARG;
  if (attn_bwd_smem_bytes() > p->max_smem) return IKBO_ERR_UNSUPPORTED;
  // per work unit, its 128 tile rows' LSE and D (the work list holds at most
  // max_units units); the two user prefixes (key blocks, query tiles)
  const size_t rows = static_cast<size_t>(p->max_units) * ATT_BM;
  if (grow(&p->d_abwd_lse, &p->abwd_lse_elems, rows, stream) != cudaSuccess ||
      grow(&p->d_abwd_drow, &p->abwd_drow_elems, rows, stream) != cudaSuccess ||
      grow(&p->d_abwd_blk, &p->abwd_blk_elems, 2 * (static_cast<size_t>(p->n_users) + 1), stream) != cudaSuccess)
    return IKBO_ERR_CUDA;

  AttnBwdParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.perm = p->d_perm;
  bp.work = p->d_work;
  bp.n_units = p->d_n_units;
  bp.offsets = p->d_offsets;
  bp.kv_offsets = d_kv_offsets;
  bp.blk_prefix = p->d_abwd_blk;
  bp.tile_prefix = p->d_abwd_blk + p->n_users + 1;
  bp.O = static_cast<const uint16_t*>(O);
  bp.dO = static_cast<const uint16_t*>(dO);
  bp.dQ = static_cast<uint16_t*>(dQ);
  bp.dK = static_cast<uint16_t*>(dK);
  bp.dV = static_cast<uint16_t*>(dV);
  bp.lse = p->d_abwd_lse;
  bp.Drow = p->d_abwd_drow;
  bp.lse_in = lse;
  bp.status = p->d_status;
  bp.n_cand = p->n_cand;
  bp.n_users = p->n_users;
  bp.H = p->H;
  bp.Lq = p->Lq;
  bp.Lkv = Lkv;
  bp.cands_per_tile = ATT_BM / p->Lq;
  bp.scale = scale;
  bp.scale_log2 = scale * 1.4426950408889634f;
  bp.timeout_ns = p->timeout_ns;

  // the forward's layouts: Q, dO [n_cand][H][Lq][d] one box per candidate;
  // K, V dense [n_users][H][Lkv][d] or jagged [Lkv][H][d], 128-row boxes
  const uint64_t H = static_cast<uint64_t>(p->H), Lq = static_cast<uint64_t>(p->Lq);
  CUtensorMap tmQ, tmDO, tmK, tmV;
  const uint64_t qd[4] = {ATT_D, Lq, H, static_cast<uint64_t>(p->n_cand)};
  const uint64_t qs[3] = {ATT_D * 2, Lq * ATT_D * 2, H * Lq * ATT_D * 2};
  const uint32_t qbox[4] = {64, static_cast<uint32_t>(p->Lq), 1, 1};
  if (!encode_bf16(&tmQ, Q, 4, qd, qs, qbox) || !encode_bf16(&tmDO, dO, 4, qd, qs, qbox)) return IKBO_ERR_CUDA;
  if (d_kv_offsets) {
    const uint64_t kd[3] = {ATT_D, H, static_cast<uint64_t>(Lkv)};
    const uint64_t ks[2] = {ATT_D * 2, H * ATT_D * 2};
    const uint32_t kbox[3] = {64, 1, ATT_BN};
    if (!encode_bf16(&tmK, K, 3, kd, ks, kbox) || !encode_bf16(&tmV, V, 3, kd, ks, kbox)) return IKBO_ERR_CUDA;
  } else {
    const uint64_t L = static_cast<uint64_t>(Lkv);
    const uint64_t kd[4] = {ATT_D, L, H, static_cast<uint64_t>(p->n_users)};
    const uint64_t ks[3] = {ATT_D * 2, L * ATT_D * 2, H * L * ATT_D * 2};
    const uint32_t kbox[4] = {64, ATT_BN, 1, 1};
    if (!encode_bf16(&tmK, K, 4, kd, ks, kbox) || !encode_bf16(&tmV, V, 4, kd, ks, kbox)) return IKBO_ERR_CUDA;
  }
  int launches = 0;
  const cudaError_t e = launch_attn_backward(tmQ, tmDO, tmK, tmV, bp, p->num_sms, stream, &launches);
  p->launches += static_cast<uint64_t>(launches);
  return e == cudaSuccess ? IKBO_OK : IKBO_ERR_CUDA;
}
}  // namespace

extern "C" {

int ikbo_version(void) { return 106; }

ikbo_status_t ikbo_attn_backward(ikbo_plan_t p, const void* Q, const void* K, const void* V, const void* O,
                                 const void* dO, const float* lse, const int32_t* d_kv_offsets, void* dQ, void* dK,
                                 void* dV, int Lkv, int d, float scale, cudaStream_t stream) {
  return attn_backward_launch(p, Q, K, V, O, dO, lse, d_kv_offsets, dQ, dK, dV, Lkv, d, scale, stream);
}

const char* ikbo_status_string(ikbo_status_t s) {
  switch (s) {
    case IKBO_OK: return "ok";
    case IKBO_ERR_INVALID_ARG: return "invalid argument";
    case IKBO_ERR_UNSUPPORTED: return "unsupported shape or layout";
    case IKBO_ERR_CUDA: return "CUDA error";
    case IKBO_ERR_MAP_OUT_OF_RANGE: return "map value out of range";
    case IKBO_ERR_TIMEOUT: return "device wait timed out";
    case IKBO_ERR_NOT_PLANNED: return "no request planned";
    case IKBO_ERR_INTERNAL: return "internal error (work list)";
  }
  return "unknown status";
}

ikbo_status_t ikbo_plan_create(ikbo_plan_t* out, int max_cand, int max_users, int max_heads) {
  if (!out) return IKBO_ERR_INVALID_ARG;
  *out = nullptr;
  if (max_cand < 1 || max_users < 1 || max_heads < 1) return IKBO_ERR_INVALID_ARG;
  if (max_users > SEG_MAX_USERS) return IKBO_ERR_UNSUPPORTED;
  ikbo_plan_t p = new (std::nothrow) ikbo_plan_s();
  if (!p) return IKBO_ERR_CUDA;
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    delete p;
    return IKBO_ERR_CUDA;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, p->device) != cudaSuccess) {
    delete p;
    return IKBO_ERR_CUDA;
  }
  if (prop.major != 10 || prop.minor != 3) {
    delete p;
    return IKBO_ERR_UNSUPPORTED;
  }
  p->num_sms = prop.multiProcessorCount;
  p->max_smem = prop.sharedMemPerBlockOptin;
  p->max_cand = max_cand;
  p->max_users = max_users;
  p->max_heads = max_heads;
  // every candidate run is <= cands_per_unit and each user adds at most one
  // partial run per head, so H * (n_users + n_cand) bounds the unit count
  p->max_units = static_cast<int64_t>(max_heads) * (max_users + max_cand);
  bool ok = cudaMalloc(&p->d_counts, sizeof(int32_t) * max_users) == cudaSuccess &&
            cudaMalloc(&p->d_offsets, sizeof(int32_t) * (max_users + 1)) == cudaSuccess &&
            cudaMalloc(&p->d_runs, sizeof(int32_t) * (max_users + 1)) == cudaSuccess &&
            cudaMalloc(&p->d_perm, sizeof(int32_t) * max_cand) == cudaSuccess &&
            cudaMalloc(&p->d_work, sizeof(int32_t) * 4 * p->max_units) == cudaSuccess &&
            cudaMalloc(&p->d_n_units, sizeof(int32_t)) == cudaSuccess &&
            cudaMalloc(&p->d_status, sizeof(uint32_t) * 3) == cudaSuccess &&
            cudaMemset(p->d_status, 0, sizeof(uint32_t) * 3) == cudaSuccess &&
            cudaMemset(p->d_n_units, 0, sizeof(int32_t)) == cudaSuccess;
  if (!ok) {
    free_plan(p);
    return IKBO_ERR_CUDA;
  }
  *out = p;
  return IKBO_OK;
}

void ikbo_plan_destroy(ikbo_plan_t p) {
  if (!p) return;
  cudaDeviceSynchronize();
  free_plan(p);
}

ikbo_status_t ikbo_plan_set_debug(ikbo_plan_t p, unsigned flags) {
  if (!p) return IKBO_ERR_INVALID_ARG;
  p->debug = flags;
  return IKBO_OK;
}

ikbo_status_t ikbo_plan_set_lce_schedule(ikbo_plan_t p, int schedule) {
  if (!p || schedule < LCE_SCHEDULE_AUTO || schedule > LCE_SCHEDULE_LOCAL) return IKBO_ERR_INVALID_ARG;
  p->lce_schedule = schedule;
  return IKBO_OK;
}

ikbo_status_t ikbo_plan_set_timeout_ns(ikbo_plan_t p, uint64_t timeout_ns) {
  if (!p || timeout_ns == 0) return IKBO_ERR_INVALID_ARG;
  p->timeout_ns = timeout_ns;
  return IKBO_OK;
}

uint64_t ikbo_plan_launch_count(ikbo_plan_t p) { return p ? p->launches.load() : 0; }

ikbo_status_t ikbo_plan(ikbo_plan_t p, const int32_t* d_map, int n_cand, int n_users, int H, int Lq,
                        cudaStream_t stream) {
  if (!p || !d_map) return IKBO_ERR_INVALID_ARG;
  if (n_cand < 1 || n_cand > p->max_cand || n_users < 1 || n_users > p->max_users || H < 1 || H > p->max_heads)
    return IKBO_ERR_INVALID_ARG;
  if (Lq < 8 || Lq > ATT_BM || Lq % 8 != 0) return IKBO_ERR_UNSUPPORTED;
  const int cpt = ATT_BM / Lq;
  SegParams sp;
  sp.map = d_map;
  sp.n_cand = n_cand;
  sp.n_users = n_users;
  sp.H = H;
  sp.cands_per_unit = ATT_TILES * cpt;
  sp.counts = p->d_counts;
  sp.offsets = p->d_offsets;
  sp.runs = p->d_runs;
  sp.perm = p->d_perm;
  sp.work = p->d_work;
  sp.n_units = p->d_n_units;
  sp.max_units = p->max_units;
  sp.status = p->d_status;
  if (launch_seg_build(sp, stream) != cudaSuccess) {
    p->planned = false;
    return IKBO_ERR_CUDA;
  }
  p->launches++;
  p->planned = true;
  p->d_map = d_map;
  p->n_cand = n_cand;
  p->n_users = n_users;
  p->H = H;
  p->Lq = Lq;
  p->cands_per_unit = sp.cands_per_unit;
  return IKBO_OK;
}

ikbo_status_t ikbo_plan_segments(ikbo_plan_t p, const int32_t** d_counts, const int32_t** d_offsets,
                                 const int32_t** d_perm) {
  if (!p) return IKBO_ERR_INVALID_ARG;
  if (!p->planned) return IKBO_ERR_NOT_PLANNED;
  if (d_counts) *d_counts = p->d_counts;
  if (d_offsets) *d_offsets = p->d_offsets;
  if (d_perm) *d_perm = p->d_perm;
  return IKBO_OK;
}

ikbo_status_t ikbo_plan_worklist(ikbo_plan_t p, const int32_t** d_work, const int32_t** d_n_units,
                                 int* cands_per_unit, int* max_units) {
  if (!p) return IKBO_ERR_INVALID_ARG;
  if (!p->planned) return IKBO_ERR_NOT_PLANNED;
  if (d_work) *d_work = p->d_work;
  if (d_n_units) *d_n_units = p->d_n_units;
  if (cands_per_unit) *cands_per_unit = p->cands_per_unit;
  if (max_units) *max_units = static_cast<int>(p->max_units);
  return IKBO_OK;
}

ikbo_status_t ikbo_plan_get_status(ikbo_plan_t p, cudaStream_t stream) {
  if (!p) return IKBO_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return IKBO_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, p->d_status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return IKBO_ERR_CUDA;
  if (word && cudaMemset(p->d_status, 0, sizeof(uint32_t)) != cudaSuccess) return IKBO_ERR_CUDA;
  if (word & DEV_ERR_MAP_RANGE) return IKBO_ERR_MAP_OUT_OF_RANGE;
  if (word & (DEV_ERR_FLAG_TIMEOUT | DEV_ERR_PIPE_TIMEOUT)) return IKBO_ERR_TIMEOUT;
  if (word & (DEV_ERR_BAD_WORK | DEV_ERR_SMEM_LAYOUT)) return IKBO_ERR_INTERNAL;
  return IKBO_OK;
}

ikbo_status_t ikbo_lce_forward(ikbo_plan_t p, const void* U, const void* C, const void* Wu, const void* Wc,
                               const void* b, void* Y, int K_u, int K_c, int D, int N, cudaStream_t stream) {
  return lce_launch(p, U, C, Wu, Wc, b, Y, K_u, K_c, D, N, 4, stream);
}

ikbo_status_t ikbo_lce_forward_staged(ikbo_plan_t p, const void* U, const void* C, const void* Wu, const void* Wc,
                                      const void* b, void* Y, int K_u, int K_c, int D, int N, int stage,
                                      cudaStream_t stream) {
  if (stage != 1 && stage != 3 && stage != 4) return IKBO_ERR_INVALID_ARG;
  return lce_launch(p, U, C, Wu, Wc, b, Y, K_u, K_c, D, N, stage, stream);
}


ikbo_status_t ikbo_lce_backward(ikbo_plan_t p, const void* U, const void* C, const void* Wu, const void* Wc,
                                const void* dY, void* dU, void* dC, float* dWu, float* dWc, float* db, int K_u,
                                int K_c, int D, int N, cudaStream_t stream) {
  if (!p) return IKBO_ERR_INVALID_ARG;
  if (!p->planned) return IKBO_ERR_NOT_PLANNED;
  if (!dY || (dU && !Wu) || (dC && !Wc) || (dWu && !U) || (dWc && !C)) return IKBO_ERR_INVALID_ARG;
  const void* ptrs[] = {U, C, Wu, Wc, dY, dU, dC, dWu, dWc, db};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return IKBO_ERR_INVALID_ARG;
  if (K_u < 1 || K_c < 1 || D < 1 || N < 1) return IKBO_ERR_UNSUPPORTED;
  if (D % 8 != 0 || N % 8 != 0 || N > 256) return IKBO_ERR_UNSUPPORTED;
  const int n_cand = p->n_cand, n_users = p->n_users;

  // configure every product that is asked for before launching anything.
  // Where the shape allows it (K_c <= 256, N <= 192) one candidate pass
  // reads dY and C once for dC, dW_c and the segment sum S (with db); else
  // a segment-sum kernel, the activation-gradient kernel (dC) and a
  // weight-gradient kernel (dW_c).  dU and dW_u read S at n_users.
  const bool need_S = dU || dWu || db;
  CandParams cp{};
  cp.n_cand = n_cand, cp.n_users = n_users, cp.K_c = K_c, cp.D = D, cp.N = N;
  const bool use_cand = (dC || dWc || need_S) && bwd_cand_configure(&cp, p->max_smem);
  const int cgrid = use_cand ? bwd_cand_grid(cp, p->num_sms) : 0;
  ActParams ac{}, au{};
  WgradParams wc{}, wu{};
  ac.B = n_cand, ac.M = K_c, ac.D = D, ac.N = N;
  au.B = n_users, au.M = K_u, au.D = D, au.N = N;
  wc.B = n_cand, wc.M = K_c, wc.D = D, wc.N = N;
  wu.M = K_u, wu.D = D, wu.N = N;
  wu.B = 2 * n_users;  // G = the hi/lo pair of S per user; A = U[b >> 1]
  wu.a_shift = 1;
  // dU splits K_u over more CTAs only when it runs alone: beside dW_u, whose
  // split-K CTAs form clusters, its 30 CTAs at 70:1 leave room for them
  // (118.4 vs 123.5 us for the call at 70:1; alone, dU takes 57.0 us split
  // and 61.1 unsplit, both timed with the candidate pass before it)
  if ((!use_cand && dC && !bwd_act_configure(&ac, p->max_smem, false, p->num_sms, false)) ||
      (dU && !bwd_act_configure(&au, p->max_smem, true, p->num_sms, dWu == nullptr)) ||
      (!use_cand && dWc && !bwd_wgrad_configure(&wc, p->num_sms, p->max_smem)) ||
      (dWu && !bwd_wgrad_configure(&wu, p->num_sms, p->max_smem)))
    return IKBO_ERR_UNSUPPORTED;

  const int ND = N * D;
  const int NP = (N + 63) / 64 * 64;  // rows per half of the hi/lo pair
  SegSumParams sp{};
  const size_t n_ctrl = 2;
  if (need_S) {
    sp.nch = bwd_segsum_chunks(n_cand, n_users, ND, p->num_sms);
    sp.slices = (ND + BWD_SEG_SLICE - 1) / BWD_SEG_SLICE;
    sp.NPD = NP * D;
    const size_t nS = static_cast<size_t>(n_users) * ND;
    if (grow(&p->d_bwd_Sb, &p->bwd_Sb_elems, static_cast<size_t>(n_users) * 2 * NP * D, stream) != cudaSuccess)
      return IKBO_ERR_CUDA;
    if (!use_cand && (grow(&p->d_bwd_S, &p->bwd_S_elems, nS, stream) != cudaSuccess ||
                      (sp.nch > 1 && grow(&p->d_bwd_seg, &p->bwd_seg_elems, nS * sp.nch, stream) != cudaSuccess)))
      return IKBO_ERR_CUDA;
    if (use_cand &&
        (grow(&p->d_bwd_spart, &p->bwd_spart_elems, static_cast<size_t>(cgrid) * 2 * N * 64, stream) != cudaSuccess ||
         grow(&p->d_bwd_dbcta, &p->bwd_dbcta_elems, static_cast<size_t>(cgrid) * N, stream) != cudaSuccess))
      return IKBO_ERR_CUDA;
  }
  if (use_cand && grow(&p->d_bwd_ctrl, &p->bwd_ctrl_elems, n_ctrl, stream) != cudaSuccess) return IKBO_ERR_CUDA;
  size_t wpart = 0;
  if (dWc) wpart = use_cand ? static_cast<size_t>(cp.n_mblk) * cgrid * 128 * N : bwd_wgrad_part_elems(wc);
  if (dWu && bwd_wgrad_part_elems(wu) > wpart) wpart = bwd_wgrad_part_elems(wu);
  if (wpart && grow(&p->d_bwd_wpart, &p->bwd_wpart_elems, wpart, stream) != cudaSuccess) return IKBO_ERR_CUDA;

  // tensor maps: [B][rows][D] operands with 64-wide boxes along D (rows 64 or
  // 128 high), and the weights as [M][N] with 64-wide boxes along N
  const uint64_t dyd[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(N), static_cast<uint64_t>(n_cand)};
  const uint64_t dys[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(N) * D * 2};
  // S2 [n_users][2][NP][D]: as X of dU, 2 * NP rows per user; as G of dWu,
  // NP rows per (user, half)
  const uint64_t s2x[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(2 * NP), static_cast<uint64_t>(n_users)};
  const uint64_t s2xs[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(2 * NP) * D * 2};
  const uint64_t s2g[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(NP), static_cast<uint64_t>(2 * n_users)};
  const uint64_t s2gs[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(NP) * D * 2};
  const uint32_t box64[3] = {64, 64, 1};
  const uint32_t box128[3] = {64, 128, 1};
  const uint32_t wbox[2] = {64, 128};
  CUtensorMap tmDY, tmSX, tmSG, tmWc, tmWu, tmC, tmU;
  if (!encode_bf16(&tmDY, dY, 3, dyd, dys, box64)) return IKBO_ERR_CUDA;
  tmWc = tmDY;  // placeholders, not read where the product is not asked for
  tmC = tmDY;
  if (need_S && (!encode_bf16(&tmSX, p->d_bwd_Sb, 3, s2x, s2xs, box64) ||
                 !encode_bf16(&tmSG, p->d_bwd_Sb, 3, s2g, s2gs, box64)))
    return IKBO_ERR_CUDA;
  if (dC) {
    const uint64_t wd[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K_c)};
    const uint64_t ws[1] = {static_cast<uint64_t>(N) * 2};
    if (!encode_bf16(&tmWc, Wc, 2, wd, ws, wbox)) return IKBO_ERR_CUDA;
  }
  if (dU) {
    const uint64_t wd[2] = {static_cast<uint64_t>(N), static_cast<uint64_t>(K_u)};
    const uint64_t ws[1] = {static_cast<uint64_t>(N) * 2};
    if (!encode_bf16(&tmWu, Wu, 2, wd, ws, wbox)) return IKBO_ERR_CUDA;
  }
  if (dWc) {
    const uint64_t cd[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(K_c), static_cast<uint64_t>(n_cand)};
    const uint64_t cs[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(K_c) * D * 2};
    if (!encode_bf16(&tmC, C, 3, cd, cs, box128)) return IKBO_ERR_CUDA;
  }
  if (dWu) {
    const uint64_t ud[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(K_u), static_cast<uint64_t>(n_users)};
    const uint64_t us[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(K_u) * D * 2};
    if (!encode_bf16(&tmU, U, 3, ud, us, box128)) return IKBO_ERR_CUDA;
  }

  int launches = 0;
  cudaError_t e = cudaSuccess;
  // rows N .. NP-1 of each half of the S pair must read as zeros
  if (need_S && NP != N)
    e = cudaMemsetAsync(p->d_bwd_Sb, 0, sizeof(uint16_t) * static_cast<size_t>(n_users) * 2 * NP * D, stream);
  if (e == cudaSuccess && use_cand) {
    // the grid barrier's counts start at zero (the pass leaves them so; this
    // also covers a call that ended on a timeout)
    e = cudaMemsetAsync(p->d_bwd_ctrl, 0, sizeof(uint32_t) * n_ctrl, stream);
    cp.perm = p->d_perm;
    cp.map = p->d_map;
    cp.offsets = p->d_offsets;
    cp.dC = static_cast<uint16_t*>(dC);
    cp.wpart = dWc ? p->d_bwd_wpart : nullptr;
    cp.dWc = dWc;
    cp.S2 = need_S ? p->d_bwd_Sb : nullptr;
    cp.spart = p->d_bwd_spart;
    cp.dbcta = p->d_bwd_dbcta;
    cp.db = db;
    cp.ctrl = p->d_bwd_ctrl;
    cp.status = p->d_status;
    cp.NPD = NP * D;
    cp.G = cgrid;
    cp.timeout_ns = p->timeout_ns;
    int n = 0;
    const bool coop = (p->debug & DEBUG_NO_COOPERATIVE) == 0;
    if (e == cudaSuccess) e = launch_bwd_cand(tmDY, tmC, tmWc, cp, p->num_sms, coop, stream, &n);
    if (e == cudaSuccess) launches += n;
  } else if (e == cudaSuccess && need_S) {
    sp.dY = static_cast<const uint16_t*>(dY);
    sp.offsets = p->d_offsets;
    sp.perm = p->d_perm;
    sp.S = p->d_bwd_S;
    sp.S2 = p->d_bwd_Sb;
    sp.part = p->d_bwd_seg;
    sp.n_cand = n_cand;
    sp.n_users = n_users;
    sp.ND = ND;
    e = launch_bwd_segsum(sp, stream, &launches);
    if (e == cudaSuccess && db) {
      e = launch_bwd_db(p->d_bwd_S, db, n_users, N, D, stream);
      if (e == cudaSuccess) ++launches;
    }
  }
  if (e == cudaSuccess && dC && !use_cand) {
    ac.out = static_cast<uint16_t*>(dC);
    ac.status = p->d_status;
    ac.timeout_ns = p->timeout_ns;
    e = launch_bwd_act(tmDY, tmWc, ac, p->num_sms, stream);
    if (e == cudaSuccess) ++launches;
  }
  if (e == cudaSuccess && dWc && !use_cand) {
    wc.part = p->d_bwd_wpart;
    wc.status = p->d_status;
    wc.timeout_ns = p->timeout_ns;
    e = launch_bwd_wgrad(tmC, tmDY, wc, dWc, p->num_sms, stream, &launches);
  }
  // dU and dW_u both read S and nothing else of each other: with both asked
  // for, dW_u (and its reduce) runs on the plan's second stream beside dU
  // (fork and join through events, so the call stays ordered on `stream`)
  cudaStream_t wu_stream = stream;
  if (e == cudaSuccess && dU && dWu) {
    if ((!p->side && cudaStreamCreateWithFlags(&p->side, cudaStreamNonBlocking) != cudaSuccess) ||
        (!p->ev_fork && cudaEventCreateWithFlags(&p->ev_fork, cudaEventDisableTiming) != cudaSuccess) ||
        (!p->ev_join && cudaEventCreateWithFlags(&p->ev_join, cudaEventDisableTiming) != cudaSuccess))
      e = cudaErrorMemoryAllocation;
    if (e == cudaSuccess) e = cudaEventRecord(p->ev_fork, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->side, p->ev_fork, 0);
    if (e == cudaSuccess) wu_stream = p->side;
  }
  if (e == cudaSuccess && dWu) {
    wu.part = p->d_bwd_wpart;
    wu.status = p->d_status;
    wu.timeout_ns = p->timeout_ns;
    e = launch_bwd_wgrad(tmU, tmSG, wu, dWu, p->num_sms, wu_stream, &launches);
  }
  if (e == cudaSuccess && dU) {
    au.out = static_cast<uint16_t*>(dU);
    au.status = p->d_status;
    au.timeout_ns = p->timeout_ns;
    e = launch_bwd_act(tmSX, tmWu, au, p->num_sms, stream);
    if (e == cudaSuccess) ++launches;
  }
  if (wu_stream != stream) {  // join, also after a failed launch on either stream
    const cudaError_t e2 = cudaEventRecord(p->ev_join, wu_stream);
    const cudaError_t e3 = e2 == cudaSuccess ? cudaStreamWaitEvent(stream, p->ev_join, 0) : e2;
    if (e == cudaSuccess) e = e3;
  }
  p->launches += static_cast<uint64_t>(launches);
  return e == cudaSuccess ? IKBO_OK : IKBO_ERR_CUDA;
}

ikbo_status_t ikbo_attn_forward(ikbo_plan_t p, const void* Q, const void* K, const void* V,
                                const int32_t* d_kv_offsets, void* O, int Lkv, int d, float scale,
                                cudaStream_t stream) {
  return attn_launch(p, Q, nullptr, K, V, d_kv_offsets, O, nullptr, nullptr, 0, Lkv, d, scale, stream);
}

ikbo_status_t ikbo_attn_forward_lse(ikbo_plan_t p, const void* Q, const void* K, const void* V,
                                    const int32_t* d_kv_offsets, void* O, float* lse, int Lkv, int d, float scale,
                                    cudaStream_t stream) {
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return IKBO_ERR_INVALID_ARG;
  return attn_launch(p, Q, nullptr, K, V, d_kv_offsets, O, nullptr, lse, 0, Lkv, d, scale, stream);
}

ikbo_status_t ikbo_attn_self_target_forward(ikbo_plan_t p, const void* Q, const void* Q_user, const void* K,
                                            const void* V, const int32_t* d_kv_offsets, void* O, void* O_user,
                                            int Lq_u, int Lkv, int d, float scale, cudaStream_t stream) {
  if (!Q_user) return IKBO_ERR_INVALID_ARG;
  return attn_launch(p, Q, Q_user, K, V, d_kv_offsets, O, O_user, nullptr, Lq_u, Lkv, d, scale, stream);
}

}  // extern "C"
