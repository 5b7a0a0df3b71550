// attn_bwd.cu -- broadcast attention backward (training).
//
// The IKBO write-ups say the kernels serve training when candidates
// outnumber users ("Meta Optimizes Inference for Recommendation Systems",
// the paragraph on kernels, compilation and runtime) and give no backward;
// this is the chain rule of O[i,h] = softmax(scale Q[i,h] K[u,h]^T) V[u,h],
// u = map[i].  Per query row: p = softmax(s), dP = dO V^T, D = rowsum(dO * O),
// dS = p (dP - D);  dQ = scale dS K;  and, the broadcast's transpose, the
// K/V gradients of user u sum over every candidate of u:
//   dK[u,h] = scale sum_{i in seg u} dS_i^T Q_i,   dV[u,h] = sum_i P_i^T dO_i.
//
// Two persistent kernels, one CTA per SM, 8 warps: warp 0 TMA (elected lane
// issues), warp 1 tcgen05.mma (elected lane) and TMEM owner, warps 4-7 the
// element-wise work (thread = TMEM lane = one row, 128 columns each).
//   attn_bwd_dq_kernel    per work-list unit (a 128-row tile of up to
//                         floor(128/Lq) candidates' queries, as the forward):
//                         pass 1 forms LSE over the user's key tiles, pass 2
//                         dQ += dS K.  Stores LSE and D for the next kernel.
//   attn_bwd_dkdv_kernel  per (user, head, 128-key block): loops over the
//                         query tiles of all of the user's candidates.
// P and dS are rounded to bf16 for the tensor cores (as P is in the
// forward); every accumulation is fp32.  Every wait is bounded.
#include <cuda_bf16.h>
#include <math.h>

#include "ikbo_internal.h"
#include "ptx.cuh"

namespace ikbo {

namespace {

constexpr uint32_t TILE = 128 * 128 * 2;  // a 128-row x 128-d bf16 tile: two 64-d halves
constexpr uint32_t HALF = 128 * 64 * 2;   // 16 KB

// A wait taken by a whole warp; the lanes agree on the outcome.
__device__ __forceinline__ bool wwait(uint64_t* bar, uint32_t parity, uint32_t* abort, uint64_t timeout_ns) {
  const bool ok = mbar_wait(bar, parity, abort, timeout_ns, 1);
  return __all_sync(0xffffffffu, ok);
}

// Keys of user u and its first packed row (jagged) for the K/V tensor maps.
struct UserKeys {
  int L, kv0;
};
__device__ __forceinline__ UserKeys user_keys(const AttnBwdParams& p, int u) {
  UserKeys k;
  if (p.kv_offsets) {
    k.kv0 = p.kv_offsets[u];
    k.L = max(0, p.kv_offsets[u + 1] - k.kv0);
  } else {
    k.kv0 = 0;
    k.L = p.Lkv;
  }
  return k;
}

// K or V rows [row, row + 128) of (u, h) into a 32 KB tile (two 64-d boxes).
__device__ __forceinline__ void load_kv(const AttnBwdParams& p, const CUtensorMap* tm, uint8_t* dst, uint64_t* bar,
                                        int u, int h, int kv0, int row) {
  if (p.kv_offsets) {
    tma_load_3d(dst, tm, bar, 0, h, kv0 + row);
    tma_load_3d(dst + HALF, tm, bar, 64, h, kv0 + row);
  } else {
    tma_load_4d(dst, tm, bar, 0, row, h, u);
    tma_load_4d(dst + HALF, tm, bar, 64, row, h, u);
  }
}

// The query tile of candidates cand[0..cpt) (an empty slot holds n_cand:
// TMA reads it as zeros) from a [n_cand][H][Lq][d] tensor into a 32 KB tile.
__device__ __forceinline__ void load_qtile(const AttnBwdParams& p, const CUtensorMap* tm, uint8_t* dst,
                                           uint64_t* bar, int h, const int* cand) {
  for (int j = 0; j < p.cands_per_tile; ++j) {
    uint8_t* d = dst + j * p.Lq * 128;
    tma_load_4d(d, tm, bar, 0, 0, h, cand[j]);
    tma_load_4d(d + HALF, tm, bar, 64, 0, h, cand[j]);
  }
}

// S (or S^T, dP, dP^T) = A B^T over d = 128: both tiles K-major (rows of
// 128 bytes per 64-d half), 8 steps of 16 d.
__device__ __forceinline__ void mma_rows_dot(uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
  const uint64_t ad = sdesc_sw128(a_base, 16, 1024);
  const uint64_t bd = sdesc_sw128(b_base, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = ((ks >> 2) * HALF + (ks & 3) * 32) >> 4;
    mma_bf16_ss(d_tmem, ad + off, bd + off, idesc, ks > 0 ? 1u : 0u);
  }
}

// D += A B with A from TMEM (bf16 pairs, 128 rows x 128 k = 64 columns) and B
// a [k rows][128 d] tile read MN-major (d contiguous), 8 steps of 16 k.
__device__ __forceinline__ void mma_tmem_by_tile(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, true);
  const uint64_t bd = sdesc_sw128(b_base, HALF, 1024);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_bf16_ts(d_tmem, a_tmem + ks * 8, bd + ((ks * 2048u) >> 4), idesc, (accumulate || ks > 0) ? 1u : 0u);
}

// Zero rows [r0, 128) of a 32 KB tile (both halves; the swizzle only moves
// 16-byte chunks within a row).
__device__ __forceinline__ void zero_rows(uint8_t* tile, int r0, int tid, int nthreads) {
  const int per_half = (128 - r0) * 8;  // 16-byte chunks
  for (int c = tid; c < 2 * per_half; c += nthreads) {
    const int hf = c / per_half, k = c - hf * per_half;
    reinterpret_cast<uint4*>(tile + hf * HALF + r0 * 128)[k] = make_uint4(0, 0, 0, 0);
  }
}

// ================================================================ dQ kernel
// TMEM columns: S [0,128), dP [128,256), dS (bf16 pairs) [256,320), dQ [320,448).
constexpr uint32_t TQ_S = 0, TQ_DP = 128, TQ_DS = 256, TQ_DQ = 320;
constexpr int DQ_K_STAGES = 2, DQ_V_STAGES = 2;

struct DqSmem {
  uint8_t* q;   // 32 KB
  uint8_t* go;  // dO tile, 32 KB
  uint8_t* k;   // DQ_K_STAGES x 32 KB
  uint8_t* v;   // DQ_V_STAGES x 32 KB
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* k_full;
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* s_full;   // S (pass 1) or S and dP (pass 2) computed
  uint64_t* s_free;   // ... and read by the element-wise warps
  uint64_t* ds_full;  // dS written to TMEM
  uint64_t* dq_done;  // a dQ += dS K completed (dS may be overwritten)
  uint64_t* dq_free;  // the unit's dQ was read out
  uint32_t* tmem_slot;
  uint32_t* abort;
};
constexpr uint32_t DQ_TILES = (2 + DQ_K_STAGES + DQ_V_STAGES) * TILE;
constexpr uint32_t DQ_SMEM = 1024 + DQ_TILES + 8 * (2 + 2 * DQ_K_STAGES + 2 * DQ_V_STAGES + 5) + 8;

__device__ __forceinline__ DqSmem dq_carve(uint8_t* base) {
  DqSmem s;
  s.q = base;
  s.go = base + TILE;
  s.k = base + 2 * TILE;
  s.v = s.k + DQ_K_STAGES * TILE;
  uint64_t* b = reinterpret_cast<uint64_t*>(base + DQ_TILES);
  s.q_full = b;
  s.q_empty = b + 1;
  s.k_full = b + 2;
  s.k_empty = s.k_full + DQ_K_STAGES;
  s.v_full = s.k_empty + DQ_K_STAGES;
  s.v_empty = s.v_full + DQ_V_STAGES;
  s.s_full = s.v_empty + DQ_V_STAGES;
  s.s_free = s.s_full + 1;
  s.ds_full = s.s_free + 1;
  s.dq_done = s.ds_full + 1;
  s.dq_free = s.dq_done + 1;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.dq_free + 1);
  s.abort = s.tmem_slot + 1;
  return s;
}

// A work-list unit: user, head, its candidates perm[start .. start+cnt).
struct QUnit {
  int u, h, start, cnt, ntiles;
  UserKeys k;
  bool ok;
};
__device__ __forceinline__ QUnit dq_unit(const AttnBwdParams& p, int unit) {
  const int4 w = __ldg(reinterpret_cast<const int4*>(p.work) + unit);
  QUnit x;
  x.u = w.x;
  x.h = w.y;
  x.start = w.z;
  x.cnt = w.w;
  x.ok = x.u >= 0 && x.u < p.n_users && x.h >= 0 && x.h < p.H && x.cnt >= 1 && x.cnt <= p.cands_per_tile &&
         x.start >= 0 && x.start + x.cnt <= p.n_cand;
  x.k = x.ok ? user_keys(p, x.u) : UserKeys{0, 0};
  x.ntiles = (x.k.L + 127) / 128;
  return x;
}

__global__ void __launch_bounds__(ABWD_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const AttnBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const DqSmem s = dq_carve(base);
  const int warp = threadIdx.x >> 5;
  const int n_units = *p.n_units;
  const int rows = p.cands_per_tile * p.Lq;
  // tile rows past the candidates' slots are never written by TMA: zero them once
  zero_rows(s.q, rows, threadIdx.x, ABWD_THREADS);
  zero_rows(s.go, rows, threadIdx.x, ABWD_THREADS);
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(s.q_full, 1);
    mbar_init(s.q_empty, 1);
    for (int i = 0; i < DQ_K_STAGES; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < DQ_V_STAGES; ++i) {
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    mbar_init(s.s_full, 1);
    mbar_init(s.s_free, 128);
    mbar_init(s.ds_full, 128);
    mbar_init(s.dq_done, 1);
    mbar_init(s.dq_free, 128);
    *s.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;

  if (warp == 0) {
    // ---- TMA: Q and dO tiles per unit; K tiles (pass 1), K and V tiles (pass 2)
    uint32_t qc = 0, kc = 0, vc = 0;
    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
      const QUnit x = dq_unit(p, unit);
      if (!x.ok) {
        if (lane_id() == 0) atomicOr(p.status, DEV_ERR_BAD_WORK);
        continue;
      }
      if (x.ntiles == 0) continue;
      int cand[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) cand[j] = j < x.cnt ? __ldg(p.perm + x.start + j) : p.n_cand;
      if (!wwait(s.q_empty, (qc & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
      ++qc;
      if (elect_one()) {
        mbar_arrive_expect_tx(s.q_full, 2u * static_cast<uint32_t>(rows) * 256u);
        load_qtile(p, &tmQ, s.q, s.q_full, x.h, cand);
        load_qtile(p, &tmDO, s.go, s.q_full, x.h, cand);
      }
      __syncwarp();
      for (int pass = 0; pass < 2; ++pass)
        for (int jt = 0; jt < x.ntiles; ++jt) {
          const int ks = static_cast<int>(kc % DQ_K_STAGES);
          if (!wwait(&s.k_empty[ks], ((kc / DQ_K_STAGES) & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
          if (elect_one()) {
            mbar_arrive_expect_tx(&s.k_full[ks], TILE);
            load_kv(p, &tmK, s.k + ks * TILE, &s.k_full[ks], x.u, x.h, x.k.kv0, jt * 128);
          }
          __syncwarp();
          ++kc;
          if (pass == 1) {
            const int vs = static_cast<int>(vc % DQ_V_STAGES);
            if (!wwait(&s.v_empty[vs], ((vc / DQ_V_STAGES) & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
            if (elect_one()) {
              mbar_arrive_expect_tx(&s.v_full[vs], TILE);
              load_kv(p, &tmV, s.v + vs * TILE, &s.v_full[vs], x.u, x.h, x.k.kv0, jt * 128);
            }
            __syncwarp();
            ++vc;
          }
        }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    uint32_t qc = 0, kc = 0, vc = 0, ns = 0, nds = 0, nu = 0;
    const uint32_t q_base = smem_u32(s.q), go_base = smem_u32(s.go);
    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
      const QUnit x = dq_unit(p, unit);
      if (!x.ok || x.ntiles == 0) continue;
      if (!wwait(s.q_full, qc & 1u, s.abort, p.timeout_ns)) goto done;
      ++qc;
      for (int jt = 0; jt < x.ntiles; ++jt) {  // pass 1: S only
        const int ks = static_cast<int>(kc % DQ_K_STAGES);
        if (!wwait(&s.k_full[ks], (kc / DQ_K_STAGES) & 1u, s.abort, p.timeout_ns)) goto done;
        if (ns > 0 && !wwait(s.s_free, (ns - 1) & 1u, s.abort, p.timeout_ns)) goto done;
        tc_fence_after();
        if (elect_one()) {
          mma_rows_dot(tmem + TQ_S, q_base, smem_u32(s.k + ks * TILE));
          mma_commit(s.s_full);
          mma_commit(&s.k_empty[ks]);
        }
        __syncwarp();
        ++ns;
        ++kc;
      }
      for (int jt = 0; jt < x.ntiles; ++jt) {  // pass 2: S, dP, then dQ += dS K
        const int ks = static_cast<int>(kc % DQ_K_STAGES);
        const int vs = static_cast<int>(vc % DQ_V_STAGES);
        const uint32_t k_base = smem_u32(s.k + ks * TILE);
        if (!wwait(&s.k_full[ks], (kc / DQ_K_STAGES) & 1u, s.abort, p.timeout_ns)) goto done;
        if (!wwait(&s.v_full[vs], (vc / DQ_V_STAGES) & 1u, s.abort, p.timeout_ns)) goto done;
        if (!wwait(s.s_free, (ns - 1) & 1u, s.abort, p.timeout_ns)) goto done;
        tc_fence_after();
        if (elect_one()) {
          mma_rows_dot(tmem + TQ_S, q_base, k_base);
          mma_rows_dot(tmem + TQ_DP, go_base, smem_u32(s.v + vs * TILE));
          mma_commit(s.s_full);
          mma_commit(&s.v_empty[vs]);
          if (jt + 1 == x.ntiles) mma_commit(s.q_empty);  // last reader of Q and dO
        }
        __syncwarp();
        ++ns;
        ++vc;
        if (!wwait(s.ds_full, nds & 1u, s.abort, p.timeout_ns)) goto done;
        ++nds;
        if (jt == 0 && nu > 0 && !wwait(s.dq_free, (nu - 1) & 1u, s.abort, p.timeout_ns)) goto done;
        tc_fence_after();
        if (elect_one()) {
          mma_tmem_by_tile(tmem + TQ_DQ, tmem + TQ_DS, k_base, jt > 0);
          mma_commit(s.dq_done);
          mma_commit(&s.k_empty[ks]);
        }
        __syncwarp();
        ++kc;
      }
      ++nu;
    }
  } else if (warp >= 4) {
    // ---- element-wise warps: thread = TMEM lane = query row r of the tile
    const int quarter = warp - 4;
    const int r = quarter * 32 + static_cast<int>(lane_id());
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const float sl = p.scale_log2;
    uint32_t ns = 0, ndq = 0;
    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
      const QUnit x = dq_unit(p, unit);
      if (!x.ok) continue;
      const int slot = r / p.Lq, q = r - slot * p.Lq;
      const bool valid = r < rows && slot < x.cnt;
      const int cand = valid ? __ldg(p.perm + x.start + slot) : 0;
      const size_t row = (static_cast<size_t>(cand) * p.H + x.h) * p.Lq + q;
      uint4* dq_row = reinterpret_cast<uint4*>(p.dQ + row * 128);
      if (x.ntiles == 0) {  // no keys: dQ = 0; no row of this user reaches the dK/dV kernel
        if (valid) {
#pragma unroll
          for (int c = 0; c < 16; ++c) dq_row[c] = make_uint4(0, 0, 0, 0);
          p.lse[row] = INFINITY;
          p.Drow[row] = 0.f;
        }
        continue;
      }
      // D = rowsum(dO * O)
      float D = 0.f;
      if (valid) {
        const uint4* orow = reinterpret_cast<const uint4*>(p.O + row * 128);
        const uint4* grow = reinterpret_cast<const uint4*>(p.dO + row * 128);
#pragma unroll 4
        for (int c = 0; c < 16; ++c) {
          const uint4 a = __ldg(orow + c), g = __ldg(grow + c);
          const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            D = fmaf(__uint_as_float(aw[k] << 16), __uint_as_float(gw[k] << 16), D);
            D = fmaf(__uint_as_float(aw[k] & 0xffff0000u), __uint_as_float(gw[k] & 0xffff0000u), D);
          }
        }
      }
      // pass 1: m, l over the user's keys (log2 domain)
      float m = -INFINITY, l = 0.f;
      for (int jt = 0; jt < x.ntiles; ++jt) {
        if (!wwait(s.s_full, ns & 1u, s.abort, p.timeout_ns)) goto done;
        ++ns;
        tc_fence_after();
        const int ncols = min(128, x.k.L - jt * 128);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + TQ_S + c * 32, v);
          tmem_ld_wait(v);
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j < ncols) mx = fmaxf(mx, __uint_as_float(v[j]) * sl);
          const float m_new = fmaxf(m, mx);
          if (m_new == -INFINITY) continue;
          float add = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j < ncols) add += ex2(fmaf(__uint_as_float(v[j]), sl, -m_new));
          l = l * ex2(m - m_new) + add;
          m = m_new;
        }
        tc_fence_before();
        mbar_arrive(s.s_free);
      }
      const float lse2 = (valid && l > 0.f) ? m + __log2f(l) : INFINITY;
      if (valid) {
        p.lse[row] = lse2;
        p.Drow[row] = D;
      }
      // pass 2: dS = P (dP - D) scale -> TMEM (bf16 pairs)
      for (int jt = 0; jt < x.ntiles; ++jt) {
        if (!wwait(s.s_full, ns & 1u, s.abort, p.timeout_ns)) goto done;
        ++ns;
        if (jt > 0) {  // the previous dQ MMA has read dS
          if (!wwait(s.dq_done, ndq & 1u, s.abort, p.timeout_ns)) goto done;
          ++ndq;
        }
        tc_fence_after();
        const int ncols = min(128, x.k.L - jt * 128);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t sv[32], dv[32], pk[16];
          tmem_ld32(tmem + lane_base + TQ_S + c * 32, sv);
          tmem_ld_wait(sv);
          tmem_ld32(tmem + lane_base + TQ_DP + c * 32, dv);
          tmem_ld_wait(dv);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int c0 = c * 32 + 2 * j;
            const float p0 = c0 < ncols ? ex2(fmaf(__uint_as_float(sv[2 * j]), sl, -lse2)) : 0.f;
            const float p1 = c0 + 1 < ncols ? ex2(fmaf(__uint_as_float(sv[2 * j + 1]), sl, -lse2)) : 0.f;
            pk[j] = pack_bf16x2(p0 * (__uint_as_float(dv[2 * j]) - D) * p.scale,
                                p1 * (__uint_as_float(dv[2 * j + 1]) - D) * p.scale);
          }
          tmem_st16(tmem + lane_base + TQ_DS + c * 16, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(s.s_free);
        mbar_arrive(s.ds_full);
      }
      // epilogue: dQ (fp32 TMEM) -> bf16 row
      if (!wwait(s.dq_done, ndq & 1u, s.abort, p.timeout_ns)) goto done;
      ++ndq;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + TQ_DQ + c * 32, v);
        tmem_ld_wait(v);
        if (valid) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            dq_row[c * 4 + k] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                                           pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                                           pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                                           pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
        }
      }
      tc_fence_before();
      mbar_arrive(s.dq_free);
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (*s.abort && threadIdx.x == 0) atomicOr(p.status, DEV_ERR_PIPE_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================= dK/dV kernel
// TMEM columns: S^T [0,128) (then P^T as bf16 pairs in [0,64)), dP^T [128,256)
// (then dS^T in [128,192)), dV [256,384), dK [384,512).  Each P^T / dS^T
// chunk is written over columns its own chunk of S^T / dP^T has been read from.
constexpr uint32_t TK_ST = 0, TK_DPT = 128, TK_DV = 256, TK_DK = 384;

struct KvSmem {
  uint8_t* k;      // 32 KB, the key block
  uint8_t* v;      // 32 KB
  uint8_t* q;      // 2 x 32 KB query tiles
  uint8_t* go;     // 2 x 32 KB dO tiles
  float* lse;      // [2][128]
  float* drow;     // [2][128]
  uint64_t* kv_full;
  uint64_t* kv_empty;
  uint64_t* q_full;   // [2]
  uint64_t* q_empty;  // [2]
  uint64_t* st_full;  // S^T and dP^T computed
  uint64_t* pds_full; // P^T and dS^T written
  uint64_t* pv_done;  // dV, dK products of a tile completed
  uint64_t* acc_free; // the block's dV, dK read out
  uint32_t* tmem_slot;
  uint32_t* abort;
};
constexpr uint32_t KV_TILES = 6 * TILE;
constexpr uint32_t KV_SMEM = 1024 + KV_TILES + 4 * 2 * 128 * 4 + 8 * 10 + 8;

__device__ __forceinline__ KvSmem kv_carve(uint8_t* base) {
  KvSmem s;
  s.k = base;
  s.v = base + TILE;
  s.q = base + 2 * TILE;
  s.go = base + 4 * TILE;
  s.lse = reinterpret_cast<float*>(base + KV_TILES);
  s.drow = s.lse + 2 * 128;
  uint64_t* b = reinterpret_cast<uint64_t*>(s.drow + 2 * 128);
  s.kv_full = b;
  s.kv_empty = b + 1;
  s.q_full = b + 2;
  s.q_empty = b + 4;
  s.st_full = b + 6;
  s.pds_full = b + 7;
  s.pv_done = b + 8;
  s.acc_free = b + 9;
  s.tmem_slot = reinterpret_cast<uint32_t*>(b + 10);
  s.abort = s.tmem_slot + 1;
  return s;
}

// Item = (global key block gb, head h), gb over the users' key blocks in
// user order (blk_prefix[u] = blocks of users before u).
struct KvItem {
  int u, h, kb;
  UserKeys k;
  int seg0, count, ntq;  // the user's candidates perm[seg0 .. seg0+count), ntq query tiles
};
__device__ __forceinline__ KvItem kv_item(const AttnBwdParams& p, int item) {
  KvItem x;
  x.h = item % p.H;
  const int gb = item / p.H;
  int lo = 0, hi = p.n_users - 1;  // the user whose blocks contain gb
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.blk_prefix + mid) <= gb) lo = mid; else hi = mid - 1;
  }
  x.u = lo;
  x.kb = gb - __ldg(p.blk_prefix + lo);
  x.k = user_keys(p, x.u);
  x.seg0 = __ldg(p.offsets + x.u);
  x.count = __ldg(p.offsets + x.u + 1) - x.seg0;
  x.ntq = (x.count + p.cands_per_tile - 1) / p.cands_per_tile;
  return x;
}

__global__ void __launch_bounds__(ABWD_THREADS, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                         const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                         const AttnBwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const KvSmem s = kv_carve(base);
  const int warp = threadIdx.x >> 5;
  const int n_items = __ldg(p.blk_prefix + p.n_users) * p.H;
  const int cpt = p.cands_per_tile, rows = cpt * p.Lq;
  for (int b = 0; b < 2; ++b) {
    zero_rows(s.q + b * TILE, rows, threadIdx.x, ABWD_THREADS);
    zero_rows(s.go + b * TILE, rows, threadIdx.x, ABWD_THREADS);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(s.kv_full, 1);
    mbar_init(s.kv_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.q_full[b], 1);
      mbar_init(&s.q_empty[b], 1);
    }
    mbar_init(s.st_full, 1);
    mbar_init(s.pds_full, 128);
    mbar_init(s.pv_done, 1);
    mbar_init(s.acc_free, 128);
    *s.abort = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;

  if (warp == 0) {
    // ---- TMA: the key block's K and V, then per query tile Q, dO (TMA) and
    // the rows' LSE and D (plain loads by the warp's lanes)
    uint32_t ni = 0, tq = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const KvItem x = kv_item(p, item);
      if (x.ntq == 0) continue;
      if (ni > 0 && !wwait(s.kv_empty, (ni - 1) & 1u, s.abort, p.timeout_ns)) goto done;
      ++ni;
      if (elect_one()) {
        mbar_arrive_expect_tx(s.kv_full, 2 * TILE);
        load_kv(p, &tmK, s.k, s.kv_full, x.u, x.h, x.k.kv0, x.kb * 128);
        load_kv(p, &tmV, s.v, s.kv_full, x.u, x.h, x.k.kv0, x.kb * 128);
      }
      __syncwarp();
      for (int t = 0; t < x.ntq; ++t, ++tq) {
        const int b = static_cast<int>(tq & 1u);
        if (!wwait(&s.q_empty[b], ((tq >> 1) & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
        const int first = t * cpt, n = min(cpt, x.count - first);
        int cand[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) cand[j] = j < n ? __ldg(p.perm + x.seg0 + first + j) : p.n_cand;
        for (int r = static_cast<int>(lane_id()); r < 128; r += 32) {
          const int slot = r / p.Lq, q = r - slot * p.Lq;
          float lse = INFINITY, dr = 0.f;  // rows without a query: P = 0
          if (r < rows && slot < n) {
            const size_t row = (static_cast<size_t>(__ldg(p.perm + x.seg0 + first + slot)) * p.H + x.h) * p.Lq + q;
            lse = p.lse[row];
            dr = p.Drow[row];
          }
          s.lse[b * 128 + r] = lse;
          s.drow[b * 128 + r] = dr;
        }
        __syncwarp();
        if (elect_one()) {
          mbar_arrive_expect_tx(&s.q_full[b], 2u * static_cast<uint32_t>(rows) * 256u);
          load_qtile(p, &tmQ, s.q + b * TILE, &s.q_full[b], x.h, cand);
          load_qtile(p, &tmDO, s.go + b * TILE, &s.q_full[b], x.h, cand);
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer
    uint32_t ni = 0, tq = 0;
    const uint32_t k_base = smem_u32(s.k), v_base = smem_u32(s.v);
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const KvItem x = kv_item(p, item);
      if (x.ntq == 0) continue;
      if (!wwait(s.kv_full, ni & 1u, s.abort, p.timeout_ns)) goto done;
      for (int t = 0; t < x.ntq; ++t, ++tq) {
        const int b = static_cast<int>(tq & 1u);
        const uint32_t q_base = smem_u32(s.q + b * TILE), go_base = smem_u32(s.go + b * TILE);
        if (!wwait(&s.q_full[b], (tq >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
        // S^T and dP^T overwrite the previous tile's P^T and dS^T: wait for their readers
        if (tq > 0 && !wwait(s.pv_done, (tq - 1) & 1u, s.abort, p.timeout_ns)) goto done;
        tc_fence_after();
        if (elect_one()) {
          mma_rows_dot(tmem + TK_ST, k_base, q_base);
          mma_rows_dot(tmem + TK_DPT, v_base, go_base);
          mma_commit(s.st_full);
          if (t + 1 == x.ntq) mma_commit(s.kv_empty);  // last reader of K and V
        }
        __syncwarp();
        if (!wwait(s.pds_full, tq & 1u, s.abort, p.timeout_ns)) goto done;
        if (t == 0 && ni > 0 && !wwait(s.acc_free, (ni - 1) & 1u, s.abort, p.timeout_ns)) goto done;
        tc_fence_after();
        if (elect_one()) {
          mma_tmem_by_tile(tmem + TK_DV, tmem + TK_ST, go_base, t > 0);  // dV += P^T dO
          mma_tmem_by_tile(tmem + TK_DK, tmem + TK_DPT, q_base, t > 0);  // dK += dS^T Q
          mma_commit(s.pv_done);
          mma_commit(&s.q_empty[b]);
        }
        __syncwarp();
      }
      ++ni;
    }
  } else if (warp >= 4) {
    // ---- element-wise warps: thread = TMEM lane = key row of the block
    const int quarter = warp - 4;
    const int rk = quarter * 32 + static_cast<int>(lane_id());
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const float sl = p.scale_log2;
    uint32_t tq = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const KvItem x = kv_item(p, item);
      const int key = x.kb * 128 + rk;
      const bool kvalid = key < x.k.L;
      const size_t krow = p.kv_offsets ? (static_cast<size_t>(x.k.kv0 + key) * p.H + x.h)
                                       : ((static_cast<size_t>(x.u) * p.H + x.h) * p.Lkv + key);
      uint4* dk_row = reinterpret_cast<uint4*>(p.dK + krow * 128);
      uint4* dv_row = reinterpret_cast<uint4*>(p.dV + krow * 128);
      if (x.ntq == 0) {  // no candidate reads these keys: zero gradients
        if (kvalid) {
#pragma unroll
          for (int c = 0; c < 16; ++c) dk_row[c] = dv_row[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      for (int t = 0; t < x.ntq; ++t, ++tq) {
        const int b = static_cast<int>(tq & 1u);
        // the producer's lanes stored this tile's LSE and D before arriving on q_full[b]
        if (!wwait(&s.q_full[b], (tq >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
        if (!wwait(s.st_full, tq & 1u, s.abort, p.timeout_ns)) goto done;
        tc_fence_after();
        const float* lse = s.lse + b * 128;
        const float* drow = s.drow + b * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t sv[32], dv[32], pp[16], pd[16];
          tmem_ld32(tmem + lane_base + TK_ST + c * 32, sv);
          tmem_ld_wait(sv);
          tmem_ld32(tmem + lane_base + TK_DPT + c * 32, dv);
          tmem_ld_wait(dv);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int q0 = c * 32 + 2 * j;
            const float p0 = kvalid ? ex2(fmaf(__uint_as_float(sv[2 * j]), sl, -lse[q0])) : 0.f;
            const float p1 = kvalid ? ex2(fmaf(__uint_as_float(sv[2 * j + 1]), sl, -lse[q0 + 1])) : 0.f;
            pp[j] = pack_bf16x2(p0, p1);
            pd[j] = pack_bf16x2(p0 * (__uint_as_float(dv[2 * j]) - drow[q0]) * p.scale,
                                p1 * (__uint_as_float(dv[2 * j + 1]) - drow[q0 + 1]) * p.scale);
          }
          tmem_st16(tmem + lane_base + TK_ST + c * 16, pp);
          tmem_st16(tmem + lane_base + TK_DPT + c * 16, pd);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(s.pds_full);
      }
      // epilogue: the block's dV and dK rows
      if (!wwait(s.pv_done, (tq - 1) & 1u, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
#pragma unroll 1
      for (int g = 0; g < 2; ++g) {
        uint4* out = g == 0 ? dv_row : dk_row;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + (g == 0 ? TK_DV : TK_DK) + c * 32, v);
          tmem_ld_wait(v);
          if (kvalid) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
              out[c * 4 + k] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                                          pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                                          pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                                          pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
          }
        }
      }
      tc_fence_before();
      mbar_arrive(s.acc_free);
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (*s.abort && threadIdx.x == 0) atomicOr(p.status, DEV_ERR_PIPE_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// blk_prefix[u] = sum over users v < u of ceil(L_v / 128); one CTA, a scan
// over chunks of users.
__global__ void __launch_bounds__(1024) attn_bwd_blocks_kernel(const int32_t* kv_offsets, int n_users, int Lkv,
                                                               int32_t* blk_prefix) {
  __shared__ int32_t part[1024];
  const int per = (n_users + 1023) / 1024;
  const int u0 = threadIdx.x * per;
  int32_t sum = 0;
  for (int u = u0; u < min(u0 + per, n_users); ++u) {
    const int L = kv_offsets ? max(0, kv_offsets[u + 1] - kv_offsets[u]) : Lkv;
    sum += (L + 127) / 128;
  }
  part[threadIdx.x] = sum;
  __syncthreads();
  for (int w = 1; w < 1024; w <<= 1) {  // inclusive scan of the chunk sums
    const int32_t v = threadIdx.x >= w ? part[threadIdx.x - w] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int32_t run = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0;
  for (int u = u0; u < min(u0 + per, n_users); ++u) {
    blk_prefix[u] = run;
    const int L = kv_offsets ? max(0, kv_offsets[u + 1] - kv_offsets[u]) : Lkv;
    run += (L + 127) / 128;
  }
  if (threadIdx.x == 1023) blk_prefix[n_users] = part[1023];
}

}  // namespace

// ------------------------------------------------------------------- host
size_t attn_bwd_smem_bytes() { return DQ_SMEM > KV_SMEM ? DQ_SMEM : KV_SMEM; }

cudaError_t launch_attn_backward(const CUtensorMap& tmQ, const CUtensorMap& tmDO, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const AttnBwdParams& p, int grid, cudaStream_t s,
                                 int* launches) {
  *launches = 0;
  attn_bwd_blocks_kernel<<<1, 1024, 0, s>>>(p.kv_offsets, p.n_users, p.Lkv, const_cast<int32_t*>(p.blk_prefix));
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  e = cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
  if (e != cudaSuccess) return e;
  attn_bwd_dq_kernel<<<grid, ABWD_THREADS, DQ_SMEM, s>>>(tmQ, tmDO, tmK, tmV, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  e = cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, KV_SMEM);
  if (e != cudaSuccess) return e;
  attn_bwd_dkdv_kernel<<<grid, ABWD_THREADS, KV_SMEM, s>>>(tmQ, tmDO, tmK, tmV, p);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*launches;
  return e;
}

}  // namespace ikbo
