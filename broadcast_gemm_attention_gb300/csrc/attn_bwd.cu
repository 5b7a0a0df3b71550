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
// A streaming pre-pass, then two persistent kernels, one CTA per SM, 12
// warps: warp 0 TMA (elected lane issues), warps 1-3 tcgen05.mma issuers
// (elected lane; one product chain each, warp 1 also owns TMEM), warps 4-11
// the element-wise work: warps w and w+4 share the 32 TMEM lanes of quarter
// w % 4 and split the 128 columns of every tile in halves.
//   attn_bwd_rows_kernel  D = rowsum(dO * O) of every row of every work unit
//                         (and the forward's LSE in the log2 domain), stored
//                         in tile order for both kernels; its first block
//                         also scans the users' key blocks and query tiles.
//   attn_bwd_dq_kernel    per work-list unit (a 128-row tile of up to
//                         floor(128/Lq) candidates' queries, as the forward):
//                         without the forward's LSE, pass 1 forms it over the
//                         user's key tiles (S double-buffered in TMEM) and
//                         stores it for the next kernel; pass 2 recomputes S,
//                         forms dP and dS (written over S in TMEM) and
//                         accumulates dQ += dS K.
//   attn_bwd_dkdv_kernel  per (user, head, 128-key block), keys on TMEM lanes:
//                         for every query tile of the user's candidates, in
//                         two 64-query halves on alternating TMEM buffers,
//                         S^T = K Q^T, dP^T = V dO^T, then P^T and dS^T are
//                         written over them in TMEM and dV += P^T dO,
//                         dK += dS^T Q accumulate in TMEM -- the sum over a
//                         user's candidates never leaves the chip.
// Products that read a bf16 operand written over an fp32 one in TMEM are
// waited for (commit) before anything writes those columns again; the issue
// order puts that wait behind an independent product, so the tensor pipe
// stays fed.  P and dS are rounded to bf16 for the tensor cores (as P is in
// the forward); every accumulation is fp32.  Every wait is bounded.
#include <cuda_bf16.h>
#include <math.h>

#include "bwd_internal.h"
#include "ptx.cuh"

namespace ikbo {

namespace {

constexpr uint32_t TILE = 128 * 128 * 2;  // a 128-row x 128-d bf16 tile: two 64-d halves
constexpr uint32_t HALF = 128 * 64 * 2;   // 16 KB
constexpr int EW_WARP0 = 4;
constexpr int EW_THREADS = ABWD_THREADS - 32 * EW_WARP0;  // 256

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

// Where the bf16 pairs of a 128-column fp32 TMEM tile, converted in place,
// sit: each column half (64 fp32 columns, one element-wise warp's share)
// keeps its 32 pairs at its own start, so a warp only overwrites columns it
// has already read.  k step ks (16 of the 128 elements) -> column offset.
__device__ __forceinline__ uint32_t inplace_col(int ks) { return static_cast<uint32_t>((ks >> 2) * 64 + (ks & 3) * 8); }

// D (+)= A B with A the bf16 pairs written in place over a 128-column TMEM
// tile (128 rows x 128 k) and B a [k rows][128 d] tile read MN-major (d
// contiguous), 8 steps of 16 k.
__device__ __forceinline__ void mma_inplace_by_tile(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base,
                                                    bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, true);
  const uint64_t bd = sdesc_sw128(b_base, HALF, 1024);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_bf16_ts(d_tmem, a_tmem + inplace_col(ks), bd + ((ks * 2048u) >> 4), idesc,
                (accumulate || ks > 0) ? 1u : 0u);
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

// 32 fp32 values -> 64 bytes of bf16 at dst (16-byte aligned).
__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const uint32_t (&v)[32]) {
  uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    o[k] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * k]), __uint_as_float(v[8 * k + 1])),
                      pack_bf16x2(__uint_as_float(v[8 * k + 2]), __uint_as_float(v[8 * k + 3])),
                      pack_bf16x2(__uint_as_float(v[8 * k + 4]), __uint_as_float(v[8 * k + 5])),
                      pack_bf16x2(__uint_as_float(v[8 * k + 6]), __uint_as_float(v[8 * k + 7])));
}

// Paired fp32 arithmetic (one f32x2 instruction for two lanes of work).
// (r0, r1) = (a0, a1) * (b0, b1) + (c0, c1)
__device__ __forceinline__ void fma2v(float& r0, float& r1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
  asm("{.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "mov.b64 z, {%6, %7};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\t"
      "mov.b64 {%0, %1}, w;}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
// (r0, r1) = (a0, a1) * (b0, b1)
__device__ __forceinline__ void mul2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  asm("{.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 w, x, y;\n\t"
      "mov.b64 {%0, %1}, w;}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// (r0, r1) = (a0, a1) - (b0, b1)
__device__ __forceinline__ void sub2(float& r0, float& r1, float a0, float a1, float b0, float b1) {
  asm("{.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "sub.rn.f32x2 w, x, y;\n\t"
      "mov.b64 {%0, %1}, w;}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// ================================================================ dQ kernel
// TMEM columns: S0 [0,128), S1 [128,256) (dS written over S in pass 2),
// dP [256,384), dQ [384,512).
constexpr uint32_t TQ_S = 0, TQ_DP = 256, TQ_DQ = 384;
constexpr int DQ_K_STAGES = 3, DQ_V_STAGES = 2;

struct DqSmem {
  uint8_t* q;    // 32 KB
  uint8_t* go;   // dO tile, 32 KB
  uint8_t* k;    // DQ_K_STAGES x 32 KB
  uint8_t* v;    // DQ_V_STAGES x 32 KB
  float2* xch;   // [2][128] per column half: the row's running (max, sum) after pass 1
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* do_full;
  uint64_t* do_empty;
  uint64_t* k_full;
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* s_full;    // [2] S computed into buffer b
  uint64_t* s_read;    // [2] pass 1: the element-wise warps have read buffer b
  uint64_t* s_free;    // [2] pass 2: the dQ product reading dS from buffer b completed
  uint64_t* dp_full;   // dP computed
  uint64_t* dp_read;   // dP read by the element-wise warps (the next dP may overwrite it)
  uint64_t* ds_ready;  // dS written
  uint64_t* dq_full;   // the unit's dQ is complete
  uint64_t* dq_free;   // ... and has been read out
  uint64_t* xch_full;  // every element-wise thread posted its (max, sum)
  uint32_t* tmem_slot;
  uint32_t* abort;
};
constexpr uint32_t DQ_TILES = (2 + DQ_K_STAGES + DQ_V_STAGES) * TILE;
constexpr uint32_t DQ_XCH = 2 * 128 * 8;
constexpr uint32_t DQ_BARS = 4 + 2 * DQ_K_STAGES + 2 * DQ_V_STAGES + 6 + 6;
constexpr uint32_t DQ_SMEM_USED = DQ_TILES + DQ_XCH + 8 * DQ_BARS + 8;
constexpr uint32_t DQ_SMEM = DQ_SMEM_USED;  // no alignment slack: the base must be 1024-aligned (checked)

__device__ __forceinline__ DqSmem dq_carve(uint8_t* base) {
  DqSmem s;
  s.q = base;
  s.go = base + TILE;
  s.k = base + 2 * TILE;
  s.v = s.k + DQ_K_STAGES * TILE;
  s.xch = reinterpret_cast<float2*>(base + DQ_TILES);
  uint64_t* b = reinterpret_cast<uint64_t*>(base + DQ_TILES + DQ_XCH);
  s.q_full = b++;
  s.q_empty = b++;
  s.do_full = b++;
  s.do_empty = b++;
  s.k_full = b;
  b += DQ_K_STAGES;
  s.k_empty = b;
  b += DQ_K_STAGES;
  s.v_full = b;
  b += DQ_V_STAGES;
  s.v_empty = b;
  b += DQ_V_STAGES;
  s.s_full = b;
  b += 2;
  s.s_read = b;
  b += 2;
  s.s_free = b;
  b += 2;
  s.dp_full = b++;
  s.dp_read = b++;
  s.ds_ready = b++;
  s.dq_full = b++;
  s.dq_free = b++;
  s.xch_full = b++;
  s.tmem_slot = reinterpret_cast<uint32_t*>(b);
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

// Ring position: slot and the parity of its current use.
struct Ring {
  uint32_t n = 0;
  __device__ __forceinline__ int slot(int stages) const { return static_cast<int>(n % stages); }
  __device__ __forceinline__ uint32_t parity(int stages) const { return (n / stages) & 1u; }
};

__global__ void __launch_bounds__(ABWD_THREADS, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const AttnBwdParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (smem_u32(smem_raw) & 1023u) {  // uniform across the CTA, before any barrier exists
    if (threadIdx.x == 0) atomicOr(p.status, DEV_ERR_SMEM_LAYOUT);
    return;
  }
  const DqSmem s = dq_carve(smem_raw);
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
    mbar_init(s.do_full, 1);
    mbar_init(s.do_empty, 1);
    for (int i = 0; i < DQ_K_STAGES; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < DQ_V_STAGES; ++i) {
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.s_full[b], 1);
      mbar_init(&s.s_read[b], EW_THREADS);
      mbar_init(&s.s_free[b], 1);
    }
    mbar_init(s.dp_full, 1);
    mbar_init(s.dp_read, EW_THREADS);
    mbar_init(s.ds_ready, EW_THREADS);
    mbar_init(s.dq_full, 1);
    mbar_init(s.dq_free, EW_THREADS);
    mbar_init(s.xch_full, EW_THREADS);
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
    // ---- TMA: per unit Q, the K tiles of pass 1, dO, then K and V of pass 2
    uint32_t nq = 0;
    Ring kr, vr;
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
      if (!wwait(s.q_empty, (nq & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
      if (elect_one()) {
        mbar_arrive_expect_tx(s.q_full, static_cast<uint32_t>(rows) * 256u);
        load_qtile(p, &tmQ, s.q, s.q_full, x.h, cand);
      }
      __syncwarp();
      for (int pass = p.lse_in ? 1 : 0; pass < 2; ++pass) {  // pass 1 only without the forward's LSE
        if (pass == 1) {
          if (!wwait(s.do_empty, (nq & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
          if (elect_one()) {
            mbar_arrive_expect_tx(s.do_full, static_cast<uint32_t>(rows) * 256u);
            load_qtile(p, &tmDO, s.go, s.do_full, x.h, cand);
          }
          __syncwarp();
        }
        for (int jt = 0; jt < x.ntiles; ++jt) {
          const int ks = kr.slot(DQ_K_STAGES);
          if (!wwait(&s.k_empty[ks], kr.parity(DQ_K_STAGES) ^ 1u, s.abort, p.timeout_ns)) goto done;
          if (elect_one()) {
            mbar_arrive_expect_tx(&s.k_full[ks], TILE);
            load_kv(p, &tmK, s.k + ks * TILE, &s.k_full[ks], x.u, x.h, x.k.kv0, jt * 128);
          }
          __syncwarp();
          ++kr.n;
          if (pass == 1) {
            const int vs = vr.slot(DQ_V_STAGES);
            if (!wwait(&s.v_empty[vs], vr.parity(DQ_V_STAGES) ^ 1u, s.abort, p.timeout_ns)) goto done;
            if (elect_one()) {
              mbar_arrive_expect_tx(&s.v_full[vs], TILE);
              load_kv(p, &tmV, s.v + vs * TILE, &s.v_full[vs], x.u, x.h, x.k.kv0, jt * 128);
            }
            __syncwarp();
            ++vr.n;
          }
        }
      }
      ++nq;
    }
  } else if (warp >= 1 && warp <= 3) {
    // ---- MMA issuers, one per product so that no thread's issue rate bounds
    // a tile: warp 1 S = Q K^T (and TMEM owner), warp 2 dP = dO V^T, warp 3
    // dQ += dS K.  Pass 2 per tile j: S(j) once its buffer is free (S runs
    // ahead by the two buffers), dP(j) once dP(j-1) has been read, dQ(j) once
    // dS(j) is written.  K(j) stays until dQ(j).  Every role walks the same
    // unit sequence and counts K tiles and S products the same way.
    uint32_t nq = 0, kn = 0, sn = 0, vn = 0, nds = 0, nu = 0;
    // warp 1: per S buffer, the kind of its last use (0 none, 1 pass 1, 2
    // pass 2) and the completions of s_read / s_free waited so far
    uint32_t used0 = 0, used1 = 0, reads0 = 0, reads1 = 0, frees0 = 0, frees1 = 0;
    const uint32_t q_base = smem_u32(s.q), go_base = smem_u32(s.go);
    auto issue_s = [&](int kslot, uint32_t kind, bool last_q) -> bool {
      const int b = static_cast<int>(sn & 1u);
      const uint32_t last = b ? used1 : used0;
      if (last == 1) {
        if (!wwait(&s.s_read[b], (b ? reads1 : reads0) & 1u, s.abort, p.timeout_ns)) return false;
        if (b) ++reads1; else ++reads0;
      } else if (last == 2) {
        if (!wwait(&s.s_free[b], (b ? frees1 : frees0) & 1u, s.abort, p.timeout_ns)) return false;
        if (b) ++frees1; else ++frees0;
      }
      if (b) used1 = kind; else used0 = kind;
      tc_fence_after();
      if (elect_one()) {
        mma_rows_dot(tmem + TQ_S + 128u * b, q_base, smem_u32(s.k + kslot * TILE));
        mma_commit(&s.s_full[b]);
        if (kind == 1) mma_commit(&s.k_empty[kslot]);
        if (last_q) mma_commit(s.q_empty);  // last reader of Q
      }
      __syncwarp();
      ++sn;
      return true;
    };
    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
      const QUnit x = dq_unit(p, unit);
      if (!x.ok || x.ntiles == 0) continue;
      const int n = x.ntiles;
      const int n1 = p.lse_in ? 0 : n;  // pass-1 tiles
      if (warp == 1) {
        if (!wwait(s.q_full, nq & 1u, s.abort, p.timeout_ns)) goto done;
        for (int j = 0; j < n1 + n; ++j) {  // pass 1 (S only), then pass 2
          const int ks = static_cast<int>(kn % DQ_K_STAGES);
          if (!wwait(&s.k_full[ks], (kn / DQ_K_STAGES) & 1u, s.abort, p.timeout_ns)) goto done;
          if (!issue_s(ks, j < n1 ? 1u : 2u, j + 1 == n1 + n)) goto done;
          ++kn;
        }
      } else if (warp == 2) {
        if (!wwait(s.do_full, nq & 1u, s.abort, p.timeout_ns)) goto done;
        for (int j = 0; j < n; ++j) {
          const int vs = static_cast<int>(vn % DQ_V_STAGES);
          if (!wwait(&s.v_full[vs], (vn / DQ_V_STAGES) & 1u, s.abort, p.timeout_ns)) goto done;
          if (vn > 0 && !wwait(s.dp_read, (vn - 1) & 1u, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          if (elect_one()) {
            mma_rows_dot(tmem + TQ_DP, go_base, smem_u32(s.v + vs * TILE));
            mma_commit(s.dp_full);
            mma_commit(&s.v_empty[vs]);
            if (j + 1 == n) mma_commit(s.do_empty);  // last reader of dO
          }
          __syncwarp();
          ++vn;
        }
      } else {
        const uint32_t k0 = kn + n1, s0 = sn + n1;  // this unit's pass-2 K tiles and S products
        for (int j = 0; j < n; ++j) {
          if (!wwait(s.ds_ready, nds & 1u, s.abort, p.timeout_ns)) goto done;
          ++nds;
          if (j == 0 && nu > 0 && !wwait(s.dq_free, (nu - 1) & 1u, s.abort, p.timeout_ns)) goto done;
          const uint32_t b = (s0 + j) & 1u;
          const int ks = static_cast<int>((k0 + j) % DQ_K_STAGES);
          tc_fence_after();
          if (elect_one()) {
            mma_inplace_by_tile(tmem + TQ_DQ, tmem + TQ_S + 128u * b, smem_u32(s.k + ks * TILE), j > 0);
            mma_commit(&s.s_free[b]);
            mma_commit(&s.k_empty[ks]);
            if (j + 1 == n) mma_commit(s.dq_full);
          }
          __syncwarp();
        }
        kn += n1 + n;
        sn += n1 + n;
      }
      ++nq;
      ++nu;
    }
  } else if (warp >= EW_WARP0) {
    // ---- element-wise warps: lane = query row r of the tile; grp picks the
    // half of the tile's 128 key columns (and of dQ's d columns)
    const int ew = warp - EW_WARP0, quarter = ew & 3, grp = ew >> 2;
    const int r = quarter * 32 + static_cast<int>(lane_id());
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t col0 = 64u * grp;
    const float sl = p.scale_log2;
    uint32_t sc = 0, ndp = 0, ndq = 0, nx = 0;
    for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
      const QUnit x = dq_unit(p, unit);
      if (!x.ok) continue;
      const int slot = r / p.Lq, q = r - slot * p.Lq;
      const bool valid = r < rows && slot < x.cnt;
      const int cand = valid ? __ldg(p.perm + x.start + slot) : 0;
      const size_t row = (static_cast<size_t>(cand) * p.H + x.h) * p.Lq + q;
      if (x.ntiles == 0) {  // no keys: dQ = 0; no row of this user reaches the dK/dV kernel
        if (valid) {
          uint4* dq_row = reinterpret_cast<uint4*>(p.dQ + row * 128 + col0);
#pragma unroll
          for (int c = 0; c < 8; ++c) dq_row[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      // the row's D (and the forward's LSE), formed by the pre-pass in tile order
      const float D = p.Drow[static_cast<size_t>(unit) * 128 + r];
      const float lse_tile = p.lse_in ? p.lse[static_cast<size_t>(unit) * 128 + r] : 0.f;
      float lse2;
      if (p.lse_in) {  // the forward's LSE (log2 domain; +inf for rows without a query: P = 0)
        lse2 = lse_tile;
      } else {
        // pass 1: running max and sum over this half's key columns (log2 domain)
        float m = -INFINITY, l = 0.f;
        for (int jt = 0; jt < x.ntiles; ++jt) {
          const uint32_t b = sc & 1u;
          if (!wwait(&s.s_full[b], (sc >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
          ++sc;
          tc_fence_after();
          const int kcol = jt * 128 + static_cast<int>(col0);
          uint32_t v[2][32];
          tmem_ld32(tmem + lane_base + TQ_S + 128u * b + col0, v[0]);
          tmem_ld32(tmem + lane_base + TQ_S + 128u * b + col0 + 32, v[1]);
          tmem_ld_wait(v[0]);
          tmem_ld_wait(v[1]);
          tc_fence_before();
          mbar_arrive(&s.s_read[b]);
          if (kcol + 64 > x.k.L) {  // a partial tile: columns past the keys take no part
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (kcol + c * 32 + j >= x.k.L) v[c][j] = __float_as_uint(-INFINITY);
          }
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(v[c][j]) * sl);
          const float m_new = fmaxf(m, mx);
          if (m_new == -INFINITY) continue;
          float add = 0.f;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j) add += ex2(fmaf(__uint_as_float(v[c][j]), sl, -m_new));
          l = l * ex2(m - m_new) + add;
          m = m_new;
        }
        // combine the two halves' (max, sum): post, then read the partner's
        s.xch[grp * 128 + r] = make_float2(m, l);
        mbar_arrive(s.xch_full);
        if (!wwait(s.xch_full, nx & 1u, s.abort, p.timeout_ns)) goto done;
        ++nx;
        {
          const float2 o = s.xch[(grp ^ 1) * 128 + r];
          const float mm = fmaxf(m, o.x);
          const float ll = (mm == -INFINITY) ? 0.f : l * ex2(m - mm) + o.y * ex2(o.x - mm);
          m = mm;
          l = ll;
        }
        lse2 = l > 0.f ? m + __log2f(l) : INFINITY;
      }
      if (!p.lse_in && grp == 0)  // the unit's 128 tile rows, in tile order, for the dK/dV kernel
        p.lse[static_cast<size_t>(unit) * 128 + r] = valid ? lse2 : INFINITY;
      // pass 2: P = 2^(s sl - lse), dS = P (dP - D) scale written over S.
      for (int jt = 0; jt < x.ntiles; ++jt) {
        const uint32_t b = sc & 1u;
        if (!wwait(&s.s_full[b], (sc >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
        ++sc;
        tc_fence_after();
        const int kcol = jt * 128 + static_cast<int>(col0);
        float pf[64];
        uint32_t dv[2][32];
        {
          uint32_t v[2][32];
          tmem_ld32(tmem + lane_base + TQ_S + 128u * b + col0, v[0]);
          tmem_ld32(tmem + lane_base + TQ_S + 128u * b + col0 + 32, v[1]);
          tmem_ld_wait(v[0]);
          tmem_ld_wait(v[1]);
          // dP first: the single dP buffer is released before P is formed
          if (!wwait(s.dp_full, ndp & 1u, s.abort, p.timeout_ns)) goto done;
          ++ndp;
          tc_fence_after();
          tmem_ld32(tmem + lane_base + TQ_DP + col0, dv[0]);
          tmem_ld32(tmem + lane_base + TQ_DP + col0 + 32, dv[1]);
          tmem_ld_wait(dv[0]);
          tmem_ld_wait(dv[1]);
          tc_fence_before();
          mbar_arrive(s.dp_read);  // the next dP may land
          if (kcol + 64 <= x.k.L) {  // every column of this half is a key (the common case)
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                float t0, t1;
                fma2v(t0, t1, __uint_as_float(v[c][2 * j]), __uint_as_float(v[c][2 * j + 1]), sl, sl, -lse2, -lse2);
                pf[c * 32 + 2 * j] = ex2(t0);
                pf[c * 32 + 2 * j + 1] = ex2(t1);
              }
          } else {
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int j = 0; j < 32; ++j)
                pf[c * 32 + j] =
                    kcol + c * 32 + j < x.k.L ? ex2(fmaf(__uint_as_float(v[c][j]), sl, -lse2)) : 0.f;
          }
        }
        {
          const float sc = p.scale, dsc = -D * p.scale;  // dS = P (dP scale - D scale)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float a0, a1;
              fma2v(a0, a1, __uint_as_float(dv[c][2 * j]), __uint_as_float(dv[c][2 * j + 1]), sc, sc, dsc, dsc);
              mul2(a0, a1, a0, a1, pf[c * 32 + 2 * j], pf[c * 32 + 2 * j + 1]);
              pk[j] = pack_bf16x2(a0, a1);
            }
            tmem_st16(tmem + lane_base + TQ_S + 128u * b + col0 + 16 * c, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(s.ds_ready);
      }
      // epilogue: this half's 64 d columns of dQ (fp32 TMEM) -> bf16
      if (!wwait(s.dq_full, ndq & 1u, s.abort, p.timeout_ns)) goto done;
      ++ndq;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + TQ_DQ + col0 + 32 * c, v);
        tmem_ld_wait(v);
        if (valid) store_bf16x32(p.dQ + row * 128 + col0 + 32 * c, v);
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
// Each 128-query tile is processed as two 64-query halves.  TMEM columns:
// two half-tile buffers X0 [0,128), X1 [128,256), each S^T [X, X+64) and dP^T
// [X+64, X+128) of one half (P^T and dS^T written over them as bf16 pairs),
// then dV [256,384), dK [384,512).  Halves alternate between the buffers, so
// S^T of half g+2 waits for dV of half g instead of dV of the half just
// before it, and the products, the element-wise work and the next halves'
// loads overlap.  Shared memory holds K, V and two query-tile stages.
constexpr uint32_t TK_X = 0, TK_DV = 256, TK_DK = 384;

struct KvSmem {
  uint8_t* k;      // 32 KB, the key block
  uint8_t* v;      // 32 KB
  uint8_t* q;      // 2 x 32 KB query tiles
  uint8_t* go;     // 2 x 32 KB dO tiles
  float* lse;      // [2][128]
  float* drow;     // [2][128]
  uint64_t* kv_full;
  uint64_t* kv_empty;
  uint64_t* q_full;    // [2] per query-tile stage
  uint64_t* q_empty;   // [2]
  uint64_t* s_full;    // [2] per half-tile buffer: S^T computed
  uint64_t* dp_full;   // [2] dP^T computed
  uint64_t* p_ready;   // [2] P^T written (S^T read)
  uint64_t* ds_ready;  // [2] dS^T written (dP^T read)
  uint64_t* xa_free;   // [2] dV has read the buffer's P^T (S^T may land)
  uint64_t* xb_free;   // [2] dK has read the buffer's dS^T (dP^T may land)
  uint64_t* acc_full;  // the block's dV, dK complete
  uint64_t* acc_free;  // ... and read out
  uint32_t* tmem_slot;
  uint32_t* abort;
};
constexpr uint32_t KV_TILES = 6 * TILE;
constexpr uint32_t KV_BARS = 20;
constexpr uint32_t KV_SMEM_USED = KV_TILES + 2 * 2 * 128 * 4 + 8 * KV_BARS + 8;
constexpr uint32_t KV_SMEM = KV_SMEM_USED + 1024;

__device__ __forceinline__ KvSmem kv_carve(uint8_t* base) {
  KvSmem s;
  s.k = base;
  s.v = base + TILE;
  s.q = base + 2 * TILE;
  s.go = base + 4 * TILE;
  s.lse = reinterpret_cast<float*>(base + KV_TILES);
  s.drow = s.lse + 2 * 128;
  uint64_t* b = reinterpret_cast<uint64_t*>(s.drow + 2 * 128);
  s.kv_full = b++;
  s.kv_empty = b++;
  s.q_full = b;
  b += 2;
  s.q_empty = b;
  b += 2;
  s.s_full = b;
  b += 2;
  s.dp_full = b;
  b += 2;
  s.p_ready = b;
  b += 2;
  s.ds_ready = b;
  b += 2;
  s.xa_free = b;
  b += 2;
  s.xb_free = b;
  b += 2;
  s.acc_full = b++;
  s.acc_free = b++;
  s.tmem_slot = reinterpret_cast<uint32_t*>(b);
  s.abort = s.tmem_slot + 1;
  return s;
}

// S^T or dP^T of one half: D[128 keys][64 queries] = A B^T over d = 128, A a
// [128 keys][d] tile, B rows [q0, q0 + 64) of a [128 queries][d] tile (both
// K-major), 8 steps of 16 d.
__device__ __forceinline__ void mma_half_rows_dot(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, int q0) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
  const uint64_t ad = sdesc_sw128(a_base, 16, 1024);
  const uint64_t bd = sdesc_sw128(b_base + static_cast<uint32_t>(q0) * 128u, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = ((ks >> 2) * HALF + (ks & 3) * 32) >> 4;
    mma_bf16_ss(d_tmem, ad + off, bd + off, idesc, ks > 0 ? 1u : 0u);
  }
}

// Where half-tile element pairs sit after the in-place conversion: each of
// the two element-wise warp groups keeps its 16 pairs (32 queries) at the
// start of its own 32 fp32 columns.  k step ks (16 queries) -> column offset.
__device__ __forceinline__ uint32_t half_col(int ks) { return static_cast<uint32_t>((ks >> 1) * 32 + (ks & 1) * 8); }

// D (+)= A B with A the bf16 pairs of one half written in place (128 keys x
// 64 queries) and B rows [q0, q0 + 64) of a [128 queries][128 d] tile read
// MN-major, 4 steps of 16 queries.
__device__ __forceinline__ void mma_half_by_tile(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, int q0,
                                                 bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, true);
  const uint64_t bd = sdesc_sw128(b_base + static_cast<uint32_t>(q0) * 128u, HALF, 1024);
#pragma unroll
  for (int ks = 0; ks < 4; ++ks)
    mma_bf16_ts(d_tmem, a_tmem + half_col(ks), bd + ((ks * 2048u) >> 4), idesc, (accumulate || ks > 0) ? 1u : 0u);
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
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  if (pad + KV_SMEM_USED > KV_SMEM) {  // uniform across the CTA, before any barrier exists
    if (threadIdx.x == 0) atomicOr(p.status, DEV_ERR_SMEM_LAYOUT);
    return;
  }
  const KvSmem s = kv_carve(smem_raw + pad);
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
    mbar_init(s.kv_empty, 2);  // the S^T and dP^T issuers
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s.q_full[b], 1);
      mbar_init(&s.q_empty[b], 1);
      mbar_init(&s.s_full[b], 1);
      mbar_init(&s.dp_full[b], 1);
      mbar_init(&s.p_ready[b], EW_THREADS);
      mbar_init(&s.ds_ready[b], EW_THREADS);
      mbar_init(&s.xa_free[b], 1);
      mbar_init(&s.xb_free[b], 1);
    }
    mbar_init(s.acc_full, 1);
    mbar_init(s.acc_free, EW_THREADS);
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
    // the rows' LSE and D (two bulk copies)
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
      // the user's query tiles are work units ubase .. ubase + ntq - 1 of the
      // work list (user-major, then head, then chunk): the dQ kernel left
      // their rows' LSE and D there, 128 per unit, in tile order
      const size_t ubase =
          static_cast<size_t>(p.H) * __ldg(p.tile_prefix + x.u) + static_cast<size_t>(x.h) * x.ntq;
      const int lane = static_cast<int>(lane_id());
      // lane j < n holds the tile's j-th candidate, loaded one tile ahead
      int mine = lane < min(cpt, x.count) ? __ldg(p.perm + x.seg0 + lane) : p.n_cand;
      for (int t = 0; t < x.ntq; ++t, ++tq) {
        const int b = static_cast<int>(tq & 1u);
        int cand[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) cand[j] = __shfl_sync(0xffffffffu, mine, j);
        if (!wwait(&s.q_empty[b], ((tq >> 1) & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
        if (elect_one()) {
          mbar_arrive_expect_tx(&s.q_full[b], 2u * static_cast<uint32_t>(rows) * 256u + 2u * 512u);
          load_qtile(p, &tmQ, s.q + b * TILE, &s.q_full[b], x.h, cand);
          load_qtile(p, &tmDO, s.go + b * TILE, &s.q_full[b], x.h, cand);
          bulk_load(s.lse + b * 128, p.lse + (ubase + t) * 128, 512u, &s.q_full[b]);
          bulk_load(s.drow + b * 128, p.Drow + (ubase + t) * 128, 512u, &s.q_full[b]);
        }
        __syncwarp();
        const int nf = (t + 1) * cpt, nn = min(cpt, x.count - nf);
        mine = (t + 1 < x.ntq && lane < nn) ? __ldg(p.perm + x.seg0 + nf + lane) : p.n_cand;
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ---- S^T (warp 1) and dP^T (warp 2) issuers: half g into buffer
    // X_{g&1} once dV (dK) of half g-2 has read that buffer's P^T (dS^T)
    const bool s_side = warp == 1;
    uint32_t ni = 0, tq = 0, g = 0;
    const uint32_t a_base = smem_u32(s_side ? s.k : s.v);
    uint64_t* full = s_side ? s.s_full : s.dp_full;
    uint64_t* xfree = s_side ? s.xa_free : s.xb_free;
    const uint32_t col = s_side ? 0u : 64u;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const KvItem x = kv_item(p, item);
      if (x.ntq == 0) continue;
      if (!wwait(s.kv_full, ni & 1u, s.abort, p.timeout_ns)) goto done;
      for (int t = 0; t < x.ntq; ++t, ++tq) {
        const int b = static_cast<int>(tq & 1u);
        const uint32_t b_base = smem_u32((s_side ? s.q : s.go) + b * TILE);
        if (!wwait(&s.q_full[b], (tq >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
        for (int h = 0; h < 2; ++h, ++g) {
          const int xb = static_cast<int>(g & 1u);
          if (g >= 2 && !wwait(&xfree[xb], ((g >> 1) - 1) & 1u, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          if (elect_one()) {  // S^T = K Q_h^T  or  dP^T = V dO_h^T
            mma_half_rows_dot(tmem + TK_X + 128u * xb + col, a_base, b_base, 64 * h);
            mma_commit(&full[xb]);
            if (t + 1 == x.ntq && h == 1) mma_commit(s.kv_empty);  // last reader of K (V)
          }
          __syncwarp();
        }
      }
      ++ni;
    }
  } else if (warp == 3) {
    // ---- dV / dK issuer: dV += P^T dO_h once P^T of half g is written,
    // dK += dS^T Q_h once its dS^T is
    uint32_t ni = 0, tq = 0, g = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const KvItem x = kv_item(p, item);
      if (x.ntq == 0) continue;
      for (int t = 0; t < x.ntq; ++t, ++tq) {
        const int b = static_cast<int>(tq & 1u);
        const uint32_t q_base = smem_u32(s.q + b * TILE), go_base = smem_u32(s.go + b * TILE);
        if (!wwait(&s.q_full[b], (tq >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
        for (int h = 0; h < 2; ++h, ++g) {
          const int xb = static_cast<int>(g & 1u);
          const uint32_t k = g >> 1;
          const bool first = t == 0 && h == 0;
          if (!wwait(&s.p_ready[xb], k & 1u, s.abort, p.timeout_ns)) goto done;
          if (first && ni > 0 && !wwait(s.acc_free, (ni - 1) & 1u, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          if (elect_one()) {
            mma_half_by_tile(tmem + TK_DV, tmem + TK_X + 128u * xb, go_base, 64 * h, !first);
            mma_commit(&s.xa_free[xb]);
          }
          __syncwarp();
          if (!wwait(&s.ds_ready[xb], k & 1u, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          if (elect_one()) {
            mma_half_by_tile(tmem + TK_DK, tmem + TK_X + 128u * xb + 64u, q_base, 64 * h, !first);
            mma_commit(&s.xb_free[xb]);
            if (h == 1) mma_commit(&s.q_empty[b]);  // last readers of the query tile
            if (t + 1 == x.ntq && h == 1) mma_commit(s.acc_full);
          }
          __syncwarp();
        }
      }
      ++ni;
    }
  } else if (warp >= EW_WARP0) {
    // ---- element-wise warps: lane = key row of the block; grp picks 32 of
    // each half's 64 query columns (and half of dK/dV's d columns)
    const int ew = warp - EW_WARP0, quarter = ew & 3, grp = ew >> 2;
    const int rk = quarter * 32 + static_cast<int>(lane_id());
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t col0 = 64u * grp;   // dK/dV columns in the epilogue
    const uint32_t qc = 32u * grp;     // query columns within a half
    const float sl = p.scale_log2;
    uint32_t tq = 0, ni = 0, g = 0;
    for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
      const KvItem x = kv_item(p, item);
      const int key = x.kb * 128 + rk;
      const bool kvalid = key < x.k.L;
      const size_t krow = p.kv_offsets ? (static_cast<size_t>(x.k.kv0 + key) * p.H + x.h)
                                       : ((static_cast<size_t>(x.u) * p.H + x.h) * p.Lkv + key);
      uint16_t* dk_row = p.dK + krow * 128 + col0;
      uint16_t* dv_row = p.dV + krow * 128 + col0;
      if (x.ntq == 0) {  // no candidate reads these keys: zero gradients
        if (kvalid) {
#pragma unroll
          for (int c = 0; c < 8; ++c)
            reinterpret_cast<uint4*>(dk_row)[c] = reinterpret_cast<uint4*>(dv_row)[c] = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      // every row of the warp a key (all but a user's last, partial block):
      // no per-element select
      const bool all_keys = __all_sync(0xffffffffu, kvalid);
      for (int t = 0; t < x.ntq; ++t, ++tq) {
        const int b = static_cast<int>(tq & 1u);
        // q_full[b] also covers this tile's LSE and D (bulk copies)
        if (!wwait(&s.q_full[b], (tq >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
        for (int h = 0; h < 2; ++h, ++g) {
          const int xb = static_cast<int>(g & 1u);
          const uint32_t k = g >> 1;
          const uint32_t X = TK_X + 128u * xb;
          const float* lse = s.lse + b * 128 + 64 * h + qc;
          const float* drow = s.drow + b * 128 + 64 * h + qc;
          // P^T = 2^(s sl - lse[q]), written over S^T (pairs at this group's start)
          if (!wwait(&s.s_full[xb], k & 1u, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          float pf[32];
          {
            uint32_t v[32], pk[16];
            tmem_ld32(tmem + lane_base + X + qc, v);
            tmem_ld_wait(v);
#pragma unroll
            for (int j4 = 0; j4 < 8; ++j4) {
              const float4 l4 = *reinterpret_cast<const float4*>(lse + 4 * j4);
              float t[4];
              fma2v(t[0], t[1], __uint_as_float(v[4 * j4]), __uint_as_float(v[4 * j4 + 1]), sl, sl, -l4.x, -l4.y);
              fma2v(t[2], t[3], __uint_as_float(v[4 * j4 + 2]), __uint_as_float(v[4 * j4 + 3]), sl, sl, -l4.z, -l4.w);
#pragma unroll
              for (int e = 0; e < 4; ++e) pf[4 * j4 + e] = ex2(t[e]);
            }
            if (!all_keys && !kvalid) {
#pragma unroll
              for (int j = 0; j < 32; ++j) pf[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) pk[j] = pack_bf16x2(pf[2 * j], pf[2 * j + 1]);
            tmem_st16(tmem + lane_base + X + qc, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&s.p_ready[xb]);
          // dS^T = P^T (dP^T - D[q]) scale, written over dP^T
          if (!wwait(&s.dp_full[xb], k & 1u, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          {
            uint32_t v[32], pk[16];
            tmem_ld32(tmem + lane_base + X + 64u + qc, v);
            tmem_ld_wait(v);
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const float4 d4 = *reinterpret_cast<const float4*>(drow + 8 * j4);
              const float4 e4 = *reinterpret_cast<const float4*>(drow + 8 * j4 + 4);
              const float dv8[8] = {d4.x, d4.y, d4.z, d4.w, e4.x, e4.y, e4.z, e4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {  // dS = (P scale) (dP - D)
                const int j = 8 * j4 + 2 * e;
                float a0, a1, s0, s1;
                sub2(a0, a1, __uint_as_float(v[j]), __uint_as_float(v[j + 1]), dv8[2 * e], dv8[2 * e + 1]);
                mul2(s0, s1, pf[j], pf[j + 1], p.scale, p.scale);
                mul2(a0, a1, a0, a1, s0, s1);
                pk[4 * j4 + e] = pack_bf16x2(a0, a1);
              }
            }
            tmem_st16(tmem + lane_base + X + 64u + qc, pk);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&s.ds_ready[xb]);
        }
      }
      // epilogue: this half's 64 d columns of the block's dV and dK rows
      if (!wwait(s.acc_full, ni & 1u, s.abort, p.timeout_ns)) goto done;
      ++ni;
      tc_fence_after();
#pragma unroll 1
      for (int a = 0; a < 2; ++a) {  // dV, then dK
        uint16_t* out = a == 0 ? dv_row : dk_row;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + (a == 0 ? TK_DV : TK_DK) + col0 + 32 * c, v);
          tmem_ld_wait(v);
          if (kvalid) store_bf16x32(out + 32 * c, v);
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

// blk_prefix[u] = sum over users v < u of ceil(L_v / 128) (key blocks) and
// tile_prefix[u] = sum over v < u of ceil(count_v / cpt) (query tiles); one
// CTA, a scan over chunks of users.
__device__ __forceinline__ int user_blocks(const int32_t* kv_offsets, int Lkv, int u) {
  const int L = kv_offsets ? max(0, kv_offsets[u + 1] - kv_offsets[u]) : Lkv;
  return (L + 127) / 128;
}
__device__ __forceinline__ int user_tiles(const int32_t* offsets, int cpt, int u) {
  return (max(0, offsets[u + 1] - offsets[u]) + cpt - 1) / cpt;
}

// Prefix sums over the users of their key blocks and query tiles (for the
// dK/dV kernel's work numbering), by one block of ROWS_THREADS threads.
constexpr int ROWS_THREADS = 256;
__device__ void user_prefixes(const AttnBwdParams& p) {
  __shared__ int32_t part[2][ROWS_THREADS];
  const int per = (p.n_users + ROWS_THREADS - 1) / ROWS_THREADS;
  const int u0 = static_cast<int>(threadIdx.x) * per;
  int32_t sb = 0, st = 0;
  for (int u = u0; u < min(u0 + per, p.n_users); ++u) {
    sb += user_blocks(p.kv_offsets, p.Lkv, u);
    st += user_tiles(p.offsets, p.cands_per_tile, u);
  }
  part[0][threadIdx.x] = sb;
  part[1][threadIdx.x] = st;
  __syncthreads();
  for (int w = 1; w < ROWS_THREADS; w <<= 1) {  // inclusive scans of the chunk sums
    const int32_t vb = static_cast<int>(threadIdx.x) >= w ? part[0][threadIdx.x - w] : 0;
    const int32_t vt = static_cast<int>(threadIdx.x) >= w ? part[1][threadIdx.x - w] : 0;
    __syncthreads();
    part[0][threadIdx.x] += vb;
    part[1][threadIdx.x] += vt;
    __syncthreads();
  }
  int32_t rb = threadIdx.x > 0 ? part[0][threadIdx.x - 1] : 0;
  int32_t rt = threadIdx.x > 0 ? part[1][threadIdx.x - 1] : 0;
  int32_t* blk_prefix = const_cast<int32_t*>(p.blk_prefix);
  int32_t* tile_prefix = const_cast<int32_t*>(p.tile_prefix);
  for (int u = u0; u < min(u0 + per, p.n_users); ++u) {
    blk_prefix[u] = rb;
    tile_prefix[u] = rt;
    rb += user_blocks(p.kv_offsets, p.Lkv, u);
    rt += user_tiles(p.offsets, p.cands_per_tile, u);
  }
  if (threadIdx.x == ROWS_THREADS - 1) {
    blk_prefix[p.n_users] = part[0][ROWS_THREADS - 1];
    tile_prefix[p.n_users] = part[1][ROWS_THREADS - 1];
  }
}

// Row statistics in tile order: for tile row r of work unit w (candidate
// perm[start + r / Lq], query r % Lq), Drow[w][r] = sum_d dO[row][d] O[row][d]
// and, given the forward's natural-log LSE, lse[w][r] = LSE[row] log2(e);
// rows without a query get D = 0 and lse = +inf.  Half a warp per row, 16
// bytes of O and of dO per lane; blocks stride over the units' rows.  Block 0
// computes the user prefixes instead.
__global__ void __launch_bounds__(ROWS_THREADS) attn_bwd_rows_kernel(const AttnBwdParams p) {
  if (blockIdx.x == 0) {
    user_prefixes(p);
    return;
  }
  const int n_units = *p.n_units;
  const int rows = p.cands_per_tile * p.Lq;
  const int sub = static_cast<int>(threadIdx.x & 15u);                               // lane within the row
  const long long nrows = static_cast<long long>(n_units) * 128;
  const long long stride = static_cast<long long>(gridDim.x - 1) * (ROWS_THREADS / 16);
  // ROWS_PER rows per half-warp at a time: their work entries, candidates
  // and O / dO loads are independent, so all of them are in flight at once
  constexpr int ROWS_PER = 4;
  for (long long t0 = static_cast<long long>(blockIdx.x - 1) * (ROWS_THREADS / 16) + (threadIdx.x >> 4); t0 < nrows;
       t0 += ROWS_PER * stride) {
    bool valid[ROWS_PER];
    size_t row[ROWS_PER];
#pragma unroll
    for (int k = 0; k < ROWS_PER; ++k) {
      const long long t = t0 + k * stride;
      valid[k] = false;
      row[k] = 0;
      if (t < nrows) {
        const int unit = static_cast<int>(t >> 7), r = static_cast<int>(t & 127);
        const int4 w = __ldg(reinterpret_cast<const int4*>(p.work) + unit);
        const int slot = r / p.Lq, q = r - slot * p.Lq;
        valid[k] = r < rows && slot < w.w && w.x >= 0 && w.x < p.n_users && w.y >= 0 && w.y < p.H && w.z >= 0 &&
                   w.z + w.w <= p.n_cand;
        if (valid[k]) {
          const int cand = __ldg(p.perm + w.z + slot);
          row[k] = (static_cast<size_t>(cand) * p.H + w.y) * p.Lq + q;
        }
      }
    }
    uint4 a[ROWS_PER], g[ROWS_PER];
    float lse[ROWS_PER];
#pragma unroll
    for (int k = 0; k < ROWS_PER; ++k) {
      a[k] = g[k] = make_uint4(0, 0, 0, 0);
      lse[k] = INFINITY;
      if (valid[k]) {
        a[k] = __ldcs(reinterpret_cast<const uint4*>(p.O + row[k] * 128) + sub);
        g[k] = __ldcs(reinterpret_cast<const uint4*>(p.dO + row[k] * 128) + sub);
        if (p.lse_in) lse[k] = __ldg(p.lse_in + row[k]) * 1.4426950408889634f;
      }
    }
#pragma unroll
    for (int k = 0; k < ROWS_PER; ++k) {
      const uint32_t aw[4] = {a[k].x, a[k].y, a[k].z, a[k].w}, gw[4] = {g[k].x, g[k].y, g[k].z, g[k].w};
      float D = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        D = fmaf(__uint_as_float(aw[e] << 16), __uint_as_float(gw[e] << 16), D);
        D = fmaf(__uint_as_float(aw[e] & 0xffff0000u), __uint_as_float(gw[e] & 0xffff0000u), D);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) D += __shfl_xor_sync(0xffffffffu, D, o);  // within the 16 lanes of the row
      const long long t = t0 + k * stride;
      if (sub == 0 && t < nrows) {
        p.Drow[t] = valid[k] ? D : 0.f;
        if (p.lse_in) p.lse[t] = lse[k];
      }
    }
  }
}

}  // namespace

// ------------------------------------------------------------------- host
size_t attn_bwd_smem_bytes() { return DQ_SMEM > KV_SMEM ? DQ_SMEM : KV_SMEM; }

cudaError_t launch_attn_backward(const CUtensorMap& tmQ, const CUtensorMap& tmDO, const CUtensorMap& tmK,
                                 const CUtensorMap& tmV, const AttnBwdParams& p, int grid, cudaStream_t s,
                                 int* launches) {
  *launches = 0;
  attn_bwd_rows_kernel<<<1 + 8 * grid, ROWS_THREADS, 0, s>>>(p);
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
