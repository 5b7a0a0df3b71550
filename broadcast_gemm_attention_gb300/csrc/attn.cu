// attn.cu -- broadcast FlashAttention for sm_103a.
//
// O[i,h] = softmax(Q[i,h] K[map[i],h]^T * scale) V[map[i],h]
//
// IKBO attention (aixai.ru, "Deep Dive: Flash Attention"): candidates that
// share a user share that user's K/V, so a kernel that keeps a user's K/V
// tiles on chip and runs all of the user's candidates' queries against them
// turns the operator from IO-bound into compute-bound.  The pages reorder the
// launch grid (candidate index before heads) so that CTAs of one user run at
// the same time; here the grouping is explicit: a work unit is one (user,
// head) and up to floor(128 / Lq) of that user's candidates (from the segment
// builder's perm), i.e. one 128-row query tile that reads every K/V tile of
// the user's head once from shared memory.  Units of the same (user, head)
// are adjacent in the work list, so neighbouring CTAs stream the same K/V
// through L2.
//
// Per CTA (persistent, one per SM, 8 warps):
//   warp 0      TMA producer: the unit's Q tile (one box per candidate and
//               d-half, gathered through perm) into one of two landing
//               buffers; K and V tiles of 128 keys through a 5-stage ring
//   warp 1      S issuer and TMEM owner: S = Q K^T into S0 / S1 alternately
//   warp 2      P.V issuer: O += P V
//   warp 3      idle
//   warps 4-7   softmax + epilogue (one thread per query row = TMEM lane)
// TMEM (512 columns): S0 S1 (128 each, fp32), P (64, bf16 pairs), Q (64,
// bf16 pairs), O (128, fp32).  Both products take A from TMEM, so shared
// memory only feeds K, V and the TMA writes.
//
// Why two issuers and a separate P: one thread can issue a tcgen05.mma only
// every ~128 cycles, while an M=128, N=128, K=16 product needs 64 cycles of
// the tensor pipe, so a lone issuer leaves the pipe half idle.  Here S(j+2)
// can be issued as soon as the softmax has read S(j) out of its buffer, and
// P.V(j-1) as soon as P(j-1) is written, so both issuers are busy while the
// softmax of tile j runs and the softmax itself never waits for a product.
//
// Online softmax in fp32 in the log2 domain (exp2 with scale*log2(e) folded
// in); the running max is only moved when it grows by more than 2^8, so O is
// rescaled rarely (the result is the same: O and l share the reference max).
#include <cuda_bf16.h>

#include "ikbo_internal.h"
#include "ptx.cuh"

namespace ikbo {

namespace {

constexpr uint32_t HALF_TILE = ATT_BM * 64 * 2;  // 128 rows x 64 bf16 = 16 KB (Q and K/V tiles alike)
constexpr float RESCALE_THRESHOLD = 8.0f;          // log2 units
constexpr int SOFTMAX_WARP0 = 4;                   // first softmax warp
constexpr uint32_t TM_S = 0;                       // S_b at TM_S + 128 b
constexpr uint32_t TM_P = 256;
constexpr uint32_t TM_Q = 320;
constexpr uint32_t TM_O = 384;

struct AttSmem {
  uint8_t* q;          // ATT_Q_BUFS landing buffers x 32 KB
  uint8_t* kv;         // ATT_STAGES x 32 KB
  uint64_t* q_full;    // [2] landing buffer loaded
  uint64_t* q_empty;   // [2] landing buffer copied into TMEM
  uint64_t* qt_ready;  // Q of the unit is in TMEM
  uint64_t* kv_full;
  uint64_t* kv_empty;
  uint64_t* s_full;    // [2] S_b computed
  uint64_t* s_free;    // [2] S_b read by the softmax
  uint64_t* p_full;    // P written
  uint64_t* pv_done;   // a P.V completed (P is free again, O is up to date)
  uint64_t* o_full;    // the unit's last P.V completed
  uint64_t* o_empty;   // the unit's epilogue has read O
  uint32_t* tmem_slot;
  uint32_t* abort;
};

__device__ __forceinline__ AttSmem carve(uint8_t* base) {
  AttSmem s;
  s.q = base;
  s.kv = base + ATT_Q_BUFS * ATT_Q_TILE_BYTES;
  uint64_t* b = reinterpret_cast<uint64_t*>(s.kv + ATT_STAGES * ATT_KV_STAGE_BYTES);
  s.q_full = b;
  s.q_empty = b + 2;
  s.qt_ready = b + 4;
  s.kv_full = b + 5;
  s.kv_empty = s.kv_full + ATT_STAGES;
  s.s_full = s.kv_empty + ATT_STAGES;
  s.s_free = s.s_full + 2;
  s.p_full = s.s_free + 2;
  s.pv_done = s.p_full + 1;
  s.o_full = s.pv_done + 1;
  s.o_empty = s.o_full + 1;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.o_empty + 1);
  s.abort = s.tmem_slot + 1;
  return s;
}

struct Unit {
  int u, h, start, cnt;
  bool ok;
  int L;       // keys of this user
  int kv0;     // first packed row (jagged) or 0
  int ntiles;  // ceil(L / 128)
};

__device__ __forceinline__ Unit decode(const AttnParams& p, int unit) {
  const int4 w = reinterpret_cast<const int4*>(p.work)[unit];
  Unit x;
  x.u = w.x;
  x.h = w.y;
  x.start = w.z;
  x.cnt = w.w;
  x.ok = x.u >= 0 && x.u < p.n_users && x.h >= 0 && x.h < p.H && x.cnt >= 1 && x.cnt <= p.cands_per_tile &&
         x.start >= 0 && x.start + x.cnt <= p.n_cand;
  if (!x.ok) {
    x.L = 0;
    x.kv0 = 0;
    x.ntiles = 0;
    return x;
  }
  if (p.kv_offsets) {
    x.kv0 = p.kv_offsets[x.u];
    x.L = p.kv_offsets[x.u + 1] - x.kv0;
    if (x.L < 0) x.L = 0;
  } else {
    x.kv0 = 0;
    x.L = p.Lkv;
  }
  x.ntiles = (x.L + ATT_BN - 1) / ATT_BN;
  return x;
}

// position of K/V load c (K of global tile g is load 2g, its V load 2g+1) in the ring
__device__ __forceinline__ int ring_stage(uint32_t c) { return static_cast<int>(c % ATT_STAGES); }
__device__ __forceinline__ uint32_t ring_phase(uint32_t c) { return (c / ATT_STAGES) & 1u; }

// Keeps the compiler from moving uses of r above a preceding tcgen05.wait.
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

__device__ __forceinline__ void tmem_ld32p(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32p(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// ------------------------------------------------------------ producer
__device__ void att_producer(const AttnParams& p, const AttSmem& s, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                             const CUtensorMap* tmV, int n_units) {
  uint32_t c = 0;   // K/V loads issued
  uint32_t qc = 0;  // Q tiles loaded
  const int cpt = p.cands_per_tile;
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit x = decode(p, unit);
    if (!x.ok) {
      atomicOr(p.status, DEV_ERR_BAD_WORK);
      continue;
    }
    if (x.ntiles == 0) continue;
    const int qb = static_cast<int>(qc & 1u);
    if (!mbar_wait(&s.q_empty[qb], ((qc >> 1) & 1u) ^ 1u, s.abort, p.timeout_ns, 1)) return;
    ++qc;
    mbar_arrive_expect_tx(&s.q_full[qb], static_cast<uint32_t>(cpt * p.Lq * ATT_D * 2));
    for (int j = 0; j < cpt; ++j) {
      // empty slots read one past the last candidate: TMA fills them with zeros
      const int cand = j < x.cnt ? p.perm[x.start + j] : p.n_cand;
      uint8_t* dst = s.q + qb * ATT_Q_TILE_BYTES + j * p.Lq * 128;
      tma_load_4d(dst, tmQ, &s.q_full[qb], 0, 0, x.h, cand);
      tma_load_4d(dst + HALF_TILE, tmQ, &s.q_full[qb], 64, 0, x.h, cand);
    }
    for (int jt = 0; jt < x.ntiles; ++jt) {
      for (int kv = 0; kv < 2; ++kv, ++c) {
        const int st = ring_stage(c);
        if (!mbar_wait(&s.kv_empty[st], ring_phase(c) ^ 1u, s.abort, p.timeout_ns, 1)) return;
        mbar_arrive_expect_tx(&s.kv_full[st], ATT_KV_STAGE_BYTES);
        uint8_t* dst = s.kv + st * ATT_KV_STAGE_BYTES;
        const CUtensorMap* tm = kv == 0 ? tmK : tmV;
        if (p.kv_offsets) {
          tma_load_3d(dst, tm, &s.kv_full[st], 0, x.h, x.kv0 + jt * ATT_BN);
          tma_load_3d(dst + HALF_TILE, tm, &s.kv_full[st], 64, x.h, x.kv0 + jt * ATT_BN);
        } else {
          tma_load_4d(dst, tm, &s.kv_full[st], 0, jt * ATT_BN, x.h, x.u);
          tma_load_4d(dst + HALF_TILE, tm, &s.kv_full[st], 64, jt * ATT_BN, x.h, x.u);
        }
      }
    }
  }
}

// ----------------------------------------------------------------- MMA
// Descriptors are built once per tile and advanced by adding (offset >> 4)
// to the start-address field; shared memory is below 256 KB, so the 14-bit
// field never carries into the next one.
//
// S = Q K^T: A = Q (TMEM, 16 d per step = 8 columns), B = K tile (K-major,
// 128 keys x 128 d as two 64-wide d halves; steps 0-3 advance 32 bytes
// inside the swizzled rows of the first half, 4-7 in the second).
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint32_t q_tmem, uint32_t k_base) {
  constexpr uint32_t idesc = idesc_bf16_f32(ATT_BM, ATT_BN, false, false);
  const uint64_t kd = sdesc_sw128(k_base, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = ((ks >> 2) * HALF_TILE + (ks & 3) * 32) >> 4;
    mma_bf16_ts(s_tmem, q_tmem + ks * 8, kd + off, idesc, ks > 0 ? 1u : 0u);
  }
}

// O += P V: A = P (TMEM, 16 keys per step = 8 columns), B = V tile (MN-major:
// d contiguous; 64-wide d halves one HALF_TILE apart, 8 key rows per
// 1024-byte atom).
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_base, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(ATT_BM, ATT_D, false, true);
  const uint64_t vd = sdesc_sw128(v_base, HALF_TILE, 1024);
#pragma unroll
  for (int ks = 0; ks < ATT_BN / 16; ++ks) {
    mma_bf16_ts(o_tmem, p_tmem + ks * 8, vd + ((ks * 2048u) >> 4), idesc, (accumulate || ks > 0) ? 1u : 0u);
  }
}

// S issuer: tile g goes to S_(g&1) once the softmax has read S(g-2) out of it.
__device__ void att_s_issuer(const AttnParams& p, const AttSmem& s, uint32_t tmem, int n_units) {
  uint32_t g = 0, qu = 0;
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit x = decode(p, unit);
    if (x.ntiles == 0) continue;
    if (!mbar_wait(s.qt_ready, qu & 1u, s.abort, p.timeout_ns, 1)) return;
    ++qu;
    for (int jt = 0; jt < x.ntiles; ++jt, ++g) {
      const int b = static_cast<int>(g & 1u);
      const uint32_t n = g >> 1;
      const uint32_t kc = 2 * g;
      if (!mbar_wait(&s.kv_full[ring_stage(kc)], ring_phase(kc), s.abort, p.timeout_ns, 1)) return;
      if (n > 0 && !mbar_wait(&s.s_free[b], (n - 1) & 1u, s.abort, p.timeout_ns, 1)) return;
      tc_fence_after();
      issue_qk(tmem + TM_S + b * 128, tmem + TM_Q, smem_u32(s.kv + ring_stage(kc) * ATT_KV_STAGE_BYTES));
      mma_commit(&s.s_full[b]);
      mma_commit(&s.kv_empty[ring_stage(kc)]);
    }
  }
}

// P.V issuer: tile g once its P is written; the unit's first one also waits
// for the previous unit's epilogue to have read O.
__device__ void att_pv_issuer(const AttnParams& p, const AttSmem& s, uint32_t tmem, int n_units) {
  uint32_t g = 0, ou = 0;
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit x = decode(p, unit);
    if (x.ntiles == 0) continue;
    for (int jt = 0; jt < x.ntiles; ++jt, ++g) {
      const uint32_t vc = 2 * g + 1;
      if (!mbar_wait(s.p_full, g & 1u, s.abort, p.timeout_ns, 1)) return;
      if (!mbar_wait(&s.kv_full[ring_stage(vc)], ring_phase(vc), s.abort, p.timeout_ns, 1)) return;
      if (jt == 0 && !mbar_wait(s.o_empty, (ou & 1u) ^ 1u, s.abort, p.timeout_ns, 1)) return;
      tc_fence_after();
      issue_pv(tmem + TM_O, tmem + TM_P, smem_u32(s.kv + ring_stage(vc) * ATT_KV_STAGE_BYTES), jt > 0);
      mma_commit(s.pv_done);
      mma_commit(&s.kv_empty[ring_stage(vc)]);
      if (jt + 1 == x.ntiles) {
        mma_commit(s.o_full);
        ++ou;
      }
    }
  }
}

// ---------------------------------------------------- softmax + epilogue
struct RowOut {
  bool pending;  // a finished unit whose O has not been written yet
  bool valid;    // this thread's row belongs to a candidate of that unit
  __nv_bfloat16* row;
  float l;
};

// O / l -> bf16 -> the row of O in global memory; then O may be overwritten.
__device__ __forceinline__ bool att_epilogue(const AttnParams& p, const AttSmem& s, uint32_t Ot, const RowOut& ro,
                                             uint32_t& ou) {
  if (!mbar_wait(s.o_full, ou & 1u, s.abort, p.timeout_ns, 1)) return false;
  ++ou;
  tc_fence_after();
  const float inv = ro.l > 0.f ? 1.0f / ro.l : 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t o[32];
    tmem_ld32(Ot + c * 32, o);
    tmem_ld_wait(o);
    if (ro.valid) {
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        pk[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
      uint4* dst = reinterpret_cast<uint4*>(ro.row + c * 32);
#pragma unroll
      for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
    }
  }
  tc_fence_before();
  mbar_arrive(s.o_empty);
  return true;
}

__device__ void att_softmax(const AttnParams& p, const AttSmem& s, uint32_t tmem, int n_units) {
  const int warp = threadIdx.x >> 5;
  const int quarter = warp & 3;                                    // TMEM lane quarter of this warp
  const int r = (quarter << 5) + static_cast<int>(lane_id());     // row = TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t Pt = tmem + lane_base + TM_P;
  const uint32_t Qt = tmem + lane_base + TM_Q;
  const uint32_t Ot = tmem + lane_base + TM_O;
  const float sl = p.scale_log2;
  uint32_t g = 0, qc = 0, ou = 0;
  RowOut prev = {false, false, nullptr, 0.f};

  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit x = decode(p, unit);
    const int slot = r / p.Lq;
    const int q = r % p.Lq;
    const bool row_valid = x.ok && r < p.cands_per_tile * p.Lq && slot < x.cnt;
    __nv_bfloat16* orow = nullptr;
    if (row_valid) {
      const int cand = p.perm[x.start + slot];
      orow = reinterpret_cast<__nv_bfloat16*>(p.O) + ((static_cast<size_t>(cand) * p.H + x.h) * p.Lq + q) * ATT_D;
    }
    if (x.ntiles == 0) {  // empty key range: O = 0
      if (row_valid) {
        uint4 z = make_uint4(0, 0, 0, 0);
        for (int c = 0; c < ATT_D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
      }
      continue;
    }
    // Q row: landing buffer (128-byte swizzle: 16-byte chunk c of row r sits
    // at chunk c ^ (r % 8)) -> TMEM columns of Q as bf16 pairs.  Every S of
    // the previous unit has been read by this thread already, so Q is free.
    const int qb = static_cast<int>(qc & 1u);
    if (!mbar_wait(&s.q_full[qb], (qc >> 1) & 1u, s.abort, p.timeout_ns, 1)) return;
    ++qc;
    const uint8_t* qrow = s.q + qb * ATT_Q_TILE_BYTES + r * 128;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t w[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(qrow + half * HALF_TILE + ((c ^ (r & 7)) << 4));
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
      }
      tmem_st32(Qt + half * 32, w);
    }
    tmem_st_wait();
    tc_fence_before();
    mbar_arrive(s.qt_ready);
    mbar_arrive(&s.q_empty[qb]);
    // the previous unit's O is written out while this unit's first S are computed
    if (prev.pending) {
      if (!att_epilogue(p, s, Ot, prev, ou)) return;
      prev.pending = false;
    }

    float m = -INFINITY, l = 0.f;
    for (int jt = 0; jt < x.ntiles; ++jt, ++g) {
      const int b = static_cast<int>(g & 1u);
      const uint32_t S = tmem + lane_base + TM_S + b * 128;
      if (!mbar_wait(&s.s_full[b], (g >> 1) & 1u, s.abort, p.timeout_ns, 1)) return;
      tc_fence_after();
      const int ncols = min(ATT_BN, x.L - jt * ATT_BN);
      uint32_t v[128];
      tmem_ld32p(S + 0, v);
      tmem_ld32p(S + 32, v + 32);
      tmem_ld32p(S + 64, v + 64);
      tmem_ld32p(S + 96, v + 96);
      tmem_ld_wait();
      reg_fence32(v);
      reg_fence32(v + 32);
      reg_fence32(v + 64);
      reg_fence32(v + 96);
      tc_fence_before();
      mbar_arrive(&s.s_free[b]);  // S_b may take S(g + 2) now
      if (ncols < ATT_BN) {
#pragma unroll
        for (int j = 0; j < ATT_BN; ++j)
          if (j >= ncols) v[j] = __float_as_uint(-INFINITY);
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int j = 0; j < ATT_BN; j += 4) {
        mx0 = fmaxf(mx0, __uint_as_float(v[j]));
        mx1 = fmaxf(mx1, __uint_as_float(v[j + 1]));
        mx2 = fmaxf(mx2, __uint_as_float(v[j + 2]));
        mx3 = fmaxf(mx3, __uint_as_float(v[j + 3]));
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float m_new = fmaxf(m, mx * sl);
      // tcgen05.ld/st are warp-collective: the rescale decision must be
      // uniform across the warp, so any row that needs it moves all 32
      const bool rescale = __any_sync(0xffffffffu, m_new > m + RESCALE_THRESHOLD);
      float alpha = 1.f;
      if (rescale) {
        alpha = ex2(m - m_new);  // 0 on the first tile, 1 for rows whose max did not move
        l *= alpha;
        m = m_new;
      }
      // p = 2^(s*sl - m) (masked columns give 2^-inf = 0) as bf16 pairs
      float l0 = 0.f, l1 = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float p0 = ex2(fmaf(__uint_as_float(v[2 * j]), sl, -m));
        const float p1 = ex2(fmaf(__uint_as_float(v[2 * j + 1]), sl, -m));
        l0 += p0;
        l1 += p1;
        pk[j] = pack_bf16x2(p0, p1);
      }
      l += l0 + l1;
      // P and O are free once the previous P.V has completed
      if (g > 0 && !mbar_wait(s.pv_done, (g - 1) & 1u, s.abort, p.timeout_ns, 1)) return;
      tc_fence_after();
      if (rescale && jt > 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(Ot + c * 32, o);
          tmem_ld_wait(o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
          tmem_st32(Ot + c * 32, o);
        }
      }
      tmem_st32p(Pt, pk);
      tmem_st32p(Pt + 32, pk + 32);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(s.p_full);
    }
    prev.pending = true;
    prev.valid = row_valid;
    prev.row = orow;
    prev.l = l;
  }
  if (prev.pending) att_epilogue(p, s, Ot, prev, ou);
}

__global__ void __launch_bounds__(ATT_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const AttSmem s = carve(base);
  const int warp = threadIdx.x >> 5;
  const int n_units = *p.n_units;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 128);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], 128);
    }
    mbar_init(s.qt_ready, 128);
    mbar_init(s.p_full, 128);
    mbar_init(s.pv_done, 1);
    mbar_init(s.o_full, 1);
    mbar_init(s.o_empty, 128);
    for (int i = 0; i < ATT_STAGES; ++i) {
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 1);
    }
    *s.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmQ);
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
    if (lane_id() == 0) att_producer(p, s, &tmQ, &tmK, &tmV, n_units);
  } else if (warp == 1) {
    if (lane_id() == 0) att_s_issuer(p, s, tmem, n_units);
  } else if (warp == 2) {
    if (lane_id() == 0) att_pv_issuer(p, s, tmem, n_units);
  } else if (warp >= SOFTMAX_WARP0) {
    att_softmax(p, s, tmem, n_units);
  }

  tc_fence_before();
  __syncthreads();
  if (*s.abort && threadIdx.x == 0) atomicOr(p.status, DEV_ERR_PIPE_TIMEOUT);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t attn_smem_bytes() {
  return 1024 + ATT_Q_BUFS * ATT_Q_TILE_BYTES + ATT_STAGES * ATT_KV_STAGE_BYTES + 512;
}

cudaError_t launch_attn(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV, const AttnParams& p,
                        int grid, cudaStream_t s) {
  const size_t smem = attn_smem_bytes();
  cudaError_t e =
      cudaFuncSetAttribute(attn_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  attn_fwd_kernel<<<grid, ATT_THREADS, smem, s>>>(tmQ, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace ikbo
