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
// Per CTA (persistent, one per SM, 12 warps):
//   warp 0      TMA producer for Q and K: the unit's Q tile (one box per
//               candidate and d-half, gathered through perm) into the Q
//               landing buffer; K tiles of 128 keys through a 3-stage ring
//   warp 1      S issuer and TMEM owner: S = Q K^T into S0 / S1 alternately
//   warp 2      P.V issuer: O += P V
//   warp 3      TMA producer for V (2-stage ring).  K and V have rings and
//               producers of their own so that a K load never queues
//               behind a V load that waits for a P.V several tiles back.
//   warps 4-11  softmax + epilogue, as two groups that ping-pong over the
//               key tiles: group 0 (warps 4-7) takes the even tiles of the
//               CTA's sequence (buffer S0), group 1 (warps 8-11) the odd
//               ones (S1).  A warp owns the 32 TMEM lanes (query rows) of
//               quarter w % 4 and all 128 columns of its tiles, so while one
//               group waits on its tile's loads and handshakes the other
//               group's exponentials keep the SFU busy on the same
//               scheduler.  Both groups accumulate into one O: the row's
//               reference maximum is a chain through the tiles, each tile's
//               group reading the one before from the other group (one
//               release / acquire word per row in shared memory).
// TMEM (512 columns): S0 S1 (128 each, fp32), P0 P1 (64 each, bf16 pairs),
// O (128, fp32).  Q stays in shared memory for all of a unit's S products
// (two Q tiles: the next unit's lands while this one's are read), so S(j+2)
// may be issued as soon as the softmax has read S(j), and P(j) only waits
// for P.V(j-2) to have read P_b.  A unit's O leaves through shared memory,
// in the finished unit's Q tile: a thread owns a query row, so its direct
// stores would scatter 32 rows per warp instruction; each warp writes its 32
// rows x 64 d into its own 4 KB of the staging tile and reads them back 4
// rows per instruction, 8 lanes per contiguous 128-byte half row.
//
// Why two issuers: one thread issues a tcgen05.mma only every ~80-130
// cycles, while an M=128, N=128, K=16 product needs 64 cycles of the tensor
// pipe, so one chain of products leaves the pipe partly idle.  S(j+2) is
// issued as soon as the softmax has read S(j), and P.V(j) once P(j) is
// written, so the two chains overlap each other and both softmax groups.
//
// Online softmax in fp32 in the log2 domain (exp2 with scale*log2(e) folded
// in); the running reference maximum is only moved when a tile's maximum
// exceeds it by more than 2^8, so O is rescaled rarely (the result is the
// same: O and l share the reference).  Each group keeps l over its own
// tiles; the two are brought to the last reference and added at the end.
#include <cuda_bf16.h>

#include "ikbo_internal.h"
#include "ptx.cuh"

namespace ikbo {

namespace {

constexpr uint32_t HALF_TILE = ATT_BM * 64 * 2;  // 128 rows x 64 bf16 = 16 KB (Q and K/V tiles alike)
constexpr float RESCALE_THRESHOLD = 8.0f;          // log2 units
constexpr int SOFTMAX_WARP0 = 4;                   // first softmax warp
constexpr int SOFTMAX_THREADS = ATT_THREADS - 32 * SOFTMAX_WARP0;
constexpr int GROUP_THREADS = SOFTMAX_THREADS / 2;  // one softmax group (4 warps)
constexpr int CTRL_REGS = 72;                       // per thread, warps 0-3 (after setmaxnreg)
constexpr int SOFTMAX_REGS = 216;                   // per thread, warps 4-11
static_assert(32 * SOFTMAX_WARP0 * CTRL_REGS + SOFTMAX_THREADS * SOFTMAX_REGS <= ATT_THREADS * 168,
              "register split exceeds the launch's registers");
constexpr uint32_t TM_S = 0;                       // S_b at TM_S + 128 b
constexpr uint32_t TM_P = 256;                     // P_b at TM_P + 64 b
constexpr uint32_t TM_O = 384;

// dynamic shared memory: [Q tiles][K ring][V ring] (1024-aligned for the
// 128-byte swizzle), then the barriers, two words, the row exchange and the
// reference chain
constexpr uint32_t TILE_REGION = ATT_Q_BUFS * ATT_Q_TILE_BYTES + (ATT_K_STAGES + ATT_V_STAGES) * ATT_KV_STAGE_BYTES;
constexpr int NUM_BARS = 14 + 2 * (ATT_K_STAGES + ATT_V_STAGES) + 8;
constexpr uint32_t XVAL_OFFSET = NUM_BARS * 8 + 8;
constexpr uint32_t CHAIN_OFFSET = XVAL_OFFSET + 2 * 2 * ATT_BM * 4;
constexpr uint32_t AUX_BYTES = CHAIN_OFFSET + ATT_BM * 4;
constexpr uint32_t SMEM_USED = TILE_REGION + AUX_BYTES;
constexpr uint32_t SMEM_ALLOC = 227 * 1024;
static_assert(SMEM_USED <= SMEM_ALLOC, "attention tiles do not fit in shared memory");

struct AttSmem {
  uint8_t* q;          // ATT_Q_BUFS x 32 KB: Q tiles (and the O staging of a finished unit)
  uint8_t* k;          // ATT_K_STAGES x 32 KB
  uint8_t* v;          // ATT_V_STAGES x 32 KB
  uint64_t* q_full;    // [2] Q tile landed
  uint64_t* q_empty;   // [2] the tile's unit: last S done and its O staged out
  uint64_t* s_full;    // [2] S_b computed
  uint64_t* s_free;    // [2] S_b read by group b
  uint64_t* p_full;    // [2] P_b written by group b
  uint64_t* pv_done;   // [2] the P.V of a buffer-b tile completed (P_b is free again, O is up to date)
  uint64_t* o_full;    // the unit's last P.V completed
  uint64_t* o_empty;   // the unit's epilogue has read O
  uint64_t* k_full;
  uint64_t* k_empty;
  uint64_t* v_full;
  uint64_t* v_empty;
  uint64_t* xbar;      // [4 quarters][2] row exchange between the two warps of a quarter
  uint32_t* tmem_slot;
  uint32_t* abort;
  float* xval;         // [2 buffers][2 halves][128 rows]
  uint32_t* chain;     // [128 rows] reference maximum of the last tile (high 24 bits) | its tag (low 8)
};

__device__ __forceinline__ AttSmem carve(uint8_t* base) {
  AttSmem s;
  s.q = base;
  s.k = base + ATT_Q_BUFS * ATT_Q_TILE_BYTES;
  s.v = s.k + ATT_K_STAGES * ATT_KV_STAGE_BYTES;
  uint64_t* b = reinterpret_cast<uint64_t*>(base + TILE_REGION);
  s.q_full = b;
  s.q_empty = b + 2;
  s.s_full = b + 4;
  s.s_free = b + 6;
  s.p_full = b + 8;
  s.pv_done = b + 10;
  s.o_full = b + 12;
  s.o_empty = b + 13;
  s.k_full = b + 14;
  s.k_empty = s.k_full + ATT_K_STAGES;
  s.v_full = s.k_empty + ATT_K_STAGES;
  s.v_empty = s.v_full + ATT_V_STAGES;
  s.xbar = s.v_empty + ATT_V_STAGES;
  s.tmem_slot = reinterpret_cast<uint32_t*>(base + TILE_REGION + NUM_BARS * 8);
  s.abort = s.tmem_slot + 1;
  s.xval = reinterpret_cast<float*>(base + TILE_REGION + XVAL_OFFSET);
  s.chain = reinterpret_cast<uint32_t*>(base + TILE_REGION + CHAIN_OFFSET);
  return s;
}

struct Unit {
  int u, h, start, cnt;  // self units: start = first query row of Q_user[u][h], cnt = its rows
  bool ok;
  bool self;             // the user's own queries (Q_user) rather than its candidates'
  int L;       // keys of this user
  int kv0;     // first packed row (jagged) or 0
  int ntiles;  // ceil(L / 128)
};

// Self units (see ikbo_attn_self_target_forward) follow the work list's
// units; they are numbered user-major, then head, then query tile, and carry
// this bit in their user field.
constexpr int SELF_UNIT = 1 << 30;

// The work entry is loaded one unit ahead (the load is issued early and only
// waited for where the entry is first used) so the dependent reads of the
// next unit stay off the critical path.
struct UnitCount {
  int target;  // work-list units (read once per CTA)
  int total;   // target + self units
};

template <bool kSelf>
__device__ __forceinline__ int4 load_work(const AttnParams& p, int unit, const UnitCount& n) {
  if (unit >= n.total) return make_int4(-1, -1, -1, -1);
  const int n_target = n.target;
  if (!kSelf || unit < n_target) return __ldg(reinterpret_cast<const int4*>(p.work) + unit);
  const int s = unit - n_target;
  const int per_user = p.H * p.self_tiles;
  const int u = s / per_user;
  const int rem = s - u * per_user;
  const int h = rem / p.self_tiles;
  return make_int4(u | SELF_UNIT, h, rem - h * p.self_tiles, 0);
}

template <bool kSelf>
__device__ __forceinline__ Unit decode(const AttnParams& p, int4 w) {
  Unit x;
  x.self = kSelf && w.x >= 0 && (w.x & SELF_UNIT);
  x.u = x.self ? (w.x & ~SELF_UNIT) : w.x;
  x.h = w.y;
  if (x.self) {
    x.start = w.z * p.self_rows;
    x.cnt = min(p.self_rows, p.Lq_u - x.start);
    x.ok = x.u < p.n_users && x.h >= 0 && x.h < p.H && w.z >= 0 && w.z < p.self_tiles && x.cnt >= 1;
  } else {
    x.start = w.z;
    x.cnt = w.w;
    x.ok = x.u >= 0 && x.u < p.n_users && x.h >= 0 && x.h < p.H && x.cnt >= 1 && x.cnt <= p.cands_per_tile &&
           x.start >= 0 && x.start + x.cnt <= p.n_cand;
  }
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

// stage and phase of the tile with global index g (tiles this CTA has run) in a ring
template <int kStages>
__device__ __forceinline__ int ring_stage(uint32_t g) { return static_cast<int>(g % kStages); }
template <int kStages>
__device__ __forceinline__ uint32_t ring_phase(uint32_t g) { return (g / kStages) & 1u; }

// Keeps the compiler from moving uses of r above a preceding tcgen05.wait.
__device__ __forceinline__ void reg_fence32(uint32_t* r) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

// max of three (one instruction)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// (r0, r1) = (a0, a1) * b + c: one paired fp32 FMA
__device__ __forceinline__ void fma2(float& r0, float& r1, float a0, float a1, float b, float c) {
  asm("{.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %4};\n\t"
      "mov.b64 z, {%5, %5};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\t"
      "mov.b64 {%0, %1}, w;}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (s0, s1) += (a0, a1): one paired fp32 add
__device__ __forceinline__ void add2(float& s0, float& s1, float a0, float a1) {
  asm("{.reg .b64 x, y, w;\n\t"
      "mov.b64 x, {%0, %1};\n\t"
      "mov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 w, x, y;\n\t"
      "mov.b64 {%0, %1}, w;}"
      : "+f"(s0), "+f"(s1)
      : "f"(a0), "f"(a1));
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
// Candidate ids of a unit's Q slots (empty slots read one past the last
// candidate: TMA fills them with zeros).  At most 16 slots (Lq >= 8).
struct QSlots {
  int cand[16];
};

__device__ __forceinline__ void load_slots(const AttnParams& p, const Unit& x, QSlots& q) {
#pragma unroll
  for (int j = 0; j < 16; ++j) q.cand[j] = (x.ok && !x.self && j < x.cnt) ? __ldg(p.perm + x.start + j) : p.n_cand;
}

// K or V tile jt of unit x into a ring stage
__device__ __forceinline__ void load_kv_tile(const AttnParams& p, const CUtensorMap* tm, uint8_t* dst, uint64_t* bar,
                                             const Unit& x, int jt) {
  if (p.kv_offsets) {
    tma_load_3d(dst, tm, bar, 0, x.h, x.kv0 + jt * ATT_BN);
    tma_load_3d(dst + HALF_TILE, tm, bar, 64, x.h, x.kv0 + jt * ATT_BN);
  } else {
    tma_load_4d(dst, tm, bar, 0, jt * ATT_BN, x.h, x.u);
    tma_load_4d(dst + HALF_TILE, tm, bar, 64, jt * ATT_BN, x.h, x.u);
  }
}

template <bool kSelf>
__device__ void att_producer_qk(const AttnParams& p, const AttSmem& s, const CUtensorMap* tmQ,
                                const CUtensorMap* tmQu, const CUtensorMap* tmK, const UnitCount& n_units) {
  uint32_t g = 0;   // K tiles loaded
  uint32_t qc = 0;  // Q tiles loaded
  const int cpt = p.cands_per_tile;
  int unit = blockIdx.x;
  Unit x = decode<kSelf>(p, load_work<kSelf>(p, unit, n_units));
  QSlots qs;
  load_slots(p, x, qs);
  while (unit < n_units.total) {
    const int nunit = unit + static_cast<int>(gridDim.x);
    const int4 nw = load_work<kSelf>(p, nunit, n_units);
    Unit nx;
    QSlots nqs;
    bool prefetched = false;
    if (!x.ok) atomicOr(p.status, DEV_ERR_BAD_WORK);
    if (x.ntiles > 0) {
      const int qb = static_cast<int>(qc & 1u);
      uint8_t* q = s.q + qb * ATT_Q_TILE_BYTES;
      uint64_t* qf = &s.q_full[qb];
      if (!mbar_wait(&s.q_empty[qb], ((qc >> 1) & 1u) ^ 1u, s.abort, p.timeout_ns, 1)) return;
      ++qc;
      if (x.self) {  // rows start .. start + self_rows - 1 of Q_user[u][h] (past Lq_u: TMA zero fill)
        mbar_arrive_expect_tx(qf, static_cast<uint32_t>(p.self_rows * ATT_D * 2));
        tma_load_4d(q, tmQu, qf, 0, x.start, x.h, x.u);
        tma_load_4d(q + HALF_TILE, tmQu, qf, 64, x.start, x.h, x.u);
      } else {
        mbar_arrive_expect_tx(qf, static_cast<uint32_t>(cpt * p.Lq * ATT_D * 2));
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j < cpt) {
            uint8_t* dst = q + j * p.Lq * 128;
            tma_load_4d(dst, tmQ, qf, 0, 0, x.h, qs.cand[j]);
            tma_load_4d(dst + HALF_TILE, tmQ, qf, 64, 0, x.h, qs.cand[j]);
          }
        }
      }
      for (int jt = 0; jt < x.ntiles; ++jt, ++g) {
        const int st = ring_stage<ATT_K_STAGES>(g);
        if (!mbar_wait(&s.k_empty[st], ring_phase<ATT_K_STAGES>(g) ^ 1u, s.abort, p.timeout_ns, 1)) return;
        mbar_arrive_expect_tx(&s.k_full[st], ATT_KV_STAGE_BYTES);
        load_kv_tile(p, tmK, s.k + st * ATT_KV_STAGE_BYTES, &s.k_full[st], x, jt);
        if (!prefetched) {  // the next unit's entry has arrived by now
          prefetched = true;
          nx = decode<kSelf>(p, nw);
          load_slots(p, nx, nqs);
        }
      }
    }
    if (!prefetched) {
      nx = decode<kSelf>(p, nw);
      load_slots(p, nx, nqs);
    }
    x = nx;
    qs = nqs;
    unit = nunit;
  }
}

template <bool kSelf>
__device__ void att_producer_v(const AttnParams& p, const AttSmem& s, const CUtensorMap* tmV, const UnitCount& n_units) {
  uint32_t g = 0;  // V tiles loaded
  int unit = blockIdx.x;
  int4 w = load_work<kSelf>(p, unit, n_units);
  while (unit < n_units.total) {
    const int nunit = unit + static_cast<int>(gridDim.x);
    const int4 nw = load_work<kSelf>(p, nunit, n_units);
    const Unit x = decode<kSelf>(p, w);
    for (int jt = 0; jt < x.ntiles; ++jt, ++g) {
      const int st = ring_stage<ATT_V_STAGES>(g);
      if (!mbar_wait(&s.v_empty[st], ring_phase<ATT_V_STAGES>(g) ^ 1u, s.abort, p.timeout_ns, 1)) return;
      mbar_arrive_expect_tx(&s.v_full[st], ATT_KV_STAGE_BYTES);
      load_kv_tile(p, tmV, s.v + st * ATT_KV_STAGE_BYTES, &s.v_full[st], x, jt);
    }
    w = nw;
    unit = nunit;
  }
}

// ----------------------------------------------------------------- MMA
// Descriptors are built once per tile and advanced by adding (offset >> 4)
// to the start-address field; shared memory is below 256 KB, so the 14-bit
// field never carries into the next one.
//
// S = Q K^T with K-major operands, both in shared memory (128 rows x 128 d
// as two 64-wide d halves; steps 0-3 advance 32 bytes inside the swizzled
// rows of the first half, 4-7 in the second).
__device__ __forceinline__ void issue_qk_ss(uint32_t s_tmem, uint32_t q_base, uint32_t k_base) {
  constexpr uint32_t idesc = idesc_bf16_f32(ATT_BM, ATT_BN, false, false);
  const uint64_t qd = sdesc_sw128(q_base, 16, 1024);
  const uint64_t kd = sdesc_sw128(k_base, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = ((ks >> 2) * HALF_TILE + (ks & 3) * 32) >> 4;
    mma_bf16_ss(s_tmem, qd + off, kd + off, idesc, ks > 0 ? 1u : 0u);
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

// A wait taken by a whole warp: every lane polls, and the lanes agree on the
// outcome so that a timeout never splits the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const AttSmem& s, const AttnParams& p) {
  const bool ok = mbar_wait(bar, parity, s.abort, p.timeout_ns, 1);
  return __all_sync(0xffffffffu, ok);
}

// S issuer (whole warp; one elected lane issues): tile g goes to S_(g&1)
// once group g&1 has read S(g-2) out of it; the unit's Q tile is released
// (for the unit after next) by the unit's last S.
template <bool kSelf>
__device__ void att_s_issuer(const AttnParams& p, const AttSmem& s, uint32_t tmem, const UnitCount& n_units) {
  uint32_t g = 0, qu = 0;
  int unit = blockIdx.x;
  int4 w = load_work<kSelf>(p, unit, n_units);
  while (unit < n_units.total) {
    const int nunit = unit + static_cast<int>(gridDim.x);
    const int4 nw = load_work<kSelf>(p, nunit, n_units);
    const Unit x = decode<kSelf>(p, w);
    if (x.ntiles > 0) {
      const int qb = static_cast<int>(qu & 1u);
      const uint32_t q_base = smem_u32(s.q + qb * ATT_Q_TILE_BYTES);
      for (int jt = 0; jt < x.ntiles; ++jt, ++g) {
        const int b = static_cast<int>(g & 1u);
        const uint32_t n = g >> 1;
        const int kst = ring_stage<ATT_K_STAGES>(g);
        if (!warp_wait(&s.k_full[kst], ring_phase<ATT_K_STAGES>(g), s, p)) return;
        if (n > 0 && !warp_wait(&s.s_free[b], (n - 1) & 1u, s, p)) return;
        if (jt == 0 && !warp_wait(&s.q_full[qb], (qu >> 1) & 1u, s, p)) return;
        tc_fence_after();
        if (elect_one()) {
          issue_qk_ss(tmem + TM_S + b * 128, q_base, smem_u32(s.k + kst * ATT_KV_STAGE_BYTES));
          mma_commit(&s.s_full[b]);
          mma_commit(&s.k_empty[kst]);
          if (jt + 1 == x.ntiles) mma_commit(&s.q_empty[qb]);  // the tile's last reader
        }
        __syncwarp();
      }
      ++qu;
    }
    w = nw;
    unit = nunit;
  }
}

// P.V issuer (whole warp; one elected lane issues): tile g once group g&1
// has written its P; the unit's first one also waits for the previous
// unit's epilogue to have read O.
template <bool kSelf>
__device__ void att_pv_issuer(const AttnParams& p, const AttSmem& s, uint32_t tmem, const UnitCount& n_units) {
  uint32_t g = 0, ou = 0;
  int unit = blockIdx.x;
  int4 w = load_work<kSelf>(p, unit, n_units);
  while (unit < n_units.total) {
    const int nunit = unit + static_cast<int>(gridDim.x);
    const int4 nw = load_work<kSelf>(p, nunit, n_units);
    const Unit x = decode<kSelf>(p, w);
    for (int jt = 0; jt < x.ntiles; ++jt, ++g) {
      const int vst = ring_stage<ATT_V_STAGES>(g);
      const int b = static_cast<int>(g & 1u);
      if (!warp_wait(&s.p_full[b], (g >> 1) & 1u, s, p)) return;
      if (!warp_wait(&s.v_full[vst], ring_phase<ATT_V_STAGES>(g), s, p)) return;
      if (jt == 0 && !warp_wait(s.o_empty, (ou & 1u) ^ 1u, s, p)) return;
      tc_fence_after();
      if (elect_one()) {
        issue_pv(tmem + TM_O, tmem + TM_P + b * 64, smem_u32(s.v + vst * ATT_KV_STAGE_BYTES), jt > 0);
        mma_commit(&s.pv_done[b]);
        mma_commit(&s.v_empty[vst]);
        if (jt + 1 == x.ntiles) mma_commit(s.o_full);
      }
      __syncwarp();
      if (jt + 1 == x.ntiles) ++ou;
    }
    w = nw;
    unit = nunit;
  }
}

// ---------------------------------------------------- softmax + epilogue
struct Lane {
  int quarter, half, r;  // half: the warp's group (its key tiles) and its d half of Q and O
  uint32_t xc;           // exchanges done with the partner warp
};

// Hands `mine` to the other warp of the quarter and returns its value for
// the same row.  Double-buffered by exchange count: a warp refills a buffer
// only after passing the next exchange, i.e. after its partner has read it.
__device__ __forceinline__ bool pair_exchange(const AttnParams& p, const AttSmem& s, Lane& ln, float mine,
                                              float& theirs) {
  const uint32_t buf = ln.xc & 1u;
  s.xval[buf * 256 + ln.half * 128 + ln.r] = mine;
  uint64_t* bar = &s.xbar[ln.quarter * 2 + buf];
  mbar_arrive(bar);
  if (!mbar_wait(bar, (ln.xc >> 1) & 1u, s.abort, p.timeout_ns, 1)) return false;
  theirs = s.xval[buf * 256 + (ln.half ^ 1) * 128 + ln.r];
  ++ln.xc;
  return true;
}

// The reference-maximum chain.  Tile g's group posts the row's reference
// after that tile (tag (g + 1) mod 256 in the low byte of the same 32-bit
// word, so one store publishes both and no fence is needed); tile g + 1,
// the other group's, polls the word.  The word
// is rewritten at every tile, so the word a reader finds is either the one
// it waits for or the one its own group posted a tile earlier (tag one
// less): an 8-bit tag cannot be mistaken.  Every tile, the first of a unit
// included (which ignores the value), waits for the post of the tile before
// it before posting its own, so the posts form one sequence through all of
// the CTA's tiles and none overwrites a word before it has been read.  The reference keeps the high 24
// bits of the fp32 value (both groups use exactly that value, so the
// dropped bits only move the reference by < 2^-15 relative).
__device__ __forceinline__ float chain_value(float m) { return __uint_as_float(__float_as_uint(m) & 0xFFFFFF00u); }

__device__ __forceinline__ void chain_post(const AttSmem& s, int r, uint32_t tag, float m) {
  const uint32_t w = (__float_as_uint(m) & 0xFFFFFF00u) | (tag & 0xFFu);
  asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(smem_u32(s.chain + r)), "r"(w) : "memory");
}

__device__ __forceinline__ uint32_t chain_load(const AttSmem& s, int r) {
  uint32_t w;
  asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(w) : "r"(smem_u32(s.chain + r)) : "memory");
  return w;
}

// Bounded like every wait here; the warp's lanes agree on the outcome.
__device__ __forceinline__ bool chain_wait(const AttnParams& p, const AttSmem& s, int r, uint32_t tag, float& m) {
  tag &= 0xFFu;
  uint32_t w = chain_load(s, r);
  bool ok = true;
  if ((w & 0xFFu) != tag) {
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
      w = chain_load(s, r);
      if ((w & 0xFFu) == tag) break;
      if ((it & 63u) == 0) {
        if (*s.abort) {
          ok = false;
          break;
        }
        if (globaltimer_ns() - t0 > p.timeout_ns) {
          *s.abort = 1;
          ok = false;
          break;
        }
      }
    }
  }
  m = __uint_as_float(w & 0xFFFFFF00u);
  return __all_sync(0xffffffffu, ok);
}

// Does this thread's row (TMEM lane r) hold a query of unit x: one of the
// unit's candidates' rows, or for a self unit one of its Q_user rows?
__device__ __forceinline__ bool row_valid(const Unit& x, int r, int slot, bool row_in_tile) {
  return x.ok && (x.self ? r < x.cnt : (row_in_tile && slot < x.cnt));
}

struct RowOut {
  bool pending;  // a finished unit whose O has not been written yet
  bool valid;    // this thread's row belongs to a candidate of that unit
  __nv_bfloat16* row;
  float l;       // the row sum over this warp's group's tiles, relative to m
  float m;       // the reference of this group's last tile of the unit (-inf if it had none)
  int qb;        // the unit's Q tile (its O is staged there)
};

// The row's natural-log log-sum-exp, m + log2(l) in the log2 domain, into
// the caller's lse array (the row's index is its O row's).
__device__ __forceinline__ void store_lse(const AttnParams& p, const __nv_bfloat16* orow, float lse2) {
  const size_t idx = static_cast<size_t>(reinterpret_cast<const uint16_t*>(orow) - p.O) / ATT_D;
  p.lse[idx] = lse2 * 0.69314718055994531f;
}

// The unit's epilogue, in two parts so that each group can run a tile of
// the next unit in between.  Part 1: the two groups' row sums are brought
// to the unit's last reference and added; once the unit's last P.V is done,
// O / l -> bf16 -> this warp's d half of its 32 rows into its 4 KB of the
// unit's (finished) Q tile (128-byte rows, 16-byte chunk c of row r at
// chunk c ^ (r % 8)); then O may be overwritten.
template <bool kLse>
__device__ __forceinline__ bool att_epilogue_read(const AttnParams& p, const AttSmem& s, uint32_t Ot,
                                                  const RowOut& ro, Lane& ln, uint32_t& ou) {
  float mp, lp;
  if (!pair_exchange(p, s, ln, ro.m, mp)) return false;
  const float mf = fmaxf(ro.m, mp);
  const float lm = ro.l > 0.f ? ro.l * ex2(ro.m - mf) : 0.f;
  if (!pair_exchange(p, s, ln, lm, lp)) return false;
  const float l = lm + lp;
  if (kLse && ro.valid && ln.half == 0) store_lse(p, ro.row, l > 0.f ? mf + __log2f(l) : -INFINITY);
  if (!mbar_wait(s.o_full, ou & 1u, s.abort, p.timeout_ns, 1)) return false;
  ++ou;
  tc_fence_after();
  const float inv = l > 0.f ? 1.0f / l : 0.f;
  const int lane = static_cast<int>(lane_id());
  uint8_t* stage = s.q + ro.qb * ATT_Q_TILE_BYTES + ((ln.quarter * 2 + ln.half) << 12);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    uint32_t o[32];
    tmem_ld32(Ot + c * 32, o);
    tmem_ld_wait(o);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 w;
      w.x = pack_bf16x2(__uint_as_float(o[8 * k + 0]) * inv, __uint_as_float(o[8 * k + 1]) * inv);
      w.y = pack_bf16x2(__uint_as_float(o[8 * k + 2]) * inv, __uint_as_float(o[8 * k + 3]) * inv);
      w.z = pack_bf16x2(__uint_as_float(o[8 * k + 4]) * inv, __uint_as_float(o[8 * k + 5]) * inv);
      w.w = pack_bf16x2(__uint_as_float(o[8 * k + 6]) * inv, __uint_as_float(o[8 * k + 7]) * inv);
      *reinterpret_cast<uint4*>(stage + lane * 128 + (((4 * c + k) ^ (lane & 7)) << 4)) = w;
    }
  }
  tc_fence_before();
  mbar_arrive(s.o_empty);
  return true;
}

// Part 2: the staged rows to global memory, 4 rows per store instruction (8
// lanes per contiguous 128-byte half row); then the Q tile may be refilled.
__device__ __forceinline__ void att_epilogue_store(const AttSmem& s, const RowOut& ro, const Lane& ln) {
  __syncwarp();  // every lane's staging writes are visible to the warp
  const int lane = static_cast<int>(lane_id());
  const uint8_t* stage = s.q + ro.qb * ATT_Q_TILE_BYTES + ((ln.quarter * 2 + ln.half) << 12);
  const int chunk = lane & 7;
  const uint64_t my_row = reinterpret_cast<uint64_t>(ro.row);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = 4 * i + (lane >> 3);
    const uint64_t dst_row = __shfl_sync(0xffffffffu, my_row, r);
    const bool valid = __shfl_sync(0xffffffffu, ro.valid, r);
    const uint4 w = *reinterpret_cast<const uint4*>(stage + r * 128 + ((chunk ^ (r & 7)) << 4));
    if (valid) reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dst_row) + ln.half * 64)[chunk] = w;
  }
  mbar_arrive(&s.q_empty[ro.qb]);  // the staging rows are read: the tile may take the next Q
}

// One softmax warp: the key tiles g of its group (g % 2 == group) of every
// unit, all 128 columns of its 32 rows; the previous unit's epilogue (its d
// half of O) is interleaved with the group's first tiles of the next unit:
// its O is read out after the group's first tile (so that tile overlaps the
// previous unit's last P.V) and stored after the second.
// kLse: also write each row's log-sum-exp (target units only).
template <bool kSelf, bool kLse>
__device__ void att_softmax(const AttnParams& p, const AttSmem& s, uint32_t tmem, const UnitCount& n_units) {
  const int warp = threadIdx.x >> 5;
  Lane ln;
  ln.quarter = warp & 3;                                     // TMEM lane quarter of this warp
  ln.half = (warp - SOFTMAX_WARP0) >> 2;                     // group = d half of O
  ln.r = (ln.quarter << 5) + static_cast<int>(lane_id());    // row = TMEM lane
  ln.xc = 0;
  const int grp = ln.half;
  const uint32_t lane_base = static_cast<uint32_t>(ln.quarter * 32) << 16;
  const uint32_t St = tmem + lane_base + TM_S + grp * 128;  // this group's S
  const uint32_t Pt = tmem + lane_base + TM_P + grp * 64;   // and its P
  const uint32_t Oall = tmem + lane_base + TM_O;
  const uint32_t Ot = Oall + grp * 64;
  const float sl = p.scale_log2;
  const int slot = ln.r / p.Lq;
  const int qrow = ln.r % p.Lq;
  const bool row_in_tile = ln.r < p.cands_per_tile * p.Lq;
  uint32_t g = 0, qc = 0, ou = 0;
  RowOut prev = {false, false, nullptr, 0.f, -INFINITY, 0};

  int unit = blockIdx.x;
  Unit x = decode<kSelf>(p, load_work<kSelf>(p, unit, n_units));
  bool rv = row_valid(x, ln.r, slot, row_in_tile);
  int cand = (rv && !x.self) ? __ldg(p.perm + x.start + slot) : 0;
  while (unit < n_units.total) {
    const int nunit = unit + static_cast<int>(gridDim.x);
    const int4 nw = load_work<kSelf>(p, nunit, n_units);
    Unit nx;
    bool nrv = false;
    int ncand = 0;
    bool prefetched = false;
    __nv_bfloat16* orow = nullptr;
    if (rv)
      orow = x.self ? reinterpret_cast<__nv_bfloat16*>(p.O_user) +
                          ((static_cast<size_t>(x.u) * p.H + x.h) * p.Lq_u + x.start + ln.r) * ATT_D
                    : reinterpret_cast<__nv_bfloat16*>(p.O) + ((static_cast<size_t>(cand) * p.H + x.h) * p.Lq + qrow) * ATT_D;

    if (x.ntiles == 0) {  // empty key range: O = 0 (and LSE = -inf)
      if (rv) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 8; ++c) reinterpret_cast<uint4*>(orow + grp * 64)[c] = z;
        if (kLse && grp == 0) store_lse(p, orow, -INFINITY);
      }
    } else {
      const int qb = static_cast<int>(qc & 1u);
      ++qc;
      int epi = prev.pending ? 1 : 0;  // the previous unit's epilogue: 1 read O next, 2 store it next
      int mine = 0;                     // this group's tiles of the unit so far
      float mref = -INFINITY, l = 0.f;  // this group's reference and row sum
      // this group's key tiles only: g, the tile's place in the CTA's sequence,
      // runs over g % 2 == group (visiting every tile to skip half of them
      // cost the group ~3 % of the kernel's time in loop control)
      const uint32_t g0 = g;
      for (int jt = static_cast<int>((static_cast<uint32_t>(grp) - g0) & 1u); jt < x.ntiles; jt += 2) {
        g = g0 + static_cast<uint32_t>(jt);
        if (!mbar_wait(&s.s_full[grp], (g >> 1) & 1u, s.abort, p.timeout_ns, 1)) return;
        tc_fence_after();
        const int ncols = min(ATT_BN, x.L - jt * ATT_BN);  // valid key columns of this tile
        uint32_t v[128];
        tmem_ld32p(St, v);
        tmem_ld32p(St + 32, v + 32);
        tmem_ld32p(St + 64, v + 64);
        tmem_ld32p(St + 96, v + 96);
        tmem_ld_wait();
        reg_fence32(v);
        reg_fence32(v + 32);
        reg_fence32(v + 64);
        reg_fence32(v + 96);
        tc_fence_before();
        mbar_arrive(&s.s_free[grp]);  // S_b may take S(g + 2) now
        if (ncols < ATT_BN) {
#pragma unroll
          for (int j = 0; j < ATT_BN; ++j)
            if (j >= ncols) v[j] = __float_as_uint(-INFINITY);
        }
        const uint32_t cw = chain_load(s, ln.r);  // usually posted long ago: read it early
        float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
        for (int j = 0; j < ATT_BN; j += 8) {
          mx0 = fmax3(mx0, __uint_as_float(v[j]), __uint_as_float(v[j + 1]));
          mx1 = fmax3(mx1, __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
          mx2 = fmax3(mx2, __uint_as_float(v[j + 4]), __uint_as_float(v[j + 5]));
          mx3 = fmax3(mx3, __uint_as_float(v[j + 6]), __uint_as_float(v[j + 7]));
        }
        const float mx = fmax3(mx0, mx1, fmaxf(mx2, mx3)) * sl;
        // the reference after the tile before (posted by the other group, or
        // by either at the end of the previous unit; the first tile of a unit
        // only waits for it and starts afresh)
        float mprev = __uint_as_float(cw & 0xFFFFFF00u);
        if (!__all_sync(0xffffffffu, (cw & 0xFFu) == (g & 0xFFu)) && !chain_wait(p, s, ln.r, g, mprev)) return;
        if (jt == 0) mprev = -INFINITY;
        // tcgen05.ld/st are warp-collective: the rescale decision must be
        // uniform across the warp, so any row that needs it moves all 32
        const bool rescale = __any_sync(0xffffffffu, mx > mprev + RESCALE_THRESHOLD);
        const float mj = rescale ? chain_value(fmaxf(mprev, mx)) : mprev;
        chain_post(s, ln.r, g + 1, mj);
        if (mj != mref) {  // this group's sum follows the reference (l = 0 on its first tile)
          l *= ex2(mref - mj);
          mref = mj;
        }
        // p = 2^(s*sl - mj) (masked columns give 2^-inf = 0) as bf16 pairs
        // into P_b, 32 columns at a time (P_b is free once P.V(g - 2) has
        // read it); P.V may read them after p_full
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t pk[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float t0, t1;
            fma2(t0, t1, __uint_as_float(v[64 * h + 2 * j]), __uint_as_float(v[64 * h + 2 * j + 1]), sl, -mj);
            const float p0 = ex2(t0);
            const float p1 = ex2(t1);
            add2(l0, l1, p0, p1);
            pk[j] = pack_bf16x2(p0, p1);
          }
          if (h == 0) {
            if (g >= 2 && !mbar_wait(&s.pv_done[grp], ((g >> 1) - 1) & 1u, s.abort, p.timeout_ns, 1)) return;
            tc_fence_after();
          }
          tmem_st32p(Pt + 32 * h, pk);
        }
        l += l0 + l1;
        if (rescale && jt > 0) {
          // O must hold only this unit's P.V: the previous unit's O is read out first
          if (epi == 1) {
            if (!att_epilogue_read<kLse>(p, s, Ot, prev, ln, ou)) return;
            epi = 2;
          }
          // O holds P.V of tiles 0 .. jt-1 relative to mprev: once the last of
          // them is done, scale all of O's columns of these rows to mj
          const uint32_t gp = g - 1;
          if (!mbar_wait(&s.pv_done[gp & 1u], (gp >> 1) & 1u, s.abort, p.timeout_ns, 1)) return;
          tc_fence_after();
          const float alpha = ex2(mprev - mj);
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(Oall + c * 32, o);
            tmem_ld_wait(o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(Oall + c * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&s.p_full[grp]);
        ++mine;
        if (epi == 1) {  // after the group's first tile: read out the previous unit's O
          if (!att_epilogue_read<kLse>(p, s, Ot, prev, ln, ou)) return;
          epi = 2;
        } else if (epi == 2 && mine >= 2) {  // after its second: store it
          att_epilogue_store(s, prev, ln);
          epi = 0;
        }
        if (!prefetched) {  // the next unit's entry and this row's candidate in it
          prefetched = true;
          nx = decode<kSelf>(p, nw);
          nrv = row_valid(nx, ln.r, slot, row_in_tile);
          ncand = (nrv && !nx.self) ? __ldg(p.perm + nx.start + slot) : 0;
        }
      }
      g = g0 + static_cast<uint32_t>(x.ntiles);
      if (epi == 1 && !att_epilogue_read<kLse>(p, s, Ot, prev, ln, ou)) return;
      if (epi >= 1) att_epilogue_store(s, prev, ln);
      prev.pending = true;
      prev.valid = rv;
      prev.row = orow;
      prev.l = l;
      prev.m = mref;
      prev.qb = qb;
    }
    if (!prefetched) {
      nx = decode<kSelf>(p, nw);
      nrv = row_valid(nx, ln.r, slot, row_in_tile);
      ncand = (nrv && !nx.self) ? __ldg(p.perm + nx.start + slot) : 0;
    }
    x = nx;
    rv = nrv;
    cand = ncand;
    unit = nunit;
  }
  if (prev.pending && att_epilogue_read<kLse>(p, s, Ot, prev, ln, ou)) att_epilogue_store(s, prev, ln);
}

// kSelf: the launch also runs self units (ikbo_attn_self_target_forward);
// without them the self branches compile away.  kLse: the softmax warps also
// write each row's log-sum-exp (ikbo_attn_forward_lse; never with kSelf).
template <bool kSelf, bool kLse>
__global__ void __launch_bounds__(ATT_THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQu,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;
  if (pad + SMEM_USED > SMEM_ALLOC) {  // uniform across the CTA, before any barrier exists
    if (threadIdx.x == 0) atomicOr(p.status, DEV_ERR_SMEM_LAYOUT);
    return;
  }
  const AttSmem s = carve(smem_raw + pad);
  const int warp = threadIdx.x >> 5;
  UnitCount n_units;  // work-list units, then self units
  n_units.target = (kSelf && p.self_only) ? 0 : *p.n_units;
  n_units.total = n_units.target + (kSelf ? p.n_self : 0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 1 + SOFTMAX_THREADS);  // the unit's last S, then its epilogue's staging
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.s_free[i], GROUP_THREADS);
      mbar_init(&s.p_full[i], GROUP_THREADS);
      mbar_init(&s.pv_done[i], 1);
    }
    mbar_init(s.o_full, 1);
    mbar_init(s.o_empty, SOFTMAX_THREADS);
    for (int i = 0; i < ATT_K_STAGES; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < ATT_V_STAGES; ++i) {
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    for (int i = 0; i < 8; ++i) mbar_init(&s.xbar[i], 64);
    for (int r = 0; r < ATT_BM; ++r) s.chain[r] = 0;  // tag 0: no tile has posted (tags start at 1)
    *s.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmQ);
    if (kSelf) tma_prefetch_desc(&tmQu);
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

  // registers: launched at 168 per thread (384 x 168 = 64512); the four
  // control warps give back down to CTRL_REGS and the softmax warps, which
  // hold a whole 128-column tile row each, take SOFTMAX_REGS
  // (128 x CTRL_REGS + 256 x SOFTMAX_REGS = 64512)
  if (warp < SOFTMAX_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(CTRL_REGS));
    if (warp == 0) {
      if (lane_id() == 0) att_producer_qk<kSelf>(p, s, &tmQ, &tmQu, &tmK, n_units);
    } else if (warp == 3) {
      if (lane_id() == 0) att_producer_v<kSelf>(p, s, &tmV, n_units);
    } else if (warp == 1) {
      att_s_issuer<kSelf>(p, s, tmem, n_units);
    } else {
      att_pv_issuer<kSelf>(p, s, tmem, n_units);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(SOFTMAX_REGS));
    att_softmax<kSelf, kLse>(p, s, tmem, n_units);
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

size_t attn_smem_bytes() { return SMEM_ALLOC; }

cudaError_t launch_attn(const CUtensorMap& tmQ, const CUtensorMap& tmQu, const CUtensorMap& tmK,
                        const CUtensorMap& tmV, const AttnParams& p, int grid, cudaStream_t s) {
  const size_t smem = attn_smem_bytes();
  if (p.n_self > 0 && p.lse) return cudaErrorInvalidValue;
  auto kernel = p.n_self > 0 ? attn_fwd_kernel<true, false>
                             : (p.lse ? attn_fwd_kernel<false, true> : attn_fwd_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kernel<<<grid, ATT_THREADS, smem, s>>>(tmQ, tmQu, tmK, tmV, p);
  return cudaGetLastError();
}

}  // namespace ikbo
