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
// head) and up to 2 x floor(128 / Lq) of that user's candidates (from the
// segment builder's perm), i.e. two 128-row query tiles that read every K/V
// tile once from shared memory.  Units of the same (user, head) are adjacent
// in the work list, so neighbouring CTAs stream the same K/V through L2.
//
// Per CTA (persistent, one per SM, 12 warps = 3 warpgroups):
//   warp 0      TMA producer: Q tiles (one box per candidate and d-half,
//               gathered through perm), K/V tiles through a 5-stage ring
//   warp 1      MMA issuer of query tile 0 (one lane) and TMEM owner (512
//               columns: S0 S1 O0 O1, 128 each): S_t = Q_t K^T (SS),
//               O_t += P_t V (TS: P in TMEM)
//   warp 2      MMA issuer of query tile 1
//   warp 3      idle
//   warps 4-7   softmax + epilogue of query tile 0 (one thread per row; warp w
//               reaches TMEM lanes 32*(w%4) .. +31)
//   warps 8-11  softmax + epilogue of query tile 1
// Registers: launched at 168 per thread (384 x 168 = 64512); the first
// warpgroup gives back down to 136 and the softmax warpgroups take 184 each
// (128 x 136 + 256 x 184 = 64512), enough to hold a whole 128-column row of S.
// Each query tile has its own Q buffer and full/empty barriers, so the next
// unit's Q tile t is fetched as soon as the last S_t of the current unit has
// been computed, overlapping the current unit's last P.V products.
// Online softmax in fp32 in the log2 domain (exp2 with scale*log2(e) folded
// in); the running max is only moved when it grows by more than 2^8, so O is
// rescaled rarely (the result is the same: O and l share the reference max).
// P is rounded to bf16 and written over the first 64 columns of S.
#include <cuda_bf16.h>

#include "ikbo_internal.h"
#include "ptx.cuh"

namespace ikbo {

namespace {

constexpr uint32_t HALF_TILE = ATT_BM * 64 * 2;  // 128 rows x 64 bf16 = 16 KB
constexpr float RESCALE_THRESHOLD = 8.0f;          // log2 units
constexpr int SOFTMAX_WARP0 = 4;                   // first softmax warp
constexpr uint32_t REGS_CONTROL = 136;             // warpgroup 0 after setmaxnreg.dec
constexpr uint32_t REGS_SOFTMAX = 184;             // warpgroups 1, 2 after setmaxnreg.inc

struct AttSmem {
  uint8_t* q;      // 2 tiles x 32 KB
  uint8_t* kv;     // ATT_STAGES x 32 KB
  uint64_t* q_full;   // [2]
  uint64_t* q_empty;  // [2]
  uint64_t* kv_full;
  uint64_t* kv_empty;
  uint64_t* s_full;   // [2]
  uint64_t* p_full;   // [2]
  uint64_t* o_full;   // [2]
  uint64_t* o_empty;  // [2]
  uint64_t* tok;      // [2] issuer turns
  uint32_t* tmem_slot;
  uint32_t* abort;
};

__device__ __forceinline__ AttSmem carve(uint8_t* base) {
  AttSmem s;
  s.q = base;
  s.kv = base + ATT_TILES * ATT_Q_TILE_BYTES;
  uint64_t* b = reinterpret_cast<uint64_t*>(s.kv + ATT_STAGES * ATT_KV_STAGE_BYTES);
  s.q_full = b;
  s.q_empty = b + 2;
  s.kv_full = b + 4;
  s.kv_empty = s.kv_full + ATT_STAGES;
  s.s_full = s.kv_empty + ATT_STAGES;
  s.p_full = s.s_full + 2;
  s.o_full = s.p_full + 2;
  s.o_empty = s.o_full + 2;
  s.tok = s.o_empty + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.tok + 2);
  s.abort = s.tmem_slot + 1;
  return s;
}

struct Unit {
  int u, h, start, cnt;
  int ntq;     // query tiles in use (0 = skip the unit)
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
  const int cap = 2 * p.cands_per_tile;
  const bool ok = x.u >= 0 && x.u < p.n_users && x.h >= 0 && x.h < p.H && x.cnt >= 1 && x.cnt <= cap &&
                  x.start >= 0 && x.start + x.cnt <= p.n_cand;
  if (!ok) {
    x.ntq = 0;
    x.L = 0;
    x.kv0 = 0;
    x.ntiles = 0;
    return x;
  }
  x.ntq = x.cnt > p.cands_per_tile ? 2 : 1;
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

// ------------------------------------------------------------ producer
__device__ void att_producer(const AttnParams& p, const AttSmem& s, const CUtensorMap* tmQ, const CUtensorMap* tmK,
                             const CUtensorMap* tmV, int n_units) {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t q_uses[2] = {0, 0};
  const int cpt = p.cands_per_tile;
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit x = decode(p, unit);
    if (x.ntq == 0) {
      atomicOr(p.status, DEV_ERR_BAD_WORK);
      continue;
    }
    if (x.ntiles == 0) continue;
    for (int t = 0; t < x.ntq; ++t) {
      if (!mbar_wait(&s.q_empty[t], (q_uses[t] & 1u) ^ 1u, s.abort, p.timeout_ns, 1)) return;
      ++q_uses[t];
      mbar_arrive_expect_tx(&s.q_full[t], static_cast<uint32_t>(cpt * p.Lq * ATT_D * 2));
      for (int j = 0; j < cpt; ++j) {
        const int slot = t * cpt + j;
        // empty slots read one past the last candidate: TMA fills them with zeros
        const int cand = slot < x.cnt ? p.perm[x.start + slot] : p.n_cand;
        uint8_t* dst = s.q + t * ATT_Q_TILE_BYTES + j * p.Lq * 128;
        tma_load_4d(dst, tmQ, &s.q_full[t], 0, 0, x.h, cand);
        tma_load_4d(dst + HALF_TILE, tmQ, &s.q_full[t], 64, 0, x.h, cand);
      }
    }
    for (int jt = 0; jt < x.ntiles; ++jt) {
      for (int kv = 0; kv < 2; ++kv) {
        if (!mbar_wait(&s.kv_empty[stage], phase ^ 1u, s.abort, p.timeout_ns, 1)) return;
        mbar_arrive_expect_tx(&s.kv_full[stage], ATT_KV_STAGE_BYTES);
        uint8_t* dst = s.kv + stage * ATT_KV_STAGE_BYTES;
        const CUtensorMap* tm = kv == 0 ? tmK : tmV;
        if (p.kv_offsets) {
          tma_load_3d(dst, tm, &s.kv_full[stage], 0, x.h, x.kv0 + jt * ATT_BN);
          tma_load_3d(dst + HALF_TILE, tm, &s.kv_full[stage], 64, x.h, x.kv0 + jt * ATT_BN);
        } else {
          tma_load_4d(dst, tm, &s.kv_full[stage], 0, jt * ATT_BN, x.h, x.u);
          tma_load_4d(dst + HALF_TILE, tm, &s.kv_full[stage], 64, jt * ATT_BN, x.h, x.u);
        }
        if (++stage == ATT_STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  }
}

// ----------------------------------------------------------------- MMA
// S_t = Q_t K^T: A = Q tile (K-major, 128 x 128), B = K tile (K-major).
// The d = 128 reduction is 8 steps of 16: steps 0-3 in the first 64-wide
// half (32-byte advances inside the swizzled row), 4-7 in the second.
// Descriptors are built once per tile and advanced by adding (offset >> 4)
// to the start-address field; shared memory is below 256 KB, so the 14-bit
// field never carries into the next one.
__device__ __forceinline__ void issue_qk(uint32_t s_tmem, uint32_t q_base, uint32_t k_base) {
  constexpr uint32_t idesc = idesc_bf16_f32(ATT_BM, ATT_BN, false, false);
  const uint64_t qd = sdesc_sw128(q_base, 16, 1024);
  const uint64_t kd = sdesc_sw128(k_base, 16, 1024);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = ((ks >> 2) * HALF_TILE + (ks & 3) * 32) >> 4;
    mma_bf16_ss(s_tmem, qd + off, kd + off, idesc, ks > 0 ? 1u : 0u);
  }
}

// O_t += P_t V: A = P (TMEM, 128 rows x 128 keys as 64 packed columns), B =
// V tile (MN-major: d contiguous; 64-wide d halves one HALF_TILE apart, 8 key
// rows per 1024-byte atom).  16 keys per step = 8 TMEM columns of P.
__device__ __forceinline__ void issue_pv(uint32_t o_tmem, uint32_t p_tmem, uint32_t v_base, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(ATT_BM, ATT_D, false, true);
  const uint64_t vd = sdesc_sw128(v_base, HALF_TILE, 1024);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    mma_bf16_ts(o_tmem, p_tmem + ks * 8, vd + ((ks * 2048u) >> 4), idesc, (accumulate || ks > 0) ? 1u : 0u);
  }
}

// One issuer per query tile (warp 1 issues tile 0, warp 2 tile 1), taking
// turns.  A burst is what one tile issues between two of its softmax steps:
// S_t(0) at the start of a unit, then P_t V (+ the next S_t) per key tile.
// The tensor pipe queues only a few instructions, so a lone issuer that
// stops to check its barriers lets the pipe drain; here each issuer does its
// checks while the other's burst is in the pipe.  The bursts alternate
// (tile 0's b-th, tile 1's b-th, tile 0's (b+1)-th, ...) through two token
// barriers, which keeps the tiles half a period apart, so one tile's softmax
// always overlaps the other tile's products.
// Each K/V stage is released once by each issuer (kv_empty counts 2).  When
// a unit uses only tile 0, the tile-1 issuer still walks the unit burst by
// burst -- waits for each stage to be loaded, releases it with a plain
// arrive, takes and passes its turn -- so the stage and token counts of the
// two issuers never drift apart (the parity waits could not tell the laps
// apart if one issuer ran a full lap ahead).
__device__ void att_mma(const AttnParams& p, const AttSmem& s, uint32_t tmem, int n_units, int t) {
  int stage = 0;
  uint32_t phase = 0;
  uint32_t q_uses = 0, p_uses = 0, o_uses = 0, bursts = 0;
  const uint32_t q_base = smem_u32(s.q) + t * ATT_Q_TILE_BYTES;
  const uint32_t s_tmem = tmem + t * 128;
  const uint32_t o_tmem = tmem + 256 + t * 128;
  auto advance = [&]() {
    if (++stage == ATT_STAGES) {
      stage = 0;
      phase ^= 1u;
    }
  };
  // wait until the other issuer has issued its previous burst
  auto take_turn = [&]() -> bool {
    if (t == 0) return bursts == 0 || mbar_wait(&s.tok[1], (bursts - 1) & 1u, s.abort, p.timeout_ns, 1);
    return mbar_wait(&s.tok[0], bursts & 1u, s.abort, p.timeout_ns, 1);
  };
  auto pass_turn = [&]() {
    mbar_arrive(&s.tok[t]);
    ++bursts;
  };
  // an empty tile's burst: stages go by in order, released without use
  auto pass_stages = [&](int n) -> bool {
    for (int i = 0; i < n; ++i) {
      if (!mbar_wait(&s.kv_full[stage], phase, s.abort, p.timeout_ns, 1)) return false;
      mbar_arrive(&s.kv_empty[stage]);
      advance();
    }
    if (!take_turn()) return false;
    pass_turn();
    return true;
  };
  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit x = decode(p, unit);
    if (x.ntq == 0 || x.ntiles == 0) continue;
    if (t >= x.ntq) {
      if (!pass_stages(1)) return;                                             // burst of S(0)
      for (int jt = 0; jt < x.ntiles; ++jt)
        if (!pass_stages(jt + 1 < x.ntiles ? 2 : 1)) return;                    // bursts of P.V (+ S)
      continue;
    }
    int k_stage = stage;
    if (!mbar_wait(&s.kv_full[k_stage], phase, s.abort, p.timeout_ns, 1)) return;
    advance();
    if (!mbar_wait(&s.q_full[t], q_uses & 1u, s.abort, p.timeout_ns, 1)) return;
    ++q_uses;
    if (!take_turn()) return;
    tc_fence_after();
    issue_qk(s_tmem, q_base, smem_u32(s.kv + k_stage * ATT_KV_STAGE_BYTES));
    mma_commit(&s.s_full[t]);
    if (x.ntiles == 1) mma_commit(&s.q_empty[t]);  // that was the last S_t of the unit
    mma_commit(&s.kv_empty[k_stage]);
    pass_turn();
    for (int jt = 0; jt < x.ntiles; ++jt) {
      const int v_stage = stage;
      if (!mbar_wait(&s.kv_full[v_stage], phase, s.abort, p.timeout_ns, 1)) return;
      advance();
      const bool has_next = jt + 1 < x.ntiles;
      if (has_next) {
        k_stage = stage;
        if (!mbar_wait(&s.kv_full[k_stage], phase, s.abort, p.timeout_ns, 1)) return;
        advance();
      }
      if (!mbar_wait(&s.p_full[t], p_uses & 1u, s.abort, p.timeout_ns, 1)) return;
      ++p_uses;
      if (jt == 0) {
        // the previous unit's epilogue must be done reading O_t
        if (!mbar_wait(&s.o_empty[t], (o_uses & 1u) ^ 1u, s.abort, p.timeout_ns, 1)) return;
      }
      if (!take_turn()) return;
      tc_fence_after();
      issue_pv(o_tmem, s_tmem, smem_u32(s.kv + v_stage * ATT_KV_STAGE_BYTES), jt > 0);
      mma_commit(&s.kv_empty[v_stage]);
      if (!has_next) {
        mma_commit(&s.o_full[t]);
        ++o_uses;
      } else {
        issue_qk(s_tmem, q_base, smem_u32(s.kv + k_stage * ATT_KV_STAGE_BYTES));
        mma_commit(&s.s_full[t]);
        if (jt + 2 == x.ntiles) mma_commit(&s.q_empty[t]);  // last S_t of the unit
        mma_commit(&s.kv_empty[k_stage]);
      }
      pass_turn();
    }
  }
}

// ---------------------------------------------------- softmax + epilogue
__device__ void att_softmax(const AttnParams& p, const AttSmem& s, uint32_t tmem, int n_units) {
  const int warp = threadIdx.x >> 5;
  const int wg = (warp - SOFTMAX_WARP0) >> 2;                      // query tile 0 or 1
  const int quarter = warp & 3;                                    // TMEM lane quarter of this warp
  const int r = (quarter << 5) + static_cast<int>(lane_id());     // row = TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t S = tmem + lane_base + wg * 128;
  const uint32_t Ot = tmem + lane_base + 256 + wg * 128;
  const int cpt = p.cands_per_tile;
  const float sl = p.scale_log2;
  uint32_t s_uses = 0, o_uses = 0;

  for (int unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit x = decode(p, unit);
    if (x.ntq <= wg) continue;
    const int slot = wg * cpt + r / p.Lq;
    const int q = r % p.Lq;
    const bool row_valid = r < cpt * p.Lq && slot < x.cnt;
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
    float m = -INFINITY, l = 0.f;
    for (int jt = 0; jt < x.ntiles; ++jt) {
      if (!mbar_wait(&s.s_full[wg], s_uses & 1u, s.abort, p.timeout_ns, 1)) return;
      ++s_uses;
      tc_fence_after();
      const int ncols = min(ATT_BN, x.L - jt * ATT_BN);
      // the whole 128-column row of S in registers: one wait for four loads
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
      if (ncols < ATT_BN) {
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j >= ncols) v[j] = __float_as_uint(-INFINITY);
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 128; j += 4) {
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
      // p = 2^(s*sl - m) (masked columns give 2^-inf = 0), bf16 pairs over S[0, 64)
      float l0 = 0.f, l1 = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float p0 = ex2(fmaf(__uint_as_float(v[c * 32 + 2 * j]), sl, -m));
          const float p1 = ex2(fmaf(__uint_as_float(v[c * 32 + 2 * j + 1]), sl, -m));
          l0 += p0;
          l1 += p1;
          pk[j] = pack_bf16x2(p0, p1);
        }
        tmem_st16(S + c * 16, pk);
      }
      l += l0 + l1;
      if (rescale && jt > 0) {
        // O_t of the previous tiles: the P.V that wrote it completed before this S
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
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_full[wg]);
    }
    // epilogue: O / l -> bf16 -> O[cand, h, q, :]
    if (!mbar_wait(&s.o_full[wg], o_uses & 1u, s.abort, p.timeout_ns, 1)) return;
    ++o_uses;
    tc_fence_after();
    const float inv = l > 0.f ? 1.0f / l : 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tmem_ld32(Ot + c * 32, o);
      tmem_ld_wait(o);
      if (row_valid) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          pk[j] = pack_bf16x2(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
      }
    }
    tc_fence_before();
    mbar_arrive(&s.o_empty[wg]);
  }
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
      mbar_init(&s.q_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
      mbar_init(&s.o_full[i], 1);
      mbar_init(&s.o_empty[i], 128);
      mbar_init(&s.tok[i], 1);
    }
    for (int i = 0; i < ATT_STAGES; ++i) {
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 2);  // one release per query tile
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

  if (warp < SOFTMAX_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(REGS_CONTROL));
    if (warp == 0) {
      if (lane_id() == 0) att_producer(p, s, &tmQ, &tmK, &tmV, n_units);
    } else if (warp == 1 || warp == 2) {
      if (lane_id() == 0) att_mma(p, s, tmem, n_units, warp - 1);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(REGS_SOFTMAX));
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
  return 1024 + ATT_TILES * ATT_Q_TILE_BYTES + ATT_STAGES * ATT_KV_STAGE_BYTES + 256;
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
