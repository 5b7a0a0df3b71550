// lce.cu -- fused Linear Compression Embedding with in-kernel broadcast.
//
// Y[i][n][d] = sum_k Wc[k][n] C[i][k][d] + P[map[i]][n][d],
// P[u][n][d] = b[n] + sum_k Wu[k][n] U[u][k][d].
//
// This is the four-stage IKBO LCE of aixai.ru, "Deep Dive: Linear
// Compression" (and "Meta Optimizes Inference for Recommendation Systems",
// LCE case), rebuilt for sm_103a:
//   stage 1, split along K: the user GEMM runs at n_users, the candidate GEMM
//     at n_cand; only the small user result P is broadcast;
//   stage 2, K padding: K is padded with zeros to the MMA step, but only in
//     shared memory -- TMA fills the out-of-bounds rows of both operands with
//     zeros, so no padded copy of any tensor exists;
//   stage 3, broadcast-add in the candidate GEMM's epilogue: the epilogue
//     reads P[map[i]] by index and adds it in registers; Y is written once;
//   stage 4, one persistent warp-specialised launch: user tiles and candidate
//     tiles share the launch, user tiles first in every CTA's static order,
//     and a candidate epilogue acquires the release flag of its user tile.
//
// Schedules of one persistent kernel body (one CTA per SM):
//   two launches: the user tiles, then the candidate tiles;
//   one launch: user tiles first in every CTA's list, candidate tiles after;
//   local partials: one launch of candidate tiles only; before the first
//     candidate tile of each (user, D block) a CTA computes that user's
//     partial itself, into TMEM, and its epilogue keeps it in registers --
//     no workspace, no hand-off between CTAs (the user GEMM is repeated by the
//     few CTAs that share a user: the work is small and U stays in L2).
// Per CTA:
//   warp 0  TMA producer   (A ring: U[u] or C[i] chunks; W chunks / resident Wc)
//   warp 1  MMA issuer     (tcgen05.mma, fp32 accumulators in TMEM, 2 buffers)
//   warp 2  TMEM owner     (alloc / dealloc of 512 columns)
//   warps 4-11 epilogue    (tcgen05.ld, + P or + b, bf16 or fp32 stores)
//
// Tile: 128 rows of D (TMEM lanes) x N_mma columns (N rounded up to 16) of
// one candidate (or user).  Operands are MN-major (D and N are the contiguous
// dimensions in memory), staged by TMA with 128-byte swizzle: a box of 64
// elements along D (or N) by 64 k rows, 8 KB.
#include <cuda_bf16.h>

#include "ikbo_internal.h"
#include "ptx.cuh"

namespace ikbo {

namespace {

constexpr uint32_t BOX_BYTES = 64 * 64 * 2;  // one 64 x 64 bf16 box

struct LceSmem {
  uint8_t* w_region;
  uint8_t* a_ring;
  uint64_t* a_full;
  uint64_t* a_empty;
  uint64_t* w_full;
  uint64_t* w_empty;
  uint8_t* wu_ring;    // local-partial schedule: full-width W_u chunks (NB boxes each)
  uint64_t* wu_full;
  uint64_t* wu_empty;
  uint64_t* wc_full;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint64_t* pub;  // the 128 epilogue threads finished writing a user partial
  uint32_t* tmem_slot;
  uint32_t* abort;
  long long* range;  // local-partial schedule: this CTA's [q0, q1) of candidate tiles
};

__device__ __forceinline__ LceSmem carve(uint8_t* base, const LceParams& p) {
  LceSmem s;
  s.w_region = base;
  s.a_ring = base + p.w_region_bytes;
  s.wu_ring = s.a_ring + static_cast<size_t>(p.stages) * LCE_A_STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(s.wu_ring + static_cast<size_t>(p.wu_slots) * p.NB * BOX_BYTES);
  s.a_full = bars;
  s.a_empty = s.a_full + p.stages;
  s.w_full = s.a_empty + p.stages;
  s.w_empty = s.w_full + p.w_slots;
  s.wu_full = s.w_empty + p.w_slots;
  s.wu_empty = s.wu_full + p.wu_slots;
  s.wc_full = s.wu_empty + p.wu_slots;
  s.acc_full = s.wc_full + 1;
  s.acc_empty = s.acc_full + 2;
  s.pub = s.acc_empty + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.pub + 1);
  s.abort = s.tmem_slot + 1;
  s.range = reinterpret_cast<long long*>(s.abort + 1);
  return s;
}

// Units: user tiles (u, D block, 64-wide N block) first, then candidate
// tiles (i, D block) covering all of N.  User tiles are split along N so that
// the user phase, which every candidate epilogue waits for, is spread over
// more SMs and each of its tiles loads and writes a third as much.
struct UnitInfo {
  bool is_user;
  bool local;  // a user tile of the local-partial schedule: all of N, kept in this CTA
  int row;     // user u or candidate i
  int dblk;    // 128-row block of D
  int nblk;    // user tiles: 64-wide block of N
};

__device__ __forceinline__ UnitInfo unit_info(const LceParams& p, int unit) {
  UnitInfo x;
  x.is_user = unit < p.n_user_units;
  x.local = false;
  if (x.is_user) {
    x.nblk = unit % p.NB;
    const int ud = unit / p.NB;
    x.row = ud / p.n_dblk;
    x.dblk = ud - x.row * p.n_dblk;
  } else {
    const int idx = unit - p.n_user_units;
    const int pos = idx / p.n_dblk;  // position in the candidate order
    x.dblk = idx - pos * p.n_dblk;
    x.nblk = 0;
    const int i = p.order ? __ldg(p.order + pos) : pos;
    x.row = (i >= 0 && i < p.n_cand) ? i : pos;
  }
  return x;
}

// The t-th unit of this CTA within [u0, u1), or -1 past its end.  User tiles
// are dealt round-robin.  Candidate tiles, numbered D-block-major over the
// candidate order (q = dblk * n_cand + position), go out as one contiguous
// range of q per CTA: a CTA stays within one D block (crossing at most one
// boundary) on consecutive candidates that mostly share a user, so its
// epilogue loads that user's partial once and keeps it in registers.
//
// In the one-launch schedule (u0 == 0 and u1 == n_units) every CTA first
// computes its user tiles (round-robin), then its range of candidate tiles;
// while each CTA has at most one user tile, the ranges are weighted so that
// a CTA with one takes two candidate tiles fewer.
__device__ __forceinline__ long long fused_q_start(const LceParams& p, int b) {
  const int g = static_cast<int>(gridDim.x);
  const long long nq = static_cast<long long>(p.n_cand) * p.n_dblk;
  if (b >= g) return nq;
  const long long uu = p.n_user_units;
  long long w = uu <= g ? (2ll << 8) : 0;  // candidate tiles a user tile stands for, in 1/256
  long long tq = ((nq << 8) + w * uu) / g;
  if (tq < w) {  // too few candidate tiles to lighten anyone
    w = 0;
    tq = (nq << 8) / g;
  }
  const long long cum = (b * tq - w * (b < uu ? b : uu) + 128) >> 8;
  return cum < 0 ? 0 : (cum > nq ? nq : cum);
}

// The local-partial schedule weights its ranges: a CTA pays for one local user
// tile per (user, D block) its range touches, and with equal numbers of
// candidate tiles the CTAs whose range crosses a user boundary end last.  So
// the range boundaries split V(q) = c*q + h*(user runs starting before q)
// evenly, q counting candidate tiles D-block-major over the candidate order.
// c and h are the bytes a candidate tile streams from HBM (C in, Y out) and
// 0.8 x the bytes of a user tile (U and W_u, mostly L2 hits).  Within a D
// block, a position in (offsets[u], offsets[u + 1]] of a non-empty user u
// has runs[u + 1] run starts before it; warp 3 of every CTA evaluates the
// same function, so the ranges tile [0, nq).  The boundary search probes 32
// users per warp-wide load (one load for up to 32 users).  All lanes must
// call these.
struct RunProbe {
  int stride;          // users per lane in this round
  long long end, beg;  // the end (and, in the last round, the start) of the lane's user's run
  long long nr;        // non-empty runs up to and including that user
};

__device__ __forceinline__ RunProbe run_probe(const LceParams& p, int lo, int hi) {
  RunProbe r;
  r.stride = (hi - lo + 32) >> 5;
  const int u = min(lo + (static_cast<int>(lane_id()) + 1) * r.stride - 1, hi);
  // the last user's run ends at n_cand even if invalid map entries left
  // candidates out of the offsets (the plan flags those)
  r.end = u == p.n_users - 1 ? p.n_cand : __ldg(p.seg_offsets + u + 1);
  r.beg = r.stride == 1 ? __ldg(p.seg_offsets + u) : 0;
  r.nr = __ldg(p.seg_runs + u + 1);
  return r;
}

// the first q with V(q) >= T; r is the first round's probe (lo 0, hi n_users - 1)
__device__ __forceinline__ long long local_q_start(const LceParams& p, long long T, long long c, long long h,
                                                   long long vrow, long long vtot, long long nq, RunProbe r) {
  if (T <= 0) return 0;
  if (T >= vtot) return nq;
  const long long dblk = (T - 1) / vrow;  // dblk * vrow < T <= (dblk + 1) * vrow
  const long long R = T - dblk * vrow;
  // the first user whose run ends at V >= R (V at the last run's end is vrow)
  int lo = 0, hi = p.n_users - 1;
  for (;;) {
    const uint32_t ok = __ballot_sync(0xffffffffu, c * r.end + h * r.nr >= R);
    const int l = ok ? __ffs(ok) - 1 : 31;
    if (r.stride == 1) {
      const long long beg = __shfl_sync(0xffffffffu, r.beg, l);
      const long long nr = __shfl_sync(0xffffffffu, r.nr, l);
      const long long need = R - h * nr;
      long long pos = need <= 0 ? 1 : (need + c - 1) / c;
      if (pos < beg + 1) pos = beg + 1;
      return dblk * p.n_cand + (pos < p.n_cand ? pos : p.n_cand);
    }
    const int nlo = lo + l * r.stride;
    hi = min(nlo + r.stride - 1, hi);
    lo = nlo;
    r = run_probe(p, lo, hi);
  }
}

__device__ __forceinline__ void local_range(const LceParams& p, long long& q0, long long& q1) {
  const int g = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  const long long nq = static_cast<long long>(p.n_cand) * p.n_dblk;
  // with one user the even split already cuts at the D-block boundary
  if (p.seg_offsets == nullptr || p.seg_runs == nullptr || p.n_users < 2) {
    q0 = b * nq / g;
    q1 = (b + 1) * nq / g;
    return;
  }
  const RunProbe r = run_probe(p, 0, p.n_users - 1);
  const long long runs = __ldg(p.seg_runs + p.n_users);
  const long long c = 5ll * LCE_BM * (p.K_c + p.N);
  const long long h = 4ll * p.K_u * (LCE_BM + p.N);
  const long long vrow = c * p.n_cand + h * runs;
  const long long vtot = vrow * p.n_dblk;
  q0 = local_q_start(p, b * vtot / g, c, h, vrow, vtot, nq, r);
  q1 = local_q_start(p, (b + 1) * vtot / g, c, h, vrow, vtot, nq, r);
}

__device__ __forceinline__ int cta_unit(const LceParams& p, int u0, int u1, int t, long long lq0, long long lq1) {
  const int g = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
  const int uu = p.n_user_units;
  if (u0 == 0 && u1 == uu) {  // user launch
    const int unit = b + t * g;
    return unit < u1 ? unit : -1;
  }
  long long q0, q1;
  if (u0 == 0) {  // one launch: this CTA's user tiles first
    const int nu = uu > b ? (uu - b + g - 1) / g : 0;
    if (t < nu) return b + t * g;
    t -= nu;
    q0 = fused_q_start(p, b);
    q1 = fused_q_start(p, b + 1);
  } else if (lq0 >= 0) {  // local partials: the weighted range
    q0 = lq0;
    q1 = lq1;
  } else {  // candidate launch
    const long long nq = static_cast<long long>(p.n_cand) * p.n_dblk;
    q0 = b * nq / g;
    q1 = (b + 1) * nq / g;
  }
  if (t >= q1 - q0) return -1;
  const int q = static_cast<int>(q0 + t);
  const int dblk = q / p.n_cand;
  const int pos = q - dblk * p.n_cand;
  return uu + pos * p.n_dblk + dblk;
}

constexpr int LCE_PHASE_CAND = 0, LCE_PHASE_USER = 1, LCE_PHASE_BOTH = 2, LCE_PHASE_LOCAL = 3;

// The units a CTA runs, in order: its units of [u0, u1), and in the
// local-partial schedule, before a candidate tile whose (user, D block)
// differs from the previous one, a local user tile for that pair.  Every
// role walks the same sequence, a whole warp at a time: the lanes look up 32
// units at once (list position -> unit -> candidate -> user) and each step
// takes its unit from one lane, so the dependent global loads of a lookup --
// half a microsecond each while HBM streams -- are paid once per 32 units
// instead of on every tile's critical path.  All lanes must call walk_next.
struct Walk {
  int t = 0;      // next index in this CTA's list
  int t0 = -32;   // list index of lane 0's window entry
  int w_unit = -1, w_row = 0, w_dblk = 0, w_nblk = 0, w_user = -1;  // this lane's entry
  int cur_u = -1, cur_dblk = -1;
  bool held = false;
  UnitInfo next;
  int next_user = -1;
  long long q0 = -1, q1 = -1;  // the local schedule's range of candidate tiles
  const long long* range = nullptr;  // where warp 3 posts it (shared memory)
};

// The local schedule's range is computed once per CTA by warp 3 while the
// other warps start; the 11 warps that walk or post it meet on named barrier 1.
constexpr int LCE_RANGE_BAR = 1, LCE_RANGE_THREADS = 32 * 11;

template <int kPhase>
__device__ __forceinline__ bool walk_next(const LceParams& p, int u0, int u1, Walk& w, UnitInfo& x, int& user) {
  if (kPhase == LCE_PHASE_LOCAL && w.held) {
    x = w.next;
    user = w.next_user;
    w.held = false;
    return true;
  }
  if (w.t - w.t0 >= 32) {
    if (kPhase == LCE_PHASE_LOCAL && w.q0 < 0) {
      named_barrier_sync(LCE_RANGE_BAR, LCE_RANGE_THREADS);
      w.q0 = w.range[0];
      w.q1 = w.range[1];
    }
    w.t0 = w.t;
    w.w_unit = cta_unit(p, u0, u1, w.t0 + static_cast<int>(lane_id()), w.q0, w.q1);
    if (w.w_unit >= 0) {
      const UnitInfo y = unit_info(p, w.w_unit);
      w.w_row = y.row;
      w.w_dblk = y.dblk;
      w.w_nblk = y.nblk;
      w.w_user = y.is_user ? y.row : __ldg(p.map + y.row);
    }
  }
  const int k = w.t - w.t0;
  const int unit = __shfl_sync(0xffffffffu, w.w_unit, k);
  if (unit < 0) return false;
  ++w.t;
  x.is_user = unit < p.n_user_units;
  x.local = false;
  x.row = __shfl_sync(0xffffffffu, w.w_row, k);
  x.dblk = __shfl_sync(0xffffffffu, w.w_dblk, k);
  x.nblk = __shfl_sync(0xffffffffu, w.w_nblk, k);
  user = __shfl_sync(0xffffffffu, w.w_user, k);
  if (kPhase == LCE_PHASE_LOCAL && user >= 0 && user < p.n_users && (user != w.cur_u || x.dblk != w.cur_dblk)) {
    w.cur_u = user;
    w.cur_dblk = x.dblk;
    w.next = x;
    w.next_user = user;
    w.held = true;
    x.is_user = true;
    x.local = true;
    x.row = user;
    x.nblk = 0;
  }
  return true;
}

// columns of a user tile's accumulator (a multiple of 16, at most 64)
__device__ __forceinline__ int user_tile_n(const LceParams& p, int nblk) { return min(64, p.N_mma - nblk * 64); }

// ------------------------------------------------------------ producer
// A wait taken by a whole warp: every lane polls, and the lanes agree on the
// outcome so that a timeout never splits the warp.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const LceSmem& s, const LceParams& p) {
  const bool ok = mbar_wait(bar, parity, s.abort, p.timeout_ns, 1);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void load_wc(const LceParams& p, const LceSmem& s, const CUtensorMap* tmWc) {
  mbar_arrive_expect_tx(s.wc_full, static_cast<uint32_t>(p.kc_c * p.NB) * BOX_BYTES);
  for (int kc = 0; kc < p.kc_c; ++kc)
    for (int nb = 0; nb < p.NB; ++nb)
      tma_load_2d(s.w_region + (static_cast<size_t>(kc) * p.NB + nb) * BOX_BYTES, tmWc, s.wc_full, nb * 64,
                  kc * LCE_BK);
}

// TMA producer: the whole warp runs the loop and waits; one elected lane
// issues the copies.
template <int kPhase>
__device__ void lce_producer(const LceParams& p, const LceSmem& s, const CUtensorMap* tmU, const CUtensorMap* tmC,
                             const CUtensorMap* tmWu, const CUtensorMap* tmWc, int u0, int u1) {
  int stage = 0;
  uint32_t a_phase = 0;
  int wslot = 0;
  uint32_t w_phase = 0;
  uint32_t w_uses[LCE_MAX_W_SLOTS] = {0, 0, 0, 0, 0, 0, 0, 0};
  int uslot = 0;
  uint32_t u_phase = 0;
  bool wc_loaded = false;
  const uint32_t w_chunk_bytes = static_cast<uint32_t>(p.NB) * BOX_BYTES;
  if (kPhase == LCE_PHASE_LOCAL) {  // no user tile uses the W region: W_c lands at once
    if (elect_one()) load_wc(p, s, tmWc);
    __syncwarp();
    wc_loaded = true;
  }

  Walk walk;
  walk.range = s.range;
  for (;;) {
    UnitInfo x;
    int user;
    if (!walk_next<kPhase>(p, u0, u1, walk, x, user)) break;
    const CUtensorMap* tmA = x.is_user ? tmU : tmC;
    const int kc_n = x.is_user ? p.kc_u : p.kc_c;
    const int d0 = x.dblk * LCE_BM;
    if (!x.is_user && !wc_loaded) {
      // every W slot used by the user phase must be drained before Wc lands
      for (int w = 0; w < p.w_slots; ++w)
        if (w_uses[w] > 0 && !warp_wait(&s.w_empty[w], (w_uses[w] - 1) & 1u, s, p)) return;
      if (elect_one()) load_wc(p, s, tmWc);
      __syncwarp();
      wc_loaded = true;
    }
    for (int kc = 0; kc < kc_n; ++kc) {
      if (!warp_wait(&s.a_empty[stage], a_phase ^ 1u, s, p)) return;
      const bool wu_ring = kPhase == LCE_PHASE_LOCAL && x.local;  // all NB boxes of this K chunk of W_u
      if (wu_ring && !warp_wait(&s.wu_empty[uslot], u_phase ^ 1u, s, p)) return;
      if (!wu_ring && x.is_user && !warp_wait(&s.w_empty[wslot], w_phase ^ 1u, s, p)) return;
      if (elect_one()) {
        uint8_t* dst = s.a_ring + static_cast<size_t>(stage) * LCE_A_STAGE_BYTES;
        mbar_arrive_expect_tx(&s.a_full[stage], LCE_A_STAGE_BYTES);
        tma_load_3d(dst, tmA, &s.a_full[stage], d0, kc * LCE_BK, x.row);
        tma_load_3d(dst + BOX_BYTES, tmA, &s.a_full[stage], d0 + 64, kc * LCE_BK, x.row);
        if (wu_ring) {
          uint8_t* wdst = s.wu_ring + static_cast<size_t>(uslot) * w_chunk_bytes;
          mbar_arrive_expect_tx(&s.wu_full[uslot], w_chunk_bytes);
          for (int nb = 0; nb < p.NB; ++nb)
            tma_load_2d(wdst + static_cast<size_t>(nb) * BOX_BYTES, tmWu, &s.wu_full[uslot], nb * 64, kc * LCE_BK);
        } else if (x.is_user) {
          mbar_arrive_expect_tx(&s.w_full[wslot], BOX_BYTES);
          tma_load_2d(s.w_region + static_cast<size_t>(wslot) * BOX_BYTES, tmWu, &s.w_full[wslot], x.nblk * 64,
                      kc * LCE_BK);
        }
      }
      __syncwarp();
      if (wu_ring) {
        if (++uslot == p.wu_slots) {
          uslot = 0;
          u_phase ^= 1u;
        }
      } else if (x.is_user) {
        w_uses[wslot] += 1;
        if (++wslot == p.w_slots) {
          wslot = 0;
          w_phase ^= 1u;
        }
      }
      if (++stage == p.stages) {
        stage = 0;
        a_phase ^= 1u;
      }
    }
  }
}

// ----------------------------------------------------------------- MMA
// MMA issuer: the whole warp runs the loop (its values stay warp-uniform) and
// one elected lane issues; a lone lane pays far more per tcgen05.mma.
template <int kPhase>
__device__ void lce_mma(const LceParams& p, const LceSmem& s, uint32_t tmem, int u0, int u1) {
  const uint32_t idesc_c = idesc_bf16_f32(LCE_BM, static_cast<uint32_t>(p.N_mma), true, true);
  const uint32_t w_chunk_bytes = static_cast<uint32_t>(p.NB) * BOX_BYTES;
  int stage = 0;
  uint32_t a_phase = 0;
  int wslot = 0;
  uint32_t w_phase = 0;
  int uslot = 0;
  uint32_t u_phase = 0;
  bool wc_ready = false;
  Walk walk;
  walk.range = s.range;
  for (int local = 0;; ++local) {
    UnitInfo x;
    int user;
    if (!walk_next<kPhase>(p, u0, u1, walk, x, user)) break;
    const bool wu_ring = kPhase == LCE_PHASE_LOCAL && x.local;  // W_u from the full-width ring
    const int kc_n = x.is_user ? p.kc_u : p.kc_c;
    int ks_left = x.is_user ? p.ks_u : p.ks_c;
    const bool one_acc = p.mode & LCE_MODE_ONE_ACC;
    const int buf = one_acc ? 0 : (local & 1);
    const uint32_t use = static_cast<uint32_t>(one_acc ? local : (local >> 1));
    if (!warp_wait(&s.acc_empty[buf], (use & 1u) ^ 1u, s, p)) return;
    if (!x.is_user && !wc_ready) {
      if (!warp_wait(s.wc_full, 0, s, p)) return;
      wc_ready = true;
    }
    tc_fence_after();
    const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf) * 256u;
    const uint32_t idesc = (x.is_user && !wu_ring)
                               ? idesc_bf16_f32(LCE_BM, static_cast<uint32_t>(user_tile_n(p, x.nblk)), true, true)
                               : idesc_c;
    for (int kc = 0; kc < kc_n; ++kc) {
      if (!warp_wait(&s.a_full[stage], a_phase, s, p)) return;
      if (wu_ring) {
        if (!warp_wait(&s.wu_full[uslot], u_phase, s, p)) return;
      } else if (x.is_user && !warp_wait(&s.w_full[wslot], w_phase, s, p)) {
        return;
      }
      tc_fence_after();
      const uint32_t a_base = smem_u32(s.a_ring + static_cast<size_t>(stage) * LCE_A_STAGE_BYTES);
      const uint32_t b_base =
          wu_ring ? smem_u32(s.wu_ring + static_cast<size_t>(uslot) * w_chunk_bytes)
                  : smem_u32(s.w_region + (x.is_user ? static_cast<size_t>(wslot) * BOX_BYTES
                                                     : static_cast<size_t>(kc) * w_chunk_bytes));
      const int nsteps = ks_left < 4 ? ks_left : 4;
      // 16 k rows of 128 bytes per MMA step; 64-element blocks along M / N
      // are one box apart; steps advance the start address by 2048 bytes
      const uint64_t adesc = sdesc_sw128(a_base, BOX_BYTES, 1024u);
      const uint64_t bdesc = sdesc_sw128(b_base, BOX_BYTES, 1024u);
      const uint32_t acc0 = kc > 0 ? 1u : 0u;
      if (elect_one()) {
        if (nsteps == 4) {
#pragma unroll
          for (int st = 0; st < 4; ++st)
            mma_bf16_ss(d_tmem, adesc + st * (2048u >> 4), bdesc + st * (2048u >> 4), idesc, st > 0 ? 1u : acc0);
        } else {
          for (int st = 0; st < nsteps; ++st)
            mma_bf16_ss(d_tmem, adesc + st * (2048u >> 4), bdesc + st * (2048u >> 4), idesc, st > 0 ? 1u : acc0);
        }
        mma_commit(&s.a_empty[stage]);
        if (wu_ring)
          mma_commit(&s.wu_empty[uslot]);
        else if (x.is_user)
          mma_commit(&s.w_empty[wslot]);
      }
      __syncwarp();
      ks_left -= nsteps;
      if (wu_ring) {
        if (++uslot == p.wu_slots) {
          uslot = 0;
          u_phase ^= 1u;
        }
      } else if (x.is_user) {
        if (++wslot == p.w_slots) {
          wslot = 0;
          w_phase ^= 1u;
        }
      }
      if (++stage == p.stages) {
        stage = 0;
        a_phase ^= 1u;
      }
    }
    if (elect_one()) mma_commit(&s.acc_full[buf]);
    __syncwarp();
  }
}

// Wait until every user tile of this launch has published its partial
// (flags[k] == epoch for all k).  The lanes of the warp poll the flags in
// parallel, so when they are already set (the user kernel ran first on the
// stream) this costs one round trip per warp and launch.  Gives up after
// timeout_ns, or at once if another wait of this launch already gave up.
__device__ __forceinline__ bool wait_all_user_partials(const LceParams& p) {
  const int nflags = p.n_user_units;
  const uint64_t t0 = globaltimer_ns();
  for (int base = 0; base < nflags; base += 32) {
    const int k = base + static_cast<int>(lane_id());
    for (;;) {
      const bool mine = k >= nflags || ld_acquire_gpu(p.flags + k) == p.epoch;
      if (__all_sync(0xffffffffu, mine)) break;
      int give_up = 0;
      if (lane_id() == 0) {
        if (ld_volatile_u32(p.timeout_epoch) == p.epoch) {
          give_up = 1;
        } else if (globaltimer_ns() - t0 > p.timeout_ns) {
          atomicOr(p.status, DEV_ERR_FLAG_TIMEOUT);
          atomicExch(p.timeout_epoch, p.epoch);
          give_up = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, give_up, 0)) return false;
      __nanosleep(256);
    }
  }
  return true;
}

// The user partial P[u][n][d] = b[n] + sum_k Wu[k][n] U[u][k][d] for the 32
// columns n0 .. n0+31 of row d, on the CUDA cores (fp32, ascending k).  Only
// for candidate tiles whose user tiles never published within the wait
// bound: the tile then still writes its Y, from this slower copy of the
// partial (another summation order than the tensor cores', same inputs).
__device__ __noinline__ void user_partial_cuda_cores(const LceParams& p, int u, int d, int n0, float* out) {
#pragma unroll 1
  for (int j = 0; j < 32; ++j) {
    const int n = n0 + j;
    out[j] = (p.bias && n < p.N) ? __bfloat162float(__ushort_as_bfloat16(__ldg(p.bias + n))) : 0.f;
  }
  if (d >= p.D) return;
  const uint16_t* ur = p.U + static_cast<size_t>(u) * p.K_u * p.D + d;
#pragma unroll 1
  for (int k = 0; k < p.K_u; ++k) {
    const float a = __bfloat162float(__ushort_as_bfloat16(__ldg(ur + static_cast<size_t>(k) * p.D)));
    const uint16_t* w = p.Wu + static_cast<size_t>(k) * p.N + n0;
#pragma unroll 4
    for (int j = 0; j < 32; ++j)
      if (n0 + j < p.N) out[j] = fmaf(__bfloat162float(__ushort_as_bfloat16(__ldg(w + j))), a, out[j]);
  }
}

// ------------------------------------------------------------ epilogue
// Eight warps: warp w reads TMEM lane quarter w % 4 (rows 32*(w%4) .. +31 of
// the D block) and every other 32-column chunk, starting at (w - 4) / 4.
// Candidate tiles fetch their P[map[i]] chunks before waiting for the
// accumulator, so the L2 latency of that gather hides behind the MMA.
constexpr int EPI_PREFETCH = 3;  // chunks of P held in registers ahead of the accumulator

template <int kPhase>
__device__ void lce_epilogue(const LceParams& p, const LceSmem& s, uint32_t tmem, int u0, int u1) {
  const int warp = threadIdx.x >> 5;
  const int quarter = warp & 3;
  const int half = (warp - LCE_EPI_WARP0) >> 2;
  const int et = quarter * 32 + static_cast<int>(lane_id());  // TMEM lane = row of the D block
  const bool leader = warp == LCE_EPI_WARP0 && lane_id() == 0;
  const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
  const int nchunks = (p.N + 31) / 32;
  int local = 0;
  uint32_t pubs = 0;
  int users_ready = -1;  // candidate tiles: -1 not checked yet, 1 all user partials seen, 0 gave up
  // the user partial of the current (user, D block), kept across tiles
  float pre[EPI_PREFETCH][32];
  int pre_u = -1, pre_dblk = -1;
  Walk walk;
  walk.range = s.range;
  for (;; ++local) {
    UnitInfo x;
    int user;  // candidate tiles: map[i] (the warp's lanes looked it up together)
    if (!walk_next<kPhase>(p, u0, u1, walk, x, user)) break;
    const bool one_acc = p.mode & LCE_MODE_ONE_ACC;
    const int buf = one_acc ? 0 : (local & 1);
    const uint32_t use = static_cast<uint32_t>(one_acc ? local : (local >> 1));
    const int d = x.dblk * LCE_BM + et;
    const bool dok = d < p.D;
    const size_t ND = static_cast<size_t>(p.N) * p.D;
    const uint32_t t_acc = tmem + lane_base + static_cast<uint32_t>(buf) * 256u;
    if (kPhase == LCE_PHASE_LOCAL && x.local) {
      // this CTA's own partial of (user, D block): accumulator + b -> registers;
      // b is loaded before the wait, so its latency hides behind the MMA
#pragma unroll
      for (int k = 0; k < EPI_PREFETCH; ++k) {
        const int c = half + 2 * k;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int n = c * 32 + j;
          pre[k][j] = (p.bias && n < p.N) ? __bfloat162float(__ushort_as_bfloat16(__ldg(p.bias + n))) : 0.f;
        }
      }
      if (!warp_wait(&s.acc_full[buf], use & 1u, s, p)) return;
      tc_fence_after();
#pragma unroll
      for (int k = 0; k < EPI_PREFETCH; ++k) {
        const int c = half + 2 * k;
        if (c < nchunks) {
          uint32_t v[32];
          tmem_ld32(t_acc + c * 32, v);
          tmem_ld_wait(v);
#pragma unroll
          for (int j = 0; j < 32; ++j) pre[k][j] += __uint_as_float(v[j]);
        }
      }
      tc_fence_before();
      mbar_arrive(&s.acc_empty[buf]);
      pre_u = x.row;
      pre_dblk = x.dblk;
    } else if (x.is_user) {
      // this tile holds columns n0 .. n0 + nw - 1 of P
      const int n0 = x.nblk * 64;
      const int nw = user_tile_n(p, x.nblk);
      if (!warp_wait(&s.acc_full[buf], use & 1u, s, p)) return;
      tc_fence_after();
      float* P = p.partial + static_cast<size_t>(x.row) * ND + d;
      for (int c = half; c * 32 < nw; c += 2) {
        // the bias of this chunk, loaded before any store (the stores could
        // otherwise alias it and serialise every load behind them)
        float bias[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int n = n0 + c * 32 + j;
          bias[j] = (p.bias && n < p.N) ? __bfloat162float(__ushort_as_bfloat16(__ldg(p.bias + n))) : 0.f;
        }
        uint32_t v[32];
        tmem_ld32(t_acc + c * 32, v);
        tmem_ld_wait(v);
        float* pp = P + static_cast<size_t>(n0 + c * 32) * p.D;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (n0 + c * 32 + j < p.N && dok) __stcg(pp, __uint_as_float(v[j]) + bias[j]);
          pp += p.D;
        }
      }
      tc_fence_before();
      mbar_arrive(&s.acc_empty[buf]);
      // publish: the writers arrive on an mbarrier (release at CTA scope), and
      // the one thread that has seen all of them arrive fences and releases
      // the flag at GPU scope, which covers their stores (cumulativity)
      mbar_arrive(s.pub);
      if (leader) {
        const bool all = mbar_wait(s.pub, pubs & 1u, s.abort, p.timeout_ns, 1);
        if (all && !(p.debug & DEBUG_WITHHOLD_USER_PARTIAL)) {
          __threadfence();
          st_release_gpu(p.flags + (x.row * p.n_dblk + x.dblk) * p.NB + x.nblk, p.epoch);
        }
      }
      ++pubs;
    } else {
      const int i = x.row;
      const bool add_p = !(p.mode & LCE_MODE_NO_PARTIAL);
      const int u = add_p ? user : 0;
      const bool uok = u >= 0 && u < p.n_users;
      if (!uok && leader) atomicOr(p.status, DEV_ERR_MAP_RANGE);
      if (kPhase != LCE_PHASE_LOCAL && add_p && users_ready < 0) users_ready = wait_all_user_partials(p) ? 1 : 0;
      // the partials never came (the wait ran out): this CTA forms them itself
      const bool fallback = kPhase != LCE_PHASE_LOCAL && add_p && users_ready == 0;
      // local partials: the walk put this (user, D block)'s own tile just before
      bool ready = uok && (kPhase == LCE_PHASE_LOCAL || !add_p || users_ready == 1 || fallback);
      if (kPhase == LCE_PHASE_LOCAL && ready && (pre_u != u || pre_dblk != x.dblk)) {
        if (leader) atomicOr(p.status, DEV_ERR_BAD_WORK);
        ready = false;
      }
      const float* P = p.partial + static_cast<size_t>(uok ? u : 0) * ND + d;
      if (!add_p && pre_u != -2) {  // decomposed stage: no partial here (a later launch adds it)
        pre_u = -2;
#pragma unroll
        for (int k = 0; k < EPI_PREFETCH; ++k)
#pragma unroll
          for (int j = 0; j < 32; ++j) pre[k][j] = 0.f;
      }
      if (kPhase != LCE_PHASE_LOCAL && add_p && ready && (u != pre_u || x.dblk != pre_dblk)) {
        pre_u = u;
        pre_dblk = x.dblk;
#pragma unroll
        for (int k = 0; k < EPI_PREFETCH; ++k) {
          const int c = half + 2 * k;
          if (fallback) {
            float t[32];
            if (c < nchunks) user_partial_cuda_cores(p, u, d, c * 32, t);
#pragma unroll
            for (int j = 0; j < 32; ++j) pre[k][j] = (c * 32 + j < p.N && dok) ? t[j] : 0.f;
            continue;
          }
          const float* pp = P + static_cast<size_t>(c * 32) * p.D;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            pre[k][j] = (c * 32 + j < p.N && dok) ? __ldcg(pp) : 0.f;
            pp += p.D;
          }
        }
      }
      if (!warp_wait(&s.acc_full[buf], use & 1u, s, p)) return;
      tc_fence_after();
      if (ready) {
        __nv_bfloat16* Y = reinterpret_cast<__nv_bfloat16*>(p.Y) + static_cast<size_t>(i) * ND + d;
#pragma unroll
        for (int k = 0; k < EPI_PREFETCH; ++k) {
          const int c = half + 2 * k;
          if (c >= nchunks) break;
          uint32_t v[32];
          tmem_ld32(t_acc + c * 32, v);
          tmem_ld_wait(v);
          __nv_bfloat16* y = Y + static_cast<size_t>(c * 32) * p.D;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c * 32 + j < p.N && dok) *y = __float2bfloat16_rn(__uint_as_float(v[j]) + pre[k][j]);
            y += p.D;
          }
        }
        for (int c = half + 2 * EPI_PREFETCH; kPhase != LCE_PHASE_LOCAL && c < nchunks; c += 2) {  // N > 192
          uint32_t v[32];
          tmem_ld32(t_acc + c * 32, v);
          float pu[32];
          const float* pp = P + static_cast<size_t>(c * 32) * p.D;
          if (fallback) {
            float t[32];
            user_partial_cuda_cores(p, u, d, c * 32, t);
#pragma unroll
            for (int j = 0; j < 32; ++j) pu[j] = t[j];
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              pu[j] = (add_p && c * 32 + j < p.N && dok) ? __ldcg(pp + static_cast<size_t>(j) * p.D) : 0.f;
          }
          tmem_ld_wait(v);
          __nv_bfloat16* y = Y + static_cast<size_t>(c * 32) * p.D;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c * 32 + j < p.N && dok) *y = __float2bfloat16_rn(__uint_as_float(v[j]) + pu[j]);
            y += p.D;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s.acc_empty[buf]);
    }
  }
}

// One body, launched either as two kernels -- kPhase LCE_PHASE_USER computes
// the user tiles (P and their release flags), then LCE_PHASE_CAND the
// candidate tiles, which acquire the flags and add P in their epilogue -- or
// as one (LCE_PHASE_BOTH: user tiles first in every CTA's list;
// LCE_PHASE_LOCAL: candidate tiles with each CTA's own user partials).  The grid
// never exceeds the SM count and takes one CTA per SM.  LCE_PHASE_BOTH is
// launched cooperatively, so its CTAs are resident together and a flag wait
// ends once the user tiles are done; LCE_PHASE_CAND waits only for flags of
// the launch before it.  A wait that still runs out (the debug switch that
// withholds the partials) is reported, and the waiting tiles form the
// partial on the CUDA cores instead.
template <int kPhase>
__global__ void __launch_bounds__(LCE_THREADS, 1)
    lce_kernel(const __grid_constant__ CUtensorMap tmU, const __grid_constant__ CUtensorMap tmC,
               const __grid_constant__ CUtensorMap tmWu, const __grid_constant__ CUtensorMap tmWc,
               const LceParams p) {
  const int u0 = (kPhase == LCE_PHASE_CAND || kPhase == LCE_PHASE_LOCAL) ? p.n_user_units : 0;
  const int u1 = kPhase == LCE_PHASE_USER ? p.n_user_units : p.n_units;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const LceSmem s = carve(base, p);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&s.a_full[i], 1);
      mbar_init(&s.a_empty[i], 1);
    }
    for (int i = 0; i < p.w_slots; ++i) {
      mbar_init(&s.w_full[i], 1);
      mbar_init(&s.w_empty[i], 1);
    }
    for (int i = 0; i < p.wu_slots; ++i) {
      mbar_init(&s.wu_full[i], 1);
      mbar_init(&s.wu_empty[i], 1);
    }
    mbar_init(s.wc_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], LCE_EPI_THREADS);
    }
    mbar_init(s.pub, LCE_EPI_THREADS);
    *s.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmU);
    tma_prefetch_desc(&tmC);
    tma_prefetch_desc(&tmWu);
    tma_prefetch_desc(&tmWc);
  }
  if (warp == 2) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;

  // registers: launched at 168 per thread (384 x 168 = 64512); the control
  // warpgroup gives back down to 72 and the two epilogue warpgroups take 216
  // (128 x 72 + 256 x 216 = 64512)
  if (warp < LCE_EPI_WARP0) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 72;");
    if (warp == 0) {
      lce_producer<kPhase>(p, s, &tmU, &tmC, &tmWu, &tmWc, u0, u1);
    } else if (warp == 1) {
      lce_mma<kPhase>(p, s, tmem, u0, u1);
    } else if (warp == 3 && kPhase == LCE_PHASE_LOCAL) {
      long long q0, q1;
      local_range(p, q0, q1);
      if (lane_id() == 0) {
        s.range[0] = q0;
        s.range[1] = q1;
      }
      named_barrier_arrive(LCE_RANGE_BAR, LCE_RANGE_THREADS);
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 216;");
    lce_epilogue<kPhase>(p, s, tmem, u0, u1);
  }

  tc_fence_before();
  __syncthreads();
  if (*s.abort && threadIdx.x == 0) atomicOr(p.status, DEV_ERR_PIPE_TIMEOUT);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // The launch that reads the readiness flags returns them (and the timeout
  // word) to zero for the next call: the last of its CTAs to finish, after
  // every other CTA has stopped reading them, clears them.
  if (kPhase == LCE_PHASE_CAND || kPhase == LCE_PHASE_BOTH) {
    __shared__ uint32_t last_cta;
    if (threadIdx.x == 0) {
      __threadfence();
      last_cta = atomicAdd(p.done, 1u) == gridDim.x - 1 ? 1u : 0u;
    }
    __syncthreads();
    if (last_cta) {
      __threadfence();
      for (int k = static_cast<int>(threadIdx.x); k < p.n_user_units; k += static_cast<int>(blockDim.x))
        p.flags[k] = 0;
      if (threadIdx.x == 0) {
        *p.timeout_epoch = 0;
        *p.done = 0;
      }
    }
  }
}

}  // namespace

bool lce_configure(LceParams* lp, size_t max_smem) {
  if (lp->K_u < 1 || lp->K_c < 1 || lp->D < 1 || lp->N < 1 || lp->n_users < 1 || lp->n_cand < 1) return false;
  if (lp->D % 8 != 0 || lp->N % 8 != 0 || lp->N > 256) return false;
  lp->N_mma = (lp->N + 15) / 16 * 16;
  lp->NB = (lp->N_mma + 63) / 64;
  lp->n_dblk = (lp->D + LCE_BM - 1) / LCE_BM;
  lp->n_user_units = lp->n_users * lp->n_dblk * lp->NB;
  lp->n_units = lp->n_user_units + lp->n_cand * lp->n_dblk;
  lp->kc_u = (lp->K_u + LCE_BK - 1) / LCE_BK;
  lp->kc_c = (lp->K_c + LCE_BK - 1) / LCE_BK;
  lp->ks_u = (lp->K_u + 15) / 16;
  lp->ks_c = (lp->K_c + 15) / 16;
  const int wc_boxes = lp->kc_c * lp->NB;  // W_c stays resident: one 8 KB box per (K chunk, N block)
  if (wc_boxes > 16) return false;
  const int region_boxes = wc_boxes < 2 ? 2 : wc_boxes;
  lp->w_region_bytes = static_cast<uint32_t>(region_boxes) * BOX_BYTES;
  lp->w_slots = region_boxes < LCE_MAX_W_SLOTS ? region_boxes : LCE_MAX_W_SLOTS;
  lp->wu_slots = 0;
  lp->stages = LCE_MAX_STAGES;
  while (lp->stages > 2 && lce_smem_bytes(*lp) > max_smem) --lp->stages;
  if (lce_smem_bytes(*lp) > max_smem) return false;
  // the local-partial schedule: a W_u ring after the A ring, which gives up
  // stages for it (the candidate stream runs as fast on 4 stages as on 8)
  lp->stages_local = 0;
  if (lp->N <= LCE_LOCAL_MAX_N) {
    LceParams q = *lp;
    q.wu_slots = LCE_WU_SLOTS;
    q.stages = LCE_MAX_STAGES;
    while (q.stages > 2 && lce_smem_bytes(q) > max_smem) --q.stages;
    if (lce_smem_bytes(q) <= max_smem) lp->stages_local = q.stages;
  }
  return true;
}

size_t lce_flag_count(const LceParams& lp) {
  return static_cast<size_t>(lp.n_users) * lp.n_dblk * lp.NB;
}

size_t lce_smem_bytes(const LceParams& p) {
  const size_t bars =
      sizeof(uint64_t) * (2 * p.stages + 2 * p.w_slots + 2 * p.wu_slots + 1 + 4 + 1) + 2 * sizeof(uint32_t) +
      2 * sizeof(long long);
  return 1024 + p.w_region_bytes + static_cast<size_t>(p.stages) * LCE_A_STAGE_BYTES +
         static_cast<size_t>(p.wu_slots) * p.NB * BOX_BYTES + bars;
}

// `cooperative`: launched so that all CTAs are resident at once, or not at
// all (cudaErrorCooperativeLaunchTooLarge, e.g. when fewer SMs are available
// to this context than the device has): required by the one-launch
// schedule, whose candidate tiles wait for user tiles of other CTAs.
template <int kPhase>
cudaError_t launch_phase(const CUtensorMap& tmU, const CUtensorMap& tmC, const CUtensorMap& tmWu,
                         const CUtensorMap& tmWc, const LceParams& p, int units, int num_sms, cudaStream_t s,
                         bool cooperative = false) {
  if (units <= 0) return cudaSuccess;
  const size_t smem = lce_smem_bytes(p);
  cudaError_t e = cudaFuncSetAttribute(lce_kernel<kPhase>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int grid = units < num_sms ? units : num_sms;
  if (!cooperative) {
    lce_kernel<kPhase><<<grid, LCE_THREADS, smem, s>>>(tmU, tmC, tmWu, tmWc, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(LCE_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lce_kernel<kPhase>, tmU, tmC, tmWu, tmWc, p);
}

int lce_resolve_schedule(const LceParams& p, int num_sms) {
  // local partials need the candidates grouped by user (the plan's order):
  // in map order a CTA's range could change user at every tile
  const bool local_ok = p.stages_local >= 2 && p.mode == 0 && p.order != nullptr;
  if (p.schedule == LCE_SCHEDULE_TWO || p.schedule == LCE_SCHEDULE_ONE) return p.schedule;
  if (p.schedule == LCE_SCHEDULE_LOCAL && local_ok) return LCE_SCHEDULE_LOCAL;
  // local partials wherever they apply: also with a single user, where every
  // CTA then repeats the same user tiles but needs no wait on another CTA
  // (measured 28.7 / 54.3 / 159.8 us against 32.8 / 55.3 / 161.8 for the
  // cooperative one-launch schedule at 256 / 1024 / 4096 candidates)
  if (local_ok) return LCE_SCHEDULE_LOCAL;
  if (p.n_users == 1) return LCE_SCHEDULE_ONE;
  // Plan-time choice (measured over the n_cand x ratio sweep): with few
  // candidate tiles per SM, one launch hides the user tiles under the
  // candidate tiles' start-up; with many, two launches keep every
  // candidate epilogue from waiting on user tiles still running elsewhere.
  const long long cand_tiles = static_cast<long long>(p.n_cand) * p.n_dblk;
  return cand_tiles < static_cast<long long>(LCE_ONE_LAUNCH_TILES_PER_SM) * num_sms ? LCE_SCHEDULE_ONE
                                                                                    : LCE_SCHEDULE_TWO;
}

// The user tiles and the candidate tiles: two launches on one stream, or one
// (see lce_resolve_schedule).  *launches receives the number of launches.
cudaError_t launch_lce(const CUtensorMap& tmU, const CUtensorMap& tmC, const CUtensorMap& tmWu,
                       const CUtensorMap& tmWc, const LceParams& p, int num_sms, cudaStream_t s, int* launches) {
  const int schedule = lce_resolve_schedule(p, num_sms);
  if (schedule == LCE_SCHEDULE_LOCAL) {
    LceParams q = p;
    q.stages = p.stages_local;
    q.wu_slots = LCE_WU_SLOTS;
    *launches = 1;
    return launch_phase<LCE_PHASE_LOCAL>(tmU, tmC, tmWu, tmWc, q, p.n_units - p.n_user_units, num_sms, s);
  }
  if (schedule == LCE_SCHEDULE_ONE) {
    *launches = 1;
    const cudaError_t e = launch_phase<LCE_PHASE_BOTH>(tmU, tmC, tmWu, tmWc, p, p.n_units, num_sms, s, true);
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    (void)cudaGetLastError();  // not all CTAs could be resident: two launches need no co-residency
  }
  *launches = 2;
  cudaError_t e = launch_phase<LCE_PHASE_USER>(tmU, tmC, tmWu, tmWc, p, p.n_user_units, num_sms, s);
  if (e != cudaSuccess) return e;
  return launch_phase<LCE_PHASE_CAND>(tmU, tmC, tmWu, tmWc, p, p.n_units - p.n_user_units, num_sms, s);
}

namespace {
// The decomposed stage's separate broadcast add: Y[i] = bf16(Y[i] + P[map[i]]),
// 8 elements (16 bytes of Y, 32 of P) per thread and step; D % 8 == 0.
__global__ void __launch_bounds__(256) lce_broadcast_add_kernel(const int32_t* map, const float* P, uint16_t* Y,
                                                               int n_cand, int n_users, int N, int D,
                                                               uint32_t* status) {
  const size_t nd8 = static_cast<size_t>(N) * D / 8;
  const size_t total = static_cast<size_t>(n_cand) * nd8;
  for (size_t t = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; t < total;
       t += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(t / nd8);
    const size_t e = t - static_cast<size_t>(i) * nd8;
    const int u = __ldg(map + i);
    if (u < 0 || u >= n_users) {
      if (e == 0) atomicOr(status, DEV_ERR_MAP_RANGE);
      continue;
    }
    uint4* yp = reinterpret_cast<uint4*>(Y) + t;
    const float4* pp = reinterpret_cast<const float4*>(P + (static_cast<size_t>(u) * nd8 + e) * 8);
    const uint4 y = *yp;
    const float4 a = __ldg(pp), b = __ldg(pp + 1);
    uint4 o;
    o.x = pack_bf16x2(__uint_as_float(y.x << 16) + a.x, __uint_as_float(y.x & 0xffff0000u) + a.y);
    o.y = pack_bf16x2(__uint_as_float(y.y << 16) + a.z, __uint_as_float(y.y & 0xffff0000u) + a.w);
    o.z = pack_bf16x2(__uint_as_float(y.z << 16) + b.x, __uint_as_float(y.z & 0xffff0000u) + b.y);
    o.w = pack_bf16x2(__uint_as_float(y.w << 16) + b.z, __uint_as_float(y.w & 0xffff0000u) + b.w);
    *yp = o;
  }
}
}  // namespace

// The pages' LCE stage ladder rebuilt from this kernel (see LCE_MODE_*):
// stage 1 decomposed and unfused (user tiles; candidate tiles without the
// partial; broadcast-add launch), stage 3 fused epilogue with one
// accumulator, stage 4 the full kernel.  Returns the number of launches in
// *launches.
cudaError_t launch_lce_stage(const CUtensorMap& tmU, const CUtensorMap& tmC, const CUtensorMap& tmWu,
                             const CUtensorMap& tmWc, LceParams p, int stage, int num_sms, cudaStream_t s,
                             int* launches) {
  *launches = 0;
  if (stage == 4) return launch_lce(tmU, tmC, tmWu, tmWc, p, num_sms, s, launches);
  p.mode = stage == 1 ? LCE_MODE_NO_PARTIAL : LCE_MODE_ONE_ACC;
  cudaError_t e = launch_lce(tmU, tmC, tmWu, tmWc, p, num_sms, s, launches);
  if (e != cudaSuccess) return e;
  if (stage == 1) {
    lce_broadcast_add_kernel<<<num_sms * 4, 256, 0, s>>>(p.map, p.partial, p.Y, p.n_cand, p.n_users, p.N, p.D,
                                                          p.status);
    e = cudaGetLastError();
    if (e == cudaSuccess) *launches += 1;
  }
  return e;
}

}  // namespace ikbo
