// seg.cu -- map -> per-user segments and the broadcast-attention work list.
//
// IKBO's runtime hands the kernels a candidate->user map instead of a
// replicated tensor ("Meta Optimizes Inference for Recommendation Systems",
// RO/NRO paragraph).  Broadcast attention fetches one user's K/V once for all
// of that user's candidates (aixai.ru, "Deep Dive: Flash Attention"), so the
// candidates are grouped per user first:
//   counts[u]  = #{i : map[i] = u}
//   offsets    = exclusive prefix sum of counts (offsets[n_users] = #valid)
//   perm       = candidates grouped by user, ascending i inside a user (stable);
//                candidates with a map value out of range follow, ascending
//   work       = for u, for h, for each run of <= cands_per_unit entries of
//                u's segment: (u, h, first perm position, run length)
// Everything is integer work, so the result is unique and bit-exact.
//
// One CTA of 1024 threads.  Counts and cursors live in shared memory, so the
// user count is limited to SEG_MAX_USERS.  Stability comes from processing
// the candidates in blocks of 1024 in index order and, inside a block, warp
// by warp in index order: within a warp, lanes with the same user are ranked
// by lane (match.any + popc), and one leader per user advances the cursor.
#include "ikbo_internal.h"

namespace ikbo {

constexpr int SEG_FAST_USERS = 32;  // up to this many users the stable scatter runs all warps at once

// Exclusive scan over the 1024 threads of the block; returns the prefix and
// writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = warp_sums[lane];
    int si = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, si, o);
      if (lane >= o) si += y;
    }
    warp_sums[lane] = si - s;
    if (lane == 31) warp_sums[32] = si;
  }
  __syncthreads();
  int r = incl - v + warp_sums[warp];
  *total = warp_sums[32];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(SEG_THREADS, 1) seg_build_kernel(SegParams p) {
  extern __shared__ int32_t sm[];
  int32_t* cnt = sm;                       // [n_users]
  int32_t* cursor = sm + p.n_users;        // [n_users]
  int32_t* ubase = sm + 2 * p.n_users;     // [n_users + 1]
  __shared__ int warp_sums[33];
  __shared__ int wcount[SEG_THREADS / 32][SEG_FAST_USERS];  // per warp, per user (few-user scatter)

  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int nu = p.n_users;

  for (int u = tid; u < nu; u += SEG_THREADS) cnt[u] = 0;
  __syncthreads();

  // histogram: the lanes of a warp that share a user add their count once
  bool bad = false;
  for (int base = 0; base < p.n_cand; base += SEG_THREADS) {
    const int i = base + tid;
    int u = i < p.n_cand ? p.map[i] : -1;
    if (i < p.n_cand && (u < 0 || u >= nu)) bad = true;
    if (u < 0 || u >= nu) u = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, u);
    if (u >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt[u], __popc(peers));
  }
  if (bad) atomicOr(p.status, DEV_ERR_MAP_RANGE);
  __syncthreads();

  // offsets: each thread scans a contiguous range of users
  const int per = (nu + SEG_THREADS - 1) / SEG_THREADS;
  const int lo = min(tid * per, nu), hi = min(lo + per, nu);
  int local = 0;
  for (int u = lo; u < hi; ++u) local += cnt[u];
  int total;
  int run = block_exclusive_scan(local, warp_sums, &total);
  for (int u = lo; u < hi; ++u) {
    cursor[u] = run;
    p.offsets[u] = run;
    p.counts[u] = cnt[u];
    run += cnt[u];
  }
  if (tid == 0) p.offsets[nu] = total;

  // non-empty runs before each user (the LCE weights its ranges by them)
  int local_runs = 0;
  for (int u = lo; u < hi; ++u) local_runs += cnt[u] > 0;
  int total_runs;
  int rrun = block_exclusive_scan(local_runs, warp_sums, &total_runs);
  for (int u = lo; u < hi; ++u) {
    p.runs[u] = rrun;
    rrun += cnt[u] > 0;
  }
  if (tid == 0) p.runs[nu] = total_runs;

  // work units per user: H * ceil(count / cands_per_unit)
  const int cpu = p.cands_per_unit;
  int local_units = 0;
  for (int u = lo; u < hi; ++u) local_units += p.H * ((cnt[u] + cpu - 1) / cpu);
  int total_units;
  int urun = block_exclusive_scan(local_units, warp_sums, &total_units);
  for (int u = lo; u < hi; ++u) {
    ubase[u] = urun;
    urun += p.H * ((cnt[u] + cpu - 1) / cpu);
  }
  if (tid == 0) ubase[nu] = total_units;
  __syncthreads();

  // stable scatter into perm
  const uint32_t lt_mask = (1u << lane) - 1u;
  if (nu <= SEG_FAST_USERS) {
    // few users: each candidate's place among the block's earlier candidates
    // of its user = (its user's count in the earlier warps) + (its rank in
    // its warp); the per-warp counts [warp][user] are scanned over the warps
    // by one warp per user, so no warp waits for another
    for (int base = 0; base < p.n_cand; base += SEG_THREADS) {
      const int i = base + tid;
      int u = (i < p.n_cand) ? p.map[i] : -1;
      if (u < 0 || u >= nu) u = -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, u);
      const int rank = __popc(peers & lt_mask);
      wcount[warp][lane] = 0;
      __syncwarp();
      if (u >= 0 && lane == __ffs(peers) - 1) wcount[warp][u] = __popc(peers);
      __syncthreads();
      if (warp < nu) {  // warp w scans user w's counts over the 32 warps (lane = warp index)
        const int c = wcount[lane][warp];
        int incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        wcount[lane][warp] = cursor[warp] + incl - c;  // where this warp's run of the user starts
        __syncwarp();
        if (lane == 31) cursor[warp] += incl;
      }
      __syncthreads();
      if (u >= 0) p.perm[wcount[warp][u] + rank] = i;
      __syncthreads();  // wcount is rewritten by the next block of candidates
    }
  } else {
    for (int base = 0; base < p.n_cand; base += SEG_THREADS) {
      const int i = base + tid;
      int u = (i < p.n_cand) ? p.map[i] : -1;
      if (u < 0 || u >= nu) u = -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, u);
      const int rank = __popc(peers & lt_mask);
      const int leader = __ffs(peers) - 1;
      for (int w = 0; w < SEG_THREADS / 32; ++w) {
        if (warp == w) {
          int pos = 0;
          if (u >= 0 && lane == leader) {
            pos = cursor[u];
            cursor[u] = pos + __popc(peers);
          }
          pos = __shfl_sync(0xffffffffu, pos, leader);
          if (u >= 0) p.perm[pos + rank] = i;
        }
        __syncthreads();
      }
    }
  }

  // candidates whose map value is out of range follow the valid ones in
  // perm, in index order: they belong to no user's segment, but a kernel that
  // walks every position of perm (the LCE backward's candidate pass) still
  // reaches them
  if (__syncthreads_or(bad)) {
    int tail = total;
    for (int base = 0; base < p.n_cand; base += SEG_THREADS) {
      const int i = base + tid;
      const int u = i < p.n_cand ? p.map[i] : 0;
      const bool inv = i < p.n_cand && (u < 0 || u >= nu);
      int block_inv;
      const int pre = block_exclusive_scan(inv ? 1 : 0, warp_sums, &block_inv);
      if (inv) p.perm[tail + pre] = i;
      tail += block_inv;
      __syncthreads();  // warp_sums is reused by the next scan
    }
  }

  // work list, one unit per thread iteration; user found by binary search
  int64_t n_out = total_units;
  if (n_out > p.max_units) {
    if (tid == 0) atomicOr(p.status, DEV_ERR_BAD_WORK);
    n_out = p.max_units;
  }
  for (int64_t k = tid; k < n_out; k += SEG_THREADS) {
    int a = 0, b = nu;  // find the last u with ubase[u] <= k
    while (b - a > 1) {
      int mid = (a + b) >> 1;
      if (ubase[mid] <= k) a = mid;
      else b = mid;
    }
    const int u = a;
    const int nch = (cnt[u] + cpu - 1) / cpu;
    const int r = static_cast<int>(k - ubase[u]);
    const int h = r / nch, ch = r - h * nch;
    const int first = cursor[u] - cnt[u] + ch * cpu;  // cursor[u] ended at offsets[u] + cnt[u]
    int4 unit;
    unit.x = u;
    unit.y = h;
    unit.z = first;
    unit.w = min(cpu, cnt[u] - ch * cpu);
    reinterpret_cast<int4*>(p.work)[k] = unit;
  }
  if (tid == 0) *p.n_units = static_cast<int32_t>(n_out);
}

cudaError_t launch_seg_build(const SegParams& p, cudaStream_t s) {
  const size_t smem = sizeof(int32_t) * (3 * static_cast<size_t>(p.n_users) + 1);
  static thread_local int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(seg_build_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sizeof(int32_t) * (3 * SEG_MAX_USERS + 1)));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  seg_build_kernel<<<1, SEG_THREADS, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ikbo
