// lce_bwd.cu -- LCE backward (training) with the broadcast kept implicit.
//
// The IKBO write-ups state that the same kernels serve training when the
// candidate:user ratio exceeds 1 ("Meta Optimizes Inference for
// Recommendation Systems", the paragraph on kernels, compilation and
// runtime).  The backward of Y[i] = W_u^T U[map[i]] + W_c^T C[i] + b is the
// forward's Type I split run in reverse: the transpose of "broadcast U[u] to
// every candidate of u" is "sum the gradients of u's candidates", so the user
// side never sees n_cand either:
//   S[u]  = sum_{i : map[i] = u} dY[i]          segment sum (fp32), n_users rows
//   db[n] = sum_u sum_d S[u][n][d]
//   dU[u] = W_u S[u]        dW_u = sum_u U[u] S[u]^T     (at n_users)
//   dC[i] = W_c dY[i]       dW_c = sum_i C[i] dY[i]^T    (at n_cand)
// S is rounded to bf16 for the two tensor-core products that read it.
//
// Kernels:
//   bwd_cand_kernel    the candidate side in one pass over dY (and C): dC,
//                      dW_c, S and db, ending (cooperative launch) with the
//                      finish -- or bwd_cand_finish_kernel after it
//   bwd_act_kernel     out[b][m][d] = sum_n W[m][n] X[b][n][d]   (dU; dC where
//                      the candidate pass does not apply)
//   bwd_wgrad_kernel   split-K sum_b sum_d A[b][m][d] G[b][n][d] (dW_u; dW_c
//                      where the candidate pass does not apply): the split-K
//                      CTAs of an m block add their partials as a cluster,
//                      or write them for bwd_wgrad_reduce_kernel
//   bwd_segsum_kernel / bwd_segsum_finish_kernel, bwd_db_kernel: S and db
//                      where the candidate pass does not apply
// The GEMM kernels are persistent, one CTA per SM, warp-specialised like the
// forward: TMA producer warp(s) (elected lane issues), warp 1 tcgen05.mma
// (elected lane), warp 2 TMEM owner, warps 4-11 epilogue.  Every wait on an
// mbarrier, a flag or the grid barrier is bounded.
#include <cuda_bf16.h>

#include "bwd_internal.h"
#include "ptx.cuh"

namespace ikbo {

namespace {

constexpr uint32_t BOX = 64 * 64 * 2;  // one 64 x 64 bf16 box, 8 KB

// ------------------------------------------------------------ segment sum
// S2[u][0][.] = bf16(S), S2[u][1][.] = bf16(S - bf16(S)) for 8 elements at e.
__device__ __forceinline__ void store_pair(const SegSumParams& p, int u, int e, const float (&acc)[8]) {
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    hi[j] = pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
    lo[j] = pack_bf16x2(acc[2 * j] - __uint_as_float(hi[j] << 16),
                        acc[2 * j + 1] - __uint_as_float(hi[j] & 0xffff0000u));
  }
  uint16_t* base = p.S2 + static_cast<size_t>(u) * 2 * p.NPD + e;
  *reinterpret_cast<uint4*>(base) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(base + p.NPD) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Task = (user u, chunk c of u's segment, slice s of the N*D elements); each
// thread sums 8 consecutive elements (one 16-byte load per candidate) over
// the chunk's candidates in ascending perm order.  The CTA stages 128 perm
// entries at a time in shared memory, so the dY loads do not wait on a
// dependent perm load, and each thread keeps 8 loads in flight.
__global__ void __launch_bounds__(BWD_SEG_THREADS) bwd_segsum_kernel(const SegSumParams p) {
  __shared__ int rows[BWD_SEG_THREADS];
  const int task = blockIdx.x;
  const int s = task % p.slices;
  const int uc = task / p.slices;
  const int c = uc % p.nch;
  const int u = uc / p.nch;
  const int e = s * BWD_SEG_SLICE + static_cast<int>(threadIdx.x) * 8;
  const bool active = e < p.ND;
  const int p0 = __ldg(p.offsets + u), cnt = __ldg(p.offsets + u + 1) - p0;
  const int q0 = p0 + static_cast<int>(static_cast<long long>(cnt) * c / p.nch);
  const int q1 = p0 + static_cast<int>(static_cast<long long>(cnt) * (c + 1) / p.nch);
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  auto add = [&](const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[2 * j] += __uint_as_float(w[j] << 16);
      acc[2 * j + 1] += __uint_as_float(w[j] & 0xffff0000u);
    }
  };
  const uint4 zero = make_uint4(0, 0, 0, 0);
  auto load = [&](int r) -> uint4 {
    return r < 0 ? zero : __ldcs(reinterpret_cast<const uint4*>(p.dY + static_cast<size_t>(r) * p.ND + e));
  };
  for (int base = q0; base < q1; base += BWD_SEG_THREADS) {
    const int n = min(BWD_SEG_THREADS, q1 - base);
    __syncthreads();
    if (static_cast<int>(threadIdx.x) < n) {
      const int i = __ldg(p.perm + base + threadIdx.x);
      rows[threadIdx.x] = (i >= 0 && i < p.n_cand) ? i : -1;
    }
    __syncthreads();
    if (!active) continue;
    int j = 0;
    for (; j + 8 <= n; j += 8) {
      uint4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = load(rows[j + k]);
#pragma unroll
      for (int k = 0; k < 8; ++k) add(v[k]);
    }
    for (; j < n; ++j) add(load(rows[j]));
  }
  if (!active) return;
  if (p.nch == 1) {
    float4* S = reinterpret_cast<float4*>(p.S + static_cast<size_t>(u) * p.ND + e);
    S[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    S[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    store_pair(p, u, e, acc);
  } else {
    float4* P = reinterpret_cast<float4*>(p.part + static_cast<size_t>(u * p.nch + c) * p.ND + e);
    P[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    P[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// S[u] = sum over u's chunks, in chunk order.
__global__ void __launch_bounds__(BWD_SEG_THREADS) bwd_segsum_finish_kernel(const SegSumParams p) {
  const int s = blockIdx.x % p.slices;
  const int u = blockIdx.x / p.slices;
  const int e = s * BWD_SEG_SLICE + static_cast<int>(threadIdx.x) * 8;
  if (u >= p.n_users || e >= p.ND) return;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  for (int c = 0; c < p.nch; ++c) {
    const float4* P = reinterpret_cast<const float4*>(p.part + static_cast<size_t>(u * p.nch + c) * p.ND + e);
    const float4 a = P[0], b = P[1];
    acc[0] += a.x;
    acc[1] += a.y;
    acc[2] += a.z;
    acc[3] += a.w;
    acc[4] += b.x;
    acc[5] += b.y;
    acc[6] += b.z;
    acc[7] += b.w;
  }
  float4* S = reinterpret_cast<float4*>(p.S + static_cast<size_t>(u) * p.ND + e);
  S[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  S[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  store_pair(p, u, e, acc);
}

// db[n] = sum_u sum_d S[u][n][d]: one CTA per n, a fixed reduction tree.
constexpr int BWD_DB_THREADS = 256;
__global__ void __launch_bounds__(BWD_DB_THREADS) bwd_db_kernel(const float* S, float* db, int n_users, int N,
                                                                int D) {
  __shared__ float red[BWD_DB_THREADS];
  const int n = blockIdx.x;
  float acc = 0.f;
  const int total = n_users * D;
#pragma unroll 8
  for (int t = threadIdx.x; t < total; t += BWD_DB_THREADS) {
    const int u = t / D, d = t - u * D;
    acc += S[(static_cast<size_t>(u) * N + n) * D + d];
  }
  red[threadIdx.x] = acc;
  __syncthreads();
  for (int w = BWD_DB_THREADS / 2; w > 0; w >>= 1) {
    if (static_cast<int>(threadIdx.x) < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) db[n] = red[0];
}

// ------------------------------------------------------------------------
// Shared pieces of the two GEMM kernels.

// A wait taken by a whole warp; the lanes agree on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* abort, uint64_t timeout_ns) {
  const bool ok = mbar_wait(bar, parity, abort, timeout_ns, 1);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------- activation-gradient GEMM
// Shared memory: W resident (kc chunks x m_rows rows x 128 B, K-major: row m
// holds 64 n of one chunk, 128-byte swizzle), then the X ring (stages of two
// 64 d x 64 n boxes, MN-major), then the barriers.
struct ActSmem {
  uint8_t* w;
  uint8_t* ring;
  uint64_t* a_full;
  uint64_t* a_empty;
  uint64_t* w_full;
  uint64_t* acc_full;   // [2]
  uint64_t* acc_empty;  // [2]
  uint32_t* tmem_slot;
  uint32_t* abort;
};

__host__ __device__ constexpr uint32_t act_w_bytes(int kc, int m_rows) {
  return static_cast<uint32_t>(kc) * static_cast<uint32_t>(m_rows) * 128u;
}

__device__ __forceinline__ ActSmem act_carve(uint8_t* base, const ActParams& p) {
  ActSmem s;
  s.w = base;
  s.ring = base + act_w_bytes(p.kc, p.m_rows);
  uint64_t* b = reinterpret_cast<uint64_t*>(s.ring + static_cast<size_t>(p.stages) * 2 * BOX);
  s.a_full = b;
  s.a_empty = b + p.stages;
  s.w_full = b + 2 * p.stages;
  s.acc_full = s.w_full + 1;
  s.acc_empty = s.acc_full + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.acc_empty + 2);
  s.abort = s.tmem_slot + 1;
  return s;
}

// Tiles q = (mg * n_dblk + dblk) * B + b (block of M rows, then
// D-block-major); each CTA takes one contiguous range (one tile per CTA
// when M is split, so that its resident W block is the tile's).
__device__ __forceinline__ void act_range(const ActParams& p, int& q0, int& q1) {
  const long long nq = static_cast<long long>(p.B) * p.n_dblk * p.n_mgrp;
  q0 = static_cast<int>(blockIdx.x * nq / gridDim.x);
  q1 = static_cast<int>((blockIdx.x + 1) * nq / gridDim.x);
}

__global__ void __launch_bounds__(BWD_THREADS, 1)
    bwd_act_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const ActParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const ActSmem s = act_carve(base, p);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&s.a_full[i], 1);
      mbar_init(&s.a_empty[i], 1);
    }
    mbar_init(s.w_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], BWD_THREADS - 128);
    }
    *s.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 2) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  int q0, q1;
  act_range(p, q0, q1);

  if (warp == 0) {
    // ---- TMA producer: W (the CTA's block of M rows) once, then the X
    // chunks of every tile
    if (elect_one()) {
      const int m0 = (q0 / (p.n_dblk * p.B)) * p.m_rows;
      mbar_arrive_expect_tx(s.w_full, act_w_bytes(p.kc, p.m_rows));
      for (int kc = 0; kc < p.kc; ++kc)
        for (int r = 0; r < p.m_rows; r += 128)
          tma_load_2d(s.w + (static_cast<size_t>(kc) * p.m_rows + r) * 128, &tmW, s.w_full, kc * 64, m0 + r);
    }
    __syncwarp();
    int stage = 0;
    uint32_t phase = 0;
    for (int q = q0; q < q1; ++q) {
      const int rem = q % (p.n_dblk * p.B);
      const int dblk = rem / p.B, b = rem - dblk * p.B;
      for (int kc = 0; kc < p.kcx; ++kc) {
        if (!warp_wait(&s.a_empty[stage], phase ^ 1u, s.abort, p.timeout_ns)) goto done;
        if (elect_one()) {
          uint8_t* dst = s.ring + static_cast<size_t>(stage) * 2 * BOX;
          mbar_arrive_expect_tx(&s.a_full[stage], 2 * BOX);
          tma_load_3d(dst, &tmX, &s.a_full[stage], dblk * 128, kc * 64, b);
          tma_load_3d(dst + BOX, &tmX, &s.a_full[stage], dblk * 128 + 64, kc * 64, b);
        }
        __syncwarp();
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: per chunk, every m range of the tile
    if (!warp_wait(s.w_full, 0, s.abort, p.timeout_ns)) goto done;
    int stage = 0;
    uint32_t phase = 0;
    for (int q = q0, t = 0; q < q1; ++q, ++t) {
      const int buf = p.bufs == 2 ? (t & 1) : 0;
      const uint32_t use = static_cast<uint32_t>(p.bufs == 2 ? (t >> 1) : t);
      if (!warp_wait(&s.acc_empty[buf], (use & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      for (int kc = 0; kc < p.kcx; ++kc) {
        if (!warp_wait(&s.a_full[stage], phase, s.abort, p.timeout_ns)) goto done;
        tc_fence_after();
        const int wkc = kc % p.kc;  // K rows past N read as zeros on both sides
        if (elect_one()) {
          const uint32_t a_base = smem_u32(s.ring + static_cast<size_t>(stage) * 2 * BOX);
          // X chunk, MN-major: the two 64-d boxes one BOX apart, 16 n rows per step
          const uint64_t adesc = sdesc_sw128(a_base, BOX, 1024u);
          for (int r = 0; r * 256 < p.m_pad; ++r) {
            const int nr = min(256, p.m_pad - r * 256);
            const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(nr), true, false);
            // W, K-major: rows m of 128 bytes, 8-row atoms; a 16-n step is 32 bytes
            const uint64_t bdesc =
                sdesc_sw128(smem_u32(s.w + (static_cast<size_t>(wkc) * p.m_rows + r * 256) * 128), 16, 1024u);
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * 256 + r * 256);
#pragma unroll
            for (int st = 0; st < 4; ++st)
              mma_bf16_ss(d_tmem, adesc + st * (2048u >> 4), bdesc + st * (32u >> 4), idesc,
                          (kc > 0 || st > 0) ? 1u : 0u);
          }
          mma_commit(&s.a_empty[stage]);
        }
        __syncwarp();
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (elect_one()) mma_commit(&s.acc_full[buf]);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ---- epilogue: TMEM lane = row d of the D block, columns = m
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    for (int q = q0, t = 0; q < q1; ++q, ++t) {
      const int mg = q / (p.n_dblk * p.B), rem = q - mg * (p.n_dblk * p.B);
      const int dblk = rem / p.B, b = rem - dblk * p.B;
      const int m0 = mg * p.m_rows, mlen = min(p.M - m0, p.m_rows);
      const int nchunks = (mlen + 31) / 32;
      const int buf = p.bufs == 2 ? (t & 1) : 0;
      const uint32_t use = static_cast<uint32_t>(p.bufs == 2 ? (t >> 1) : t);
      if (!warp_wait(&s.acc_full[buf], use & 1u, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      const int d = dblk * 128 + quarter * 32 + static_cast<int>(lane_id());
      const bool dok = d < p.D;
      __nv_bfloat16* out =
          reinterpret_cast<__nv_bfloat16*>(p.out) + (static_cast<size_t>(b) * p.M + m0) * p.D + d;
      for (int c = half; c < nchunks; c += 2) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(buf * 256 + c * 32), v);
        tmem_ld_wait(v);
        __nv_bfloat16* o = out + static_cast<size_t>(c * 32) * p.D;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (c * 32 + j < mlen && dok) *o = __float2bfloat16_rn(__uint_as_float(v[j]));
          o += p.D;
        }
      }
      tc_fence_before();
      mbar_arrive(&s.acc_empty[buf]);
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (*s.abort && threadIdx.x == 0) atomicOr(p.status, DEV_ERR_PIPE_TIMEOUT);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------ thread-block clusters
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster (a hardware barrier like
// __syncthreads; each path to it is bounded).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The address of this CTA's shared-memory location `saddr` in the CTA of
// cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

// ---------------------------------------------------- weight-gradient GEMM
// A unit covers a group of up to two 128-row m blocks (accumulators at TMEM
// columns 0 and 256) over one b range, so the G tiles it loads serve both
// blocks.  Stage = one 64 d x 128 m box of A per block of the group (16 KB
// each) + nb boxes of 64 d x 64 n of G (8 KB each), all K-major (d
// contiguous), 128-byte swizzle.
__host__ __device__ constexpr uint32_t wg_stage_bytes(int mg, int nb) {
  return static_cast<uint32_t>(mg) * 2 * BOX + static_cast<uint32_t>(nb) * BOX;
}

struct WgSmem {
  uint8_t* ring;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* acc_full;
  uint64_t* acc_empty;
  uint32_t* tmem_slot;
  uint32_t* abort;
};

__device__ __forceinline__ WgSmem wg_carve(uint8_t* base, const WgradParams& p) {
  WgSmem s;
  s.ring = base;
  uint64_t* b = reinterpret_cast<uint64_t*>(base + static_cast<size_t>(p.stages) * wg_stage_bytes(p.mg, p.nb));
  s.full = b;
  s.empty = b + p.stages;
  s.acc_full = b + 2 * p.stages;
  s.acc_empty = s.acc_full + 1;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.acc_empty + 1);
  s.abort = s.tmem_slot + 1;
  return s;
}

// Unit u = (m group u / R, b range u % R); b range r = [r*B/R, (r+1)*B/R),
// never empty because R <= B.  nblk = the group's m blocks inside M.
__device__ __forceinline__ void wg_unit(const WgradParams& p, int u, int& mblk0, int& nblk, int& r, int& b0,
                                        int& b1) {
  const int g = u / p.R;
  r = u - g * p.R;
  mblk0 = g * p.mg;
  nblk = min(p.mg, p.n_mblk - mblk0);
  b0 = static_cast<int>(static_cast<long long>(r) * p.B / p.R);
  b1 = static_cast<int>(static_cast<long long>(r + 1) * p.B / p.R);
}

__global__ void __launch_bounds__(BWD_THREADS, 1)
    bwd_wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmG,
                     const WgradParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const WgSmem s = wg_carve(base, p);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.stages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    mbar_init(s.acc_full, 1);
    mbar_init(s.acc_empty, BWD_THREADS - 128);
    *s.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmG);
  }
  if (warp == 2) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  const int n_units = p.n_mgrp * p.R;
  const uint32_t sbytes = wg_stage_bytes(p.mg, p.nb);
  const uint32_t g_off = static_cast<uint32_t>(p.mg) * 2 * BOX;  // G boxes after the A boxes

  if (warp == 0) {
    // ---- TMA producer
    int stage = 0;
    uint32_t phase = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
      int mblk0, nblk, r, b0, b1;
      wg_unit(p, u, mblk0, nblk, r, b0, b1);
      const uint32_t bytes = static_cast<uint32_t>(nblk) * 2 * BOX + static_cast<uint32_t>(p.nb) * BOX;
      for (int b = b0; b < b1; ++b)
        for (int dc = 0; dc < p.dc; ++dc) {
          if (!warp_wait(&s.empty[stage], phase ^ 1u, s.abort, p.timeout_ns)) goto done;
          if (elect_one()) {
            uint8_t* dst = s.ring + static_cast<size_t>(stage) * sbytes;
            mbar_arrive_expect_tx(&s.full[stage], bytes);
            for (int j = 0; j < nblk; ++j)
              tma_load_3d(dst + static_cast<size_t>(j) * 2 * BOX, &tmA, &s.full[stage], dc * 64, (mblk0 + j) * 128,
                          b >> p.a_shift);
            for (int j = 0; j < p.nb; ++j)
              tma_load_3d(dst + g_off + static_cast<size_t>(j) * BOX, &tmG, &s.full[stage], dc * 64, j * 64, b);
          }
          __syncwarp();
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: D_j[m][n] += A_j[m][d-chunk] G[n][d-chunk]^T, 4 steps of 16 d
    const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(p.n_mma), false, false);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t use = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++use) {
      int mblk0, nblk, r, b0, b1;
      wg_unit(p, u, mblk0, nblk, r, b0, b1);
      if (!warp_wait(s.acc_empty, (use & 1u) ^ 1u, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      bool first = true;
      for (int b = b0; b < b1; ++b)
        for (int dc = 0; dc < p.dc; ++dc) {
          if (!warp_wait(&s.full[stage], phase, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          if (elect_one()) {
            const uint32_t st_base = smem_u32(s.ring + static_cast<size_t>(stage) * sbytes);
            const uint64_t bdesc = sdesc_sw128(st_base + g_off, 16, 1024u);
            for (int j = 0; j < nblk; ++j) {
              const uint64_t adesc = sdesc_sw128(st_base + static_cast<uint32_t>(j) * 2 * BOX, 16, 1024u);
#pragma unroll
              for (int st = 0; st < 4; ++st)
                mma_bf16_ss(tmem + static_cast<uint32_t>(j * 256), adesc + st * (32u >> 4), bdesc + st * (32u >> 4),
                            idesc, (first && st == 0) ? 0u : 1u);
            }
            mma_commit(&s.empty[stage]);
          }
          __syncwarp();
          first = false;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      if (elect_one()) mma_commit(s.acc_full);
      __syncwarp();
    }
  } else if (warp >= 4) {
    // ---- epilogue: TMEM lane = row m of a block, columns = n -> fp32 partial
    // part[(m block * R + r) * 128 + row][n]
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int row = quarter * 32 + static_cast<int>(lane_id());
    const int nchunks = (p.N + 31) / 32;
    uint32_t use = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++use) {
      int mblk0, nblk, r, b0, b1;
      wg_unit(p, u, mblk0, nblk, r, b0, b1);
      if (!warp_wait(s.acc_full, use & 1u, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      if (p.cluster) {  // one unit per CTA, one m block: the partial goes to this CTA's own shared memory
        float* red = reinterpret_cast<float*>(s.ring) + row * (p.n_mma + 1);
        for (int c = half; c < nchunks; c += 2) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(c * 32), v);
          tmem_ld_wait(v);
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (c * 32 + k < p.N) red[c * 32 + k] = __uint_as_float(v[k]);
        }
        nblk = 0;
      }
      for (int j = 0; j < nblk; ++j) {
        float* out = p.part + (static_cast<size_t>((mblk0 + j) * p.R + r) * 128 + row) * p.N;
        for (int c = half; c < nchunks; c += 2) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(j * 256 + c * 32), v);
          tmem_ld_wait(v);
          if (c * 32 + 32 <= p.N) {
            float4* o4 = reinterpret_cast<float4*>(out + c * 32);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o4[k] = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                  __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
          } else {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (c * 32 + k < p.N) out[c * 32 + k] = __uint_as_float(v[k]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(s.acc_empty);
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (*s.abort && threadIdx.x == 0) atomicOr(p.status, DEV_ERR_PIPE_TIMEOUT);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (!p.cluster) return;
  // the R partials of m block blockIdx.x / R, in the shared memory of the R
  // CTAs of this cluster: CTA rank k writes rows [k*128/R, (k+1)*128/R) of
  // dW, each the sum of the partials in rank order (a fixed order)
  cluster_sync_all();
  {
    const uint32_t R = static_cast<uint32_t>(p.R), rank = cluster_rank();
    const int mblk = static_cast<int>(blockIdx.x) / p.R;
    const int r0 = static_cast<int>(rank * 128u / R), r1 = static_cast<int>((rank + 1u) * 128u / R);
    const int RS = p.n_mma + 1;
    const uint32_t red = smem_u32(s.ring);
    for (int e = threadIdx.x; e < (r1 - r0) * p.N; e += BWD_THREADS) {
      const int row = r0 + e / p.N, n = e - (e / p.N) * p.N;
      const int m = mblk * 128 + row;
      if (m >= p.M) continue;
      const uint32_t off = static_cast<uint32_t>(row * RS + n) * 4u;
      float v = 0.f;
      for (uint32_t k = 0; k < R; ++k) v += ld_cluster_f32(cluster_map(red + off, k));
      p.dW[static_cast<size_t>(m) * p.N + n] = v;
    }
  }
  cluster_sync_all();  // no CTA leaves while another still reads its partial
}

// dW[m][n] = sum over the b ranges of m's block.  32 outputs per CTA, 8
// threads per output each summing every 8th range, then the 8 sums in order:
// a fixed order, so the result repeats bit for bit.
constexpr int WG_RED_OUT = 32, WG_RED_SPLIT = 8;
__global__ void __launch_bounds__(WG_RED_OUT* WG_RED_SPLIT)
    bwd_wgrad_reduce_kernel(const float* part, float* dW, int M, int N, int R) {
  __shared__ float red[WG_RED_SPLIT][WG_RED_OUT + 1];
  const int o = blockIdx.x * WG_RED_OUT + threadIdx.x;
  const bool ok = o < M * N;
  float acc = 0.f;
  if (ok) {
    const int m = o / N, n = o - m * N;
    const int mblk = m >> 7, row = m & 127;
#pragma unroll 4
    for (int r = threadIdx.y; r < R; r += WG_RED_SPLIT)
      acc += part[(static_cast<size_t>(mblk * R + r) * 128 + row) * N + n];
  }
  red[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y == 0 && ok) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < WG_RED_SPLIT; ++k) t += red[k][threadIdx.x];
    dW[o] = t;
  }
}

// ============================================================ candidate pass
// See CandParams.  Per CTA (one per SM, 12 warps): warp 0 TMA producer of
// W_c and dY, warp 1 MMA issuer, warp 2 TMEM owner, warp 3 TMA producer of
// C, warps 4-11 epilogue (S sums, dC read-out, the dW_c partial).
// Units q = dh * n_cand + pos (D-block-major over the plan's grouped order),
// one contiguous range per CTA, so a CTA's consecutive units share a user
// and its S sums stay in registers.
// TMEM columns: dW_c block 0 [0, n_mma), block 1 [n_mma, 2 n_mma) (lanes =
// K_c rows, columns = n), accumulated over the CTA's units; two dC
// accumulators of 64 columns at CAND_DC_COL (lanes = K_c rows of one block,
// columns = the unit's 64 d), used in turn: accumulator c of the CTA (c =
// unit * n_mblk + block) is read out by epilogue warps 4-7 if c is even,
// 8-11 if odd.
// Shared memory: W_c ([n chunk][K_c row][64 n], 128-byte swizzle: K-major A
// of dC), the dY slots ([n chunk][64 n rows][64 d]: K-major B of dW_c and
// MN-major B of dC), the ring of C slots (128 K_c rows x 64 d: K-major A of
// dW_c), the barriers.
constexpr uint32_t CB_SLOT = 128 * 64 * 2;      // 16 KB
constexpr uint32_t CAND_DY_SLOT = 3 * BOX;      // 24 KB
constexpr uint32_t CAND_W_BYTES = 3 * 256 * 128;  // W_c: <= 3 n chunks x 256 rows x 128 B
constexpr uint32_t CAND_TILES =
    CAND_W_BYTES + BWD_CAND_DY_SLOTS * CAND_DY_SLOT + BWD_CAND_C_SLOTS * CB_SLOT;
constexpr int CAND_BARS = 2 * BWD_CAND_DY_SLOTS + 2 * BWD_CAND_C_SLOTS + 1 + 4 + 1;
constexpr size_t CAND_SMEM = 1024 + CAND_TILES + 8 * CAND_BARS + 16 + 4 * BWD_CAND_MAX_N + 16 * 4;
static_assert(CAND_SMEM <= 227 * 1024, "candidate pass does not fit in shared memory");
constexpr uint32_t CAND_DC_COL = 2 * BWD_CAND_MAX_N;  // after the two dW_c blocks
static_assert(CAND_DC_COL + 128 <= 512, "candidate pass accumulators exceed TMEM");
constexpr int CAND_EPI = BWD_THREADS - 128;  // epilogue threads

struct CandSmem {
  uint8_t* w;
  uint8_t* dy;
  uint8_t* ring;
  uint64_t* dy_full;   // [DY_SLOTS]
  uint64_t* dy_empty;  // [DY_SLOTS] MMA reads done (commit) and the S sums taken
  uint64_t* st_full;   // [C_SLOTS]
  uint64_t* st_empty;  // [C_SLOTS]
  uint64_t* w_full;    // W_c resident
  uint64_t* dc_full;   // [2]
  uint64_t* dc_empty;  // [2]
  uint64_t* wacc_full;  // the CTA's dW_c partial is complete in TMEM
  uint32_t* tmem_slot;
  uint32_t* abort;
  uint32_t* flag;      // the grid barrier was passed
  float* dbsm;         // [BWD_CAND_MAX_N] this CTA's share of db
  int4* pre;           // [4] bounds of this CTA's first finish tasks
};

__device__ __forceinline__ CandSmem cand_carve(uint8_t* base) {
  CandSmem s;
  s.w = base;
  s.dy = base + CAND_W_BYTES;
  s.ring = s.dy + BWD_CAND_DY_SLOTS * CAND_DY_SLOT;
  uint64_t* b = reinterpret_cast<uint64_t*>(base + CAND_TILES);
  s.dy_full = b;
  s.dy_empty = s.dy_full + BWD_CAND_DY_SLOTS;
  s.st_full = s.dy_empty + BWD_CAND_DY_SLOTS;
  s.st_empty = s.st_full + BWD_CAND_C_SLOTS;
  s.w_full = s.st_empty + BWD_CAND_C_SLOTS;
  s.dc_full = s.w_full + 1;
  s.dc_empty = s.dc_full + 2;
  s.wacc_full = s.dc_empty + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.wacc_full + 1);
  s.abort = s.tmem_slot + 1;
  s.flag = s.abort + 1;
  s.dbsm = reinterpret_cast<float*>(s.flag + 2);  // 8-byte aligned
  s.pre = reinterpret_cast<int4*>(s.dbsm + BWD_CAND_MAX_N);  // 16-byte aligned
  return s;
}

// Unit ranges: CTA g of G takes [g * nq / G, (g + 1) * nq / G); the CTA
// whose range holds unit x is ((x + 1) G - 1) / nq.
__device__ __forceinline__ long long cand_q0(long long nq, int g, int G) { return g * nq / G; }
__device__ __forceinline__ int cand_cta_of(long long x, long long nq, int G) {
  return static_cast<int>(((x + 1) * G - 1) / nq);
}

// The candidate (and its user, -1 if out of range) of unit q, looked up by
// the warp 32 units at a time: lane l holds unit wbase + l.  With kBounds
// also the user's segment [offsets[u], offsets[u + 1]).
struct CandWin {
  long long base = -1;
  int b = 0, u = -1, oa = 0, ob = 0;
};
template <bool kBounds = false>
__device__ __forceinline__ void cand_tile(const CandParams& p, long long q, long long q1, CandWin& w, int& b, int& u,
                                          int* oa = nullptr, int* ob = nullptr) {
  if (w.base < 0 || q >= w.base + 32) {
    w.base = q;
    const long long ql = q + static_cast<long long>(lane_id());
    w.b = 0;
    w.u = -1;
    if (ql < q1) {
      const int pos = static_cast<int>(ql % p.n_cand);
      const int bb = __ldg(p.perm + pos);
      w.b = (bb >= 0 && bb < p.n_cand) ? bb : 0;
      const int uu = (bb >= 0 && bb < p.n_cand) ? __ldg(p.map + bb) : -1;
      w.u = (uu >= 0 && uu < p.n_users) ? uu : -1;
      if (kBounds && w.u >= 0) {
        w.oa = __ldg(p.offsets + w.u);
        w.ob = __ldg(p.offsets + w.u + 1);
      }
    }
  }
  const int k = static_cast<int>(q - w.base);
  b = __shfl_sync(0xffffffffu, w.b, k);
  u = __shfl_sync(0xffffffffu, w.u, k);
  if (kBounds) {
    *oa = __shfl_sync(0xffffffffu, w.oa, k);
    *ob = __shfl_sync(0xffffffffu, w.ob, k);
  }
}

template <int kSlots>
struct SlotRing {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == kSlots) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// Epilogue thread layout for S: d pair pd (d = 2 pd, 2 pd + 1 of the unit's
// 64) = lane, rows n = 64 j + 8 ng + i (j < 3, i < 8) with ng = epilogue
// warp; acc[j][i] holds the pair.
using CandAcc = float[3][8][2];

// The final S of run (u, dh) from this thread's sums: the bf16 hi/lo pair
// the user-side products read.
__device__ __forceinline__ void cand_final(const CandParams& p, const CandAcc& acc, int u, int dh, int pd, int ng) {
  const int d = dh * 64 + 2 * pd;
  if (d >= p.D) return;  // D is a multiple of 8: both of the pair or neither
  uint16_t* s2 = p.S2 + static_cast<size_t>(u) * 2 * p.NPD + d;
#pragma unroll
  for (int j = 0; j < 3; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int n = 64 * j + 8 * ng + i;
      if (n < p.N) {
        const uint32_t hi = pack_bf16x2(acc[j][i][0], acc[j][i][1]);
        const uint32_t lo = pack_bf16x2(acc[j][i][0] - __uint_as_float(hi << 16),
                                        acc[j][i][1] - __uint_as_float(hi & 0xffff0000u));
        *reinterpret_cast<uint32_t*>(s2 + static_cast<size_t>(n) * p.D) = hi;
        *reinterpret_cast<uint32_t*>(s2 + p.NPD + static_cast<size_t>(n) * p.D) = lo;
      }
    }
}

// This CTA's share of db: per row n, the sum over the run's 64 d (a fixed
// butterfly over the warp's lanes), added to dbsm[n] run after run.  Each
// row belongs to one epilogue warp, whose lane 0 updates it.
__device__ __forceinline__ void cand_db_add(const CandParams& p, const CandAcc& acc, int ng, float* dbsm) {
  float r[3][8];
#pragma unroll
  for (int j = 0; j < 3; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float x = acc[j][i][0] + acc[j][i][1];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      r[j][i] = x;
    }
  if (lane_id() != 0) return;
#pragma unroll
  for (int j = 0; j < 3; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int n = 64 * j + 8 * ng + i;
      if (n < p.N) dbsm[n] += r[j][i];
    }
}

// A run (u, dh) ends in this CTA's range [q0, q1).  Inside the range: final
// here.  Else its sums go to partial slot 1 if the run began inside the range
// (it runs past the end), else slot 0 (it holds the range's first unit); the
// finish adds the slots of the run's CTAs in CTA order.
__device__ __forceinline__ void cand_flush(const CandParams& p, const CandAcc& acc, int u, int dh, int oa, int ob,
                                           long long q0, long long nq, int pd, int ng, float* dbsm) {
  const int G = static_cast<int>(gridDim.x);
  const long long a = static_cast<long long>(dh) * p.n_cand + oa;
  const long long e = static_cast<long long>(dh) * p.n_cand + ob;
  if (cand_cta_of(a, nq, G) == cand_cta_of(e - 1, nq, G)) {
    cand_final(p, acc, u, dh, pd, ng);
  } else {
    const int slot = a > q0 ? 1 : 0;
    float* dst = p.spart + (static_cast<size_t>(blockIdx.x) * 2 + slot) * p.N * 64 + 2 * pd;
#pragma unroll
    for (int j = 0; j < 3; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int n = 64 * j + 8 * ng + i;
        if (n < p.N) *reinterpret_cast<float2*>(dst + n * 64) = make_float2(acc[j][i][0], acc[j][i][1]);
      }
  }
  cand_db_add(p, acc, ng, dbsm);
}

// The finish, spread over G2 blocks (block g) of CF_THREADS threads whose
// warps work on three parts at once, `red` = CF_RED floats of shared memory:
//   warps 0..CF_CHUNKS-1: dW_c = the partials of the candidate pass's G
//     CTAs, added in a fixed order (warp w sums the CTAs of chunk w in CTA
//     order, 4 consecutive K_c rows of one n per lane, every load of the
//     chunk in flight at once; lane by lane the chunk sums are then added in
//     chunk order);
//   the other warps: S of the runs shared by several CTAs (their slots added
//     in CTA order), then db[n] for n = g, g + G2, ... (the CTAs' shares
//     added in CTA order).
constexpr int CF_CHUNKS = 6;
constexpr int CF_MAX_PER_CHUNK = 26;  // CTAs per chunk: G <= CF_CHUNKS * 26 = 156
constexpr int CF_THREADS = BWD_THREADS;
constexpr int CF_SIDE = CF_THREADS - 32 * CF_CHUNKS;  // threads on the runs and db
constexpr int CF_SLICES = 4;          // slices of a shared run's S
constexpr int CF_UNROLL = 8;        // pairs per thread at a time: a slice of N = 192 in one round
constexpr int CF_BATCH = 4;         // contributing CTAs per round of loads
constexpr int CF_PRE = 4;           // tasks whose bounds the candidate pass looks up ahead
constexpr int CF_RED = CF_CHUNKS * 128 + CF_CHUNKS * CF_MAX_PER_CHUNK;  // chunk sums, then the CTAs' db shares of one n
static_assert(CF_SIDE >= 64 && CF_SIDE % 32 == 0, "finish: too few threads for the runs");
// Bounds of finish task `task` (run r = (u, dh), slice): (u, dh * CF_SLICES
// + slice, c_lo, c_hi with the low bit of c_lo's slot in bit 16 of .y), or
// x = -1 when the run needs no finish (no candidates, or inside one CTA).
__device__ __forceinline__ int4 cand_task_bounds(const CandParams& p, int task) {
  const int r = task / CF_SLICES, sl = task - r * CF_SLICES;
  const int u = r / p.n_dh, dh = r - u * p.n_dh;
  const long long nq = static_cast<long long>(p.n_dh) * p.n_cand;
  const long long a = static_cast<long long>(dh) * p.n_cand + __ldg(p.offsets + u);
  const long long e = static_cast<long long>(dh) * p.n_cand + __ldg(p.offsets + u + 1);
  if (e == a) return make_int4(-1, 0, 0, 0);  // no candidates: zero from the start
  const int c_lo = cand_cta_of(a, nq, p.G), c_hi = cand_cta_of(e - 1, nq, p.G);
  if (c_lo == c_hi) return make_int4(-1, 0, 0, 0);  // final already
  const int slot_lo = a > cand_q0(nq, c_lo, p.G) ? 1 : 0;
  return make_int4(u, (dh * CF_SLICES + sl) | (slot_lo << 16), c_lo, c_hi);
}

// `pre`: the bounds of this block's first CF_PRE tasks, looked up ahead (or
// null).
__device__ __forceinline__ void cand_finish(const CandParams& p, int g, int G2, float* red, const int4* pre) {
  const int t = static_cast<int>(threadIdx.x), w = t >> 5, lane = t & 31;
  if (w < CF_CHUNKS) {
    if (!p.wpart) return;
    const int total4 = p.n_mblk * p.N * 32;  // (block, n, group of 4 rows)
    const size_t cstride = static_cast<size_t>(p.N) * 128;
    const int c0 = w * p.G / CF_CHUNKS, c1 = (w + 1) * p.G / CF_CHUNKS;
    for (int base = g * 32; base < total4; base += G2 * 32) {
      const int e4 = base + lane;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (e4 < total4) {
        const int mb = e4 / (p.N * 32), rem = e4 - mb * p.N * 32;
        const float* src = p.wpart + static_cast<size_t>(mb) * p.G * cstride + static_cast<size_t>(rem) * 4;
        float4 x[CF_MAX_PER_CHUNK];
#pragma unroll
        for (int j = 0; j < CF_MAX_PER_CHUNK; ++j)
          if (c0 + j < c1) x[j] = __ldcg(reinterpret_cast<const float4*>(src + (c0 + j) * cstride));
#pragma unroll
        for (int j = 0; j < CF_MAX_PER_CHUNK; ++j)
          if (c0 + j < c1) {
            v.x += x[j].x;
            v.y += x[j].y;
            v.z += x[j].z;
            v.w += x[j].w;
          }
      }
      reinterpret_cast<float4*>(red)[w * 32 + lane] = v;
      named_barrier_sync(1, 32 * CF_CHUNKS);
      if (w == 0 && e4 < total4) {
        float4 r = reinterpret_cast<const float4*>(red)[lane];
#pragma unroll
        for (int c = 1; c < CF_CHUNKS; ++c) {
          const float4 y = reinterpret_cast<const float4*>(red)[c * 32 + lane];
          r.x += y.x;
          r.y += y.y;
          r.z += y.z;
          r.w += y.w;
        }
        const int mb = e4 / (p.N * 32), rem = e4 - mb * p.N * 32;
        const int n = rem >> 5, k = mb * 128 + (rem & 31) * 4;
        float* dst = p.dWc + static_cast<size_t>(k) * p.N + n;
        if (k < p.K_c) dst[0] = r.x;
        if (k + 1 < p.K_c) dst[p.N] = r.y;
        if (k + 2 < p.K_c) dst[2 * p.N] = r.z;
        if (k + 3 < p.K_c) dst[3 * p.N] = r.w;
      }
      named_barrier_sync(1, 32 * CF_CHUNKS);
    }
    return;
  }
  if (!p.S2) return;
  // runs shared by several CTAs: task (run r = (u, dh), slice) goes to block
  // task mod G2; two d per thread, all of a thread's pairs of the slice and
  // CF_BATCH contributing CTAs per round of loads
  const int ts = t - 32 * CF_CHUNKS;
  const size_t slot_elems = static_cast<size_t>(p.N) * 64;
  const int pairs = p.N * 32, per_slice = (pairs + CF_SLICES - 1) / CF_SLICES;
  for (int task = g, k_task = 0; task < p.n_users * p.n_dh * CF_SLICES; task += G2, ++k_task) {
    const int4 tb = (pre && k_task < CF_PRE) ? pre[k_task] : cand_task_bounds(p, task);
    if (tb.x < 0) continue;
    const int u = tb.x, dh = (tb.y & 0xffff) / CF_SLICES, sl = (tb.y & 0xffff) - dh * CF_SLICES;
    const int slot_lo = tb.y >> 16, c_lo = tb.z, c_hi = tb.w;
    const int i0 = sl * per_slice, i1 = min(pairs, i0 + per_slice);
    for (int ib = i0 + ts; ib < i1; ib += CF_UNROLL * CF_SIDE) {
      float2 v[CF_UNROLL];
#pragma unroll
      for (int k = 0; k < CF_UNROLL; ++k) v[k] = make_float2(0.f, 0.f);
      for (int c0 = c_lo; c0 <= c_hi; c0 += CF_BATCH) {
        float2 x[CF_UNROLL][CF_BATCH];
#pragma unroll
        for (int k = 0; k < CF_UNROLL; ++k) {
          const int idx = ib + k * CF_SIDE;
          const float* src = p.spart + static_cast<size_t>(idx >> 5) * 64 + 2 * (idx & 31);
#pragma unroll
          for (int j = 0; j < CF_BATCH; ++j) {
            const int c = c0 + j;
            const int slot = c == c_lo ? slot_lo : 0;
            x[k][j] = (c <= c_hi && idx < i1)
                          ? __ldcg(reinterpret_cast<const float2*>(src + (static_cast<size_t>(c) * 2 + slot) * slot_elems))
                          : make_float2(0.f, 0.f);
          }
        }
#pragma unroll
        for (int k = 0; k < CF_UNROLL; ++k)
#pragma unroll
          for (int j = 0; j < CF_BATCH; ++j)
            if (c0 + j <= c_hi) {
              v[k].x += x[k][j].x;
              v[k].y += x[k][j].y;
            }
      }
#pragma unroll
      for (int k = 0; k < CF_UNROLL; ++k) {
        const int idx = ib + k * CF_SIDE;
        const int n = idx >> 5, d = dh * 64 + 2 * (idx & 31);
        if (idx >= i1 || d >= p.D) continue;
        uint16_t* s2 = p.S2 + static_cast<size_t>(u) * 2 * p.NPD + static_cast<size_t>(n) * p.D + d;
        const uint32_t hi = pack_bf16x2(v[k].x, v[k].y);
        *reinterpret_cast<uint32_t*>(s2) = hi;
        *reinterpret_cast<uint32_t*>(s2 + p.NPD) =
            pack_bf16x2(v[k].x - __uint_as_float(hi << 16), v[k].y - __uint_as_float(hi & 0xffff0000u));
      }
    }
  }
  // db[n] = the CTAs' shares added in CTA order: the side threads load them
  // (CTA c to thread c mod CF_SIDE), the first adds them from shared memory
  if (!p.db) return;
  float* shares = red + CF_CHUNKS * 128;
  for (int n = g; n < p.N; n += G2) {
    for (int c = ts; c < p.G; c += CF_SIDE) shares[c] = __ldcg(p.dbcta + static_cast<size_t>(c) * p.N + n);
    named_barrier_sync(2, CF_SIDE);
    if (ts == 0) {
      float v = 0.f;
      for (int c = 0; c < p.G; ++c) v += shares[c];
      p.db[n] = v;
    }
    named_barrier_sync(2, CF_SIDE);
  }
}

// Users without candidates: S = 0 (both halves of the pair); CTA g takes
// users g, g + G, ...
__device__ __forceinline__ void cand_empty_users(const CandParams& p) {
  for (int u = blockIdx.x; u < p.n_users; u += gridDim.x) {
    if (__ldg(p.offsets + u + 1) != __ldg(p.offsets + u)) continue;
    uint4* dst = reinterpret_cast<uint4*>(p.S2 + static_cast<size_t>(u) * 2 * p.NPD);
    const int n16 = 2 * p.NPD / 8;
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
  }
}

__global__ void __launch_bounds__(BWD_THREADS, 1)
    bwd_cand_kernel(const __grid_constant__ CUtensorMap tmDY, const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmW, const CandParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const CandSmem s = cand_carve(base);
  const int warp = threadIdx.x >> 5;
  const bool do_s = p.S2 != nullptr;
  const bool do_w = p.wpart != nullptr;
  const bool do_c = p.dC != nullptr;
  if (threadIdx.x == 0) {
    for (int i = 0; i < BWD_CAND_DY_SLOTS; ++i) {
      mbar_init(&s.dy_full[i], 1);
      mbar_init(&s.dy_empty[i], 1 + (do_s ? CAND_EPI : 0));
    }
    for (int i = 0; i < BWD_CAND_C_SLOTS; ++i) {
      mbar_init(&s.st_full[i], 1);
      mbar_init(&s.st_empty[i], 1);
    }
    mbar_init(s.w_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.dc_full[i], 1);
      mbar_init(&s.dc_empty[i], 128);
    }
    mbar_init(s.wacc_full, 1);
    *s.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmDY);
    if (do_w) tma_prefetch_desc(&tmC);
    if (do_c) tma_prefetch_desc(&tmW);
  }
  if (warp == 2) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  if (warp == 2 && p.fused_finish && do_s && lane_id() < CF_PRE) {
    // idle until the end: look up this CTA's first finish tasks now (the
    // grid's CTAs are the finish's blocks)
    const int task = blockIdx.x + static_cast<int>(lane_id()) * gridDim.x;
    s.pre[lane_id()] = task < p.n_users * p.n_dh * CF_SLICES ? cand_task_bounds(p, task) : make_int4(-1, 0, 0, 0);
  }
  const long long nq = static_cast<long long>(p.n_dh) * p.n_cand;
  const long long q0 = cand_q0(nq, blockIdx.x, gridDim.x), q1 = cand_q0(nq, blockIdx.x + 1, gridDim.x);
  if (do_s) cand_empty_users(p);
  const int m_rows = p.n_mblk * 128;
  const uint32_t dy_bytes = static_cast<uint32_t>(p.kcn) * BOX;

  if (warp == 0) {
    // ---- TMA producer of W_c (once) and the dY blocks
    if (do_c && elect_one()) {
      mbar_arrive_expect_tx(s.w_full, static_cast<uint32_t>(p.kcn * m_rows) * 128u);
      for (int kc = 0; kc < p.kcn; ++kc)
        for (int r = 0; r < m_rows; r += 128)
          tma_load_2d(s.w + (static_cast<size_t>(kc) * m_rows + r) * 128, &tmW, s.w_full, kc * 64, r);
    }
    __syncwarp();
    CandWin win;
    SlotRing<BWD_CAND_DY_SLOTS> dyr;
    for (long long q = q0; q < q1; ++q, dyr.next()) {
      int b, u;
      cand_tile(p, q, q1, win, b, u);
      const int dh = static_cast<int>(q / p.n_cand);
      if (!warp_wait(&s.dy_empty[dyr.slot], dyr.phase ^ 1u, s.abort, p.timeout_ns)) goto done;
      if (elect_one()) {
        uint8_t* dst = s.dy + dyr.slot * CAND_DY_SLOT;
        mbar_arrive_expect_tx(&s.dy_full[dyr.slot], dy_bytes);
        for (int j = 0; j < p.kcn; ++j) tma_load_3d(dst + j * BOX, &tmDY, &s.dy_full[dyr.slot], dh * 64, 64 * j, b);
      }
      __syncwarp();
    }
  } else if (warp == 3) {
    // ---- TMA producer of the C slots (its own warp, so that C runs ahead of
    // dY by the depth of its ring)
    if (do_w) {
      CandWin win;
      SlotRing<BWD_CAND_C_SLOTS> ring;
      for (long long q = q0; q < q1; ++q) {
        int b, u;
        cand_tile(p, q, q1, win, b, u);
        const int dh = static_cast<int>(q / p.n_cand);
        for (int mb = 0; mb < p.n_mblk; ++mb, ring.next()) {
          if (!warp_wait(&s.st_empty[ring.slot], ring.phase ^ 1u, s.abort, p.timeout_ns)) goto done;
          if (elect_one()) {
            uint64_t* bar = &s.st_full[ring.slot];
            mbar_arrive_expect_tx(bar, CB_SLOT);
            tma_load_3d(s.ring + ring.slot * CB_SLOT, &tmC, bar, dh * 64, 128 * mb, b);
          }
          __syncwarp();
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer, per unit:
    //   dC^T block mb [K_c rows][64 d] = W_c block mb (A, K-major: n) x dY (B, MN-major: d), K = n
    //   dW_c block mb [K_c rows][n] += C slot (A, K-major: d) x dY (B, K-major: d), K = the unit's 64 d
    const uint32_t idesc_w = idesc_bf16_f32(128, static_cast<uint32_t>(p.n_mma), false, false);
    constexpr uint32_t idesc_c = idesc_bf16_f32(128, 64, false, true);
    const int csteps = 4 * p.kcn;
    SlotRing<BWD_CAND_DY_SLOTS> dyr;
    SlotRing<BWD_CAND_C_SLOTS> ring;
    if (do_c && !warp_wait(s.w_full, 0, s.abort, p.timeout_ns)) goto done;
    int t = 0;
    for (long long q = q0; q < q1; ++q, ++t, dyr.next()) {
      if (!warp_wait(&s.dy_full[dyr.slot], dyr.phase, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      const uint32_t dy_base = smem_u32(s.dy + dyr.slot * CAND_DY_SLOT);
      if (do_c) {
        for (int mb = 0; mb < p.n_mblk; ++mb) {
          const int c = t * p.n_mblk + mb;
          const int acc = c & 1;
          if (!warp_wait(&s.dc_empty[acc], ((c >> 1) & 1) ^ 1u, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          if (elect_one()) {
            // descriptors built once, then advanced by adding (offset >> 4) to
            // the start-address field (shared memory is below 256 KB: no carry)
            const uint64_t ad0 = sdesc_sw128(smem_u32(s.w) + static_cast<uint32_t>(mb * 128 * 128), 16, 1024u);
            const uint64_t bd0 = sdesc_sw128(dy_base, BOX, 1024u);
            const uint32_t a_chunk = static_cast<uint32_t>(m_rows * 128) >> 4;  // one 64-n chunk of W_c
            const uint32_t d_tmem = tmem + CAND_DC_COL + static_cast<uint32_t>(acc * 64);
#pragma unroll
            for (int st = 0; st < 12; ++st) {
              if (st < csteps) {
                const uint32_t aoff = static_cast<uint32_t>(st >> 2) * a_chunk + (((st & 3) * 32) >> 4);
                const uint32_t boff = static_cast<uint32_t>((st >> 2) * BOX + (st & 3) * 2048) >> 4;
                mma_bf16_ss(d_tmem, ad0 + aoff, bd0 + boff, idesc_c, st > 0 ? 1u : 0u);
              }
            }
            mma_commit(&s.dc_full[acc]);
          }
          __syncwarp();
        }
      }
      if (do_w) {
        for (int mb = 0; mb < p.n_mblk; ++mb, ring.next()) {
          if (!warp_wait(&s.st_full[ring.slot], ring.phase, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          if (elect_one()) {
            const uint64_t adesc = sdesc_sw128(smem_u32(s.ring + ring.slot * CB_SLOT), 16, 1024u);
            const uint64_t bdesc = sdesc_sw128(dy_base, 16, 1024u);
            const uint32_t d_tmem = tmem + static_cast<uint32_t>(mb * p.n_mma);
#pragma unroll
            for (int st = 0; st < 4; ++st)
              mma_bf16_ss(d_tmem, adesc + st * (32u >> 4), bdesc + st * (32u >> 4), idesc_w,
                          (t == 0 && st == 0) ? 0u : 1u);
            mma_commit(&s.st_empty[ring.slot]);
          }
          __syncwarp();
        }
      }
      if (elect_one()) mma_commit(&s.dy_empty[dyr.slot]);  // every product of this unit has read dY
      __syncwarp();
    }
    if (do_w && elect_one()) mma_commit(s.wacc_full);
    __syncwarp();
  } else if (warp >= 4) {
    // ---- epilogue: per unit the S sums, then this group's dC accumulators;
    // at the end the CTA's dW_c partial
    const int et = static_cast<int>(threadIdx.x) - 128;
    const int quarter = warp & 3, grp = (warp - 4) >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int pd = et & 31, ng = et >> 5;
    float acc[3][8][2];
#pragma unroll
    for (int j = 0; j < 3; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[j][i][0] = acc[j][i][1] = 0.f;
    if (do_s && lane_id() == 0) {  // this CTA's share of db starts at zero (rows of this warp)
#pragma unroll
      for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) s.dbsm[64 * j + 8 * ng + i] = 0.f;
    }
    // the open run of (user, D block) and its user's segment
    int run_u = -1, run_dh = -1, run_oa = 0, run_ob = 0;
    bool bad_seen = false;
    CandWin win;
    SlotRing<BWD_CAND_DY_SLOTS> dyr;
    int t = 0;
    for (long long q = q0; q < q1; ++q, ++t, dyr.next()) {
      int b, u, oa, ob;
      cand_tile<true>(p, q, q1, win, b, u, &oa, &ob);
      const int dh = static_cast<int>(q / p.n_cand);
      if (do_s) {
        if (!warp_wait(&s.dy_full[dyr.slot], dyr.phase, s.abort, p.timeout_ns)) goto done;
        if (u < 0) {  // out of range: in no user's sum (candidates after the valid ones in perm)
          bad_seen = true;
        } else {
          if (u != run_u || dh != run_dh) {
            if (run_u >= 0) {
              cand_flush(p, acc, run_u, run_dh, run_oa, run_ob, q0, nq, pd, ng, s.dbsm);
#pragma unroll
              for (int j = 0; j < 3; ++j)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[j][i][0] = acc[j][i][1] = 0.f;
            }
            run_u = u;
            run_dh = dh;
            run_oa = oa;
            run_ob = ob;
          }
          // this thread's 48 elements of the staged block: row n = 64 j + r
          // of chunk j, bytes 4 pd .. 4 pd + 3, 16-byte chunk swizzled by r % 8 = i
          const uint8_t* blk = s.dy + dyr.slot * CAND_DY_SLOT;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            if (j < p.kcn) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int r = 8 * ng + i;
                const uint32_t w = *reinterpret_cast<const uint32_t*>(
                    blk + j * BOX + r * 128 + ((((pd >> 2) ^ i) << 4) | ((pd & 3) << 2)));
                acc[j][i][0] += __uint_as_float(w << 16);
                acc[j][i][1] += __uint_as_float(w & 0xffff0000u);
              }
            }
          }
        }
        mbar_arrive(&s.dy_empty[dyr.slot]);
      }
      if (do_c) {
        for (int mb = 0; mb < p.n_mblk; ++mb) {
          const int c = t * p.n_mblk + mb;
          if ((c & 1) != grp) continue;
          if (!warp_wait(&s.dc_full[grp], (c >> 1) & 1, s.abort, p.timeout_ns)) goto done;
          tc_fence_after();
          uint32_t v0[32], v1[32];
          const uint32_t ta = tmem + lane_base + CAND_DC_COL + static_cast<uint32_t>(grp * 64);
          tmem_ld32(ta, v0);
          tmem_ld32(ta + 32, v1);
          tmem_ld_wait(v0);
          tmem_ld_wait(v1);
          tc_fence_before();
          mbar_arrive(&s.dc_empty[grp]);
          const int k = mb * 128 + quarter * 32 + static_cast<int>(lane_id());
          if (k < p.K_c) {
            // streaming stores: dC is written once and not read here, so it
            // should not push the S slots and dW_c partials out of L2
            uint16_t* dst = p.dC + (static_cast<size_t>(b) * p.K_c + k) * p.D + dh * 64;
            const int dlim = p.D - dh * 64;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              if (8 * h < dlim)
                __stcs(reinterpret_cast<uint4*>(dst + 8 * h),
                       make_uint4(pack_bf16x2(__uint_as_float(v0[8 * h]), __uint_as_float(v0[8 * h + 1])),
                                  pack_bf16x2(__uint_as_float(v0[8 * h + 2]), __uint_as_float(v0[8 * h + 3])),
                                  pack_bf16x2(__uint_as_float(v0[8 * h + 4]), __uint_as_float(v0[8 * h + 5])),
                                  pack_bf16x2(__uint_as_float(v0[8 * h + 6]), __uint_as_float(v0[8 * h + 7]))));
            }
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              if (32 + 8 * h < dlim)
                __stcs(reinterpret_cast<uint4*>(dst + 32 + 8 * h),
                       make_uint4(pack_bf16x2(__uint_as_float(v1[8 * h]), __uint_as_float(v1[8 * h + 1])),
                                  pack_bf16x2(__uint_as_float(v1[8 * h + 2]), __uint_as_float(v1[8 * h + 3])),
                                  pack_bf16x2(__uint_as_float(v1[8 * h + 4]), __uint_as_float(v1[8 * h + 5])),
                                  pack_bf16x2(__uint_as_float(v1[8 * h + 6]), __uint_as_float(v1[8 * h + 7]))));
            }
          }
        }
      }
    }
    if (do_s) {
      if (run_u >= 0) cand_flush(p, acc, run_u, run_dh, run_oa, run_ob, q0, nq, pd, ng, s.dbsm);
      if (bad_seen && et == 0) atomicOr(p.status, DEV_ERR_MAP_RANGE);
      if (lane_id() == 0) {  // this CTA's share of db, for the finish
#pragma unroll
        for (int j = 0; j < 3; ++j)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int n = 64 * j + 8 * ng + i;
            if (n < p.N) p.dbcta[static_cast<size_t>(blockIdx.x) * p.N + n] = s.dbsm[n];
          }
      }
    }
    // the CTA's dW_c partial, stored [n][K_c row of the block] so that each
    // store of the warp covers 32 consecutive rows (TMEM lane = row, column = n)
    if (do_w && q1 > q0) {
      if (!warp_wait(s.wacc_full, 0, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      const int row = quarter * 32 + static_cast<int>(lane_id());
      const int nchunks = (p.N + 31) / 32;
      for (int mb = 0; mb < p.n_mblk; ++mb) {
        float* out = p.wpart + static_cast<size_t>(mb * gridDim.x + blockIdx.x) * p.N * 128 + row;
        for (int c = grp; c < nchunks; c += 2) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(mb * p.n_mma + c * 32), v);
          tmem_ld_wait(v);
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (c * 32 + k < p.N) out[static_cast<size_t>(c * 32 + k) * 128] = __uint_as_float(v[k]);
        }
      }
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (*s.abort && threadIdx.x == 0) atomicOr(p.status, DEV_ERR_PIPE_TIMEOUT);
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (!p.fused_finish || !(do_w || do_s)) return;
  // grid barrier (every CTA is resident: cooperative launch), then the finish
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.ctrl, 1u);
    const uint64_t t0 = globaltimer_ns();
    bool ok = true;
    while (ld_acquire_gpu(p.ctrl) < gridDim.x) {
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        ok = false;
        atomicOr(p.status, DEV_ERR_PIPE_TIMEOUT);
        break;
      }
    }
    __threadfence();
    *s.flag = ok ? 1u : 0u;
  }
  __syncthreads();
  if (*s.flag == 0) return;
  // the pipeline's shared memory is free again: the finish's sums go there
  cand_finish(p, blockIdx.x, gridDim.x, reinterpret_cast<float*>(s.dy), s.pre);
  __syncthreads();
  // the last CTA out resets the barrier for the next call
  if (threadIdx.x == 0 && atomicAdd(p.ctrl + 1, 1u) == gridDim.x - 1) {
    p.ctrl[0] = 0;
    p.ctrl[1] = 0;
  }
}

__global__ void __launch_bounds__(CF_THREADS) bwd_cand_finish_kernel(const CandParams p) {
  __shared__ float4 red[(CF_RED + 3) / 4];
  cand_finish(p, blockIdx.x, gridDim.x, reinterpret_cast<float*>(red), nullptr);
}

}  // namespace

// ------------------------------------------------------------------- host
namespace {
constexpr size_t SMEM_ALIGN_PAD = 1024;
}

int bwd_segsum_chunks(int n_cand, int n_users, int ND, int num_sms) {
  const int slices = (ND + BWD_SEG_SLICE - 1) / BWD_SEG_SLICE;
  const long long tasks = static_cast<long long>(n_users) * slices;
  const long long target = 8ll * num_sms;  // enough threads per SM to keep HBM busy
  int nch = tasks >= target ? 1 : static_cast<int>((target + tasks - 1) / tasks);
  const int cap = n_cand / (16 * n_users);  // at least ~16 candidates per chunk
  if (nch > cap) nch = cap;
  return nch < 1 ? 1 : nch;
}

cudaError_t launch_bwd_segsum(const SegSumParams& p, cudaStream_t s, int* launches) {
  bwd_segsum_kernel<<<p.n_users * p.nch * p.slices, BWD_SEG_THREADS, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *launches += 1;
  if (p.nch > 1) {
    bwd_segsum_finish_kernel<<<p.n_users * p.slices, BWD_SEG_THREADS, 0, s>>>(p);
    e = cudaGetLastError();
    if (e == cudaSuccess) *launches += 1;
  }
  return e;
}

cudaError_t launch_bwd_db(const float* S, float* db, int n_users, int N, int D, cudaStream_t s) {
  bwd_db_kernel<<<N, BWD_DB_THREADS, 0, s>>>(S, db, n_users, N, D);
  return cudaGetLastError();
}

// The candidate pass (see CandParams): false where it does not apply.
bool bwd_cand_configure(CandParams* p, size_t max_smem) {
  if (p->K_c < 1 || p->K_c > BWD_CAND_MAX_KC || p->N < 1 || p->N > BWD_CAND_MAX_N || p->D < 1) return false;
  if (CAND_SMEM > max_smem) return false;
  p->n_dh = (p->D + 63) / 64;
  p->kcn = (p->N + 63) / 64;
  p->n_mblk = (p->K_c + 127) / 128;
  p->n_mma = (p->N + 15) / 16 * 16;
  return true;
}

int bwd_cand_grid(const CandParams& p, int num_sms) {
  const long long nq = static_cast<long long>(p.n_dh) * p.n_cand;
  long long g = nq < num_sms ? nq : num_sms;
  if (g > CF_CHUNKS * CF_MAX_PER_CHUNK) g = CF_CHUNKS * CF_MAX_PER_CHUNK;  // the finish's chunks
  return static_cast<int>(g);
}

// p.G CTAs.  With a finish (dW_c, S), as one cooperative launch that ends
// with it when `cooperative`; where that is refused (not all CTAs can be
// resident) or not asked for, the pass and then the finish kernel.
// *launches receives the number of kernels.
cudaError_t launch_bwd_cand(const CUtensorMap& tmDY, const CUtensorMap& tmC, const CUtensorMap& tmW,
                            const CandParams& p, int num_sms, bool cooperative, cudaStream_t s, int* launches) {
  cudaError_t e = cudaFuncSetAttribute(bwd_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(CAND_SMEM));
  if (e != cudaSuccess) return e;
  const bool finish = p.wpart != nullptr || p.S2 != nullptr;
  CandParams q = p;
  q.fused_finish = 0;
  if (finish && cooperative) {
    q.fused_finish = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.G));
    cfg.blockDim = dim3(BWD_THREADS);
    cfg.dynamicSmemBytes = CAND_SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bwd_cand_kernel, tmDY, tmC, tmW, q);
    if (e == cudaSuccess) {
      *launches = 1;
      return e;
    }
    if (e != cudaErrorCooperativeLaunchTooLarge) return e;
    (void)cudaGetLastError();
    q.fused_finish = 0;
  }
  bwd_cand_kernel<<<p.G, BWD_THREADS, CAND_SMEM, s>>>(tmDY, tmC, tmW, q);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *launches = 1;
  if (!finish) return e;
  bwd_cand_finish_kernel<<<num_sms, CF_THREADS, 0, s>>>(q);
  e = cudaGetLastError();
  if (e == cudaSuccess) *launches = 2;
  return e;
}


size_t bwd_act_smem(const ActParams& p) {
  return SMEM_ALIGN_PAD + act_w_bytes(p.kc, p.m_rows) + static_cast<size_t>(p.stages) * 2 * BOX +
         sizeof(uint64_t) * (2 * p.stages + 1 + 4) + 2 * sizeof(uint32_t);
}

// Fills the derived fields from B, M, D, N; `pair`: X holds a hi/lo pair
// (2 * kc chunks per b).  With `split`, when the tiles are fewer than the
// SMs even with M split into 128-row blocks, each CTA takes one (tile, M
// block) and keeps only that block of W (a third of the weight at K_u = 381,
// and three times the CTAs).  False for shapes it cannot run.
bool bwd_act_configure(ActParams* p, size_t max_smem, bool pair, int num_sms, bool split) {
  if (p->B < 1 || p->M < 1 || p->D < 1 || p->N < 1) return false;
  p->n_dblk = (p->D + 127) / 128;
  p->kc = (p->N + 63) / 64;
  p->m_pad = (p->M + 15) / 16 * 16;
  p->m_rows = (p->M + 127) / 128 * 128;
  p->n_mgrp = 1;
  const int mblocks = p->m_rows / 128;
  if (split && mblocks > 1 && static_cast<long long>(p->B) * p->n_dblk * mblocks <= num_sms) {
    p->n_mgrp = mblocks;
    p->m_rows = 128;
    p->m_pad = 128;
  }
  p->bufs = p->m_pad <= 256 ? 2 : 1;
  p->kcx = pair ? 2 * p->kc : p->kc;
  if (p->m_pad > 512) return false;
  p->stages = BWD_ACT_MAX_STAGES;
  while (p->stages > 2 && bwd_act_smem(*p) > max_smem) --p->stages;
  return bwd_act_smem(*p) <= max_smem;
}

cudaError_t launch_bwd_act(const CUtensorMap& tmX, const CUtensorMap& tmW, const ActParams& p, int num_sms,
                           cudaStream_t s) {
  const size_t smem = bwd_act_smem(p);
  cudaError_t e =
      cudaFuncSetAttribute(bwd_act_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long tiles = static_cast<long long>(p.B) * p.n_dblk * p.n_mgrp;
  const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
  bwd_act_kernel<<<grid, BWD_THREADS, smem, s>>>(tmX, tmW, p);
  return cudaGetLastError();
}

size_t bwd_wgrad_smem(const WgradParams& p) {
  return SMEM_ALIGN_PAD + static_cast<size_t>(p.stages) * wg_stage_bytes(p.mg, p.nb) +
         sizeof(uint64_t) * (2 * p.stages + 2) + 2 * sizeof(uint32_t);
}

bool bwd_wgrad_configure(WgradParams* p, int num_sms, size_t max_smem) {
  if (p->B < 1 || p->M < 1 || p->D < 1 || p->N < 1 || p->N > 256) return false;
  p->n_mblk = (p->M + 127) / 128;
  // One m block per unit: grouping two blocks per unit (one G load serving
  // both) doubles the b ranges and so the fp32 partials, and measured slower
  // at the 70:1 shape (dW_c: the second read of dY mostly hits L2 anyway).
  p->mg = 1;
  p->n_mgrp = (p->n_mblk + p->mg - 1) / p->mg;
  // b ranges: enough to fill the SMs, but at least two batches each (fewer
  // partials for the reduce; measured 132.7 vs 134.8 us for the LCE backward
  // at the 70:1 shape, where dW_u's 2 n_users batches would give one each)
  int R = num_sms / p->n_mgrp;
  if (R > p->B / 2) R = p->B / 2;
  if (R < 1) R = 1;
  p->R = R;
  p->dc = (p->D + 63) / 64;
  p->n_mma = (p->N + 15) / 16 * 16;
  p->nb = (p->n_mma + 63) / 64;
  p->stages = BWD_WG_MAX_STAGES;
  while (p->stages > 2 && bwd_wgrad_smem(*p) > max_smem) --p->stages;
  return bwd_wgrad_smem(*p) <= max_smem;
}

size_t bwd_wgrad_part_elems(const WgradParams& p) {
  return static_cast<size_t>(p.n_mblk) * p.R * 128 * p.N;
}

// The split-K kernel (partials into p.part) and the in-order reduce into dW.
// With mg == 1, R <= 16 and the R CTAs of an m block co-schedulable as a
// cluster, one launch (the partials are added through distributed shared
// memory); else the partials kernel and the reduce kernel.
cudaError_t launch_bwd_wgrad(const CUtensorMap& tmA, const CUtensorMap& tmG, const WgradParams& p, float* dW,
                             int num_sms, cudaStream_t s, int* launches) {
  const size_t smem = bwd_wgrad_smem(p);
  cudaError_t e =
      cudaFuncSetAttribute(bwd_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int units = p.n_mgrp * p.R;
  const size_t red_bytes = static_cast<size_t>(128) * (p.n_mma + 1) * sizeof(float);
  if (p.mg == 1 && p.R >= 2 && p.R <= 16 && red_bytes <= static_cast<size_t>(p.stages) * wg_stage_bytes(p.mg, p.nb)) {
    WgradParams q = p;
    q.cluster = 1;
    q.dW = dW;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units));
    cfg.blockDim = dim3(BWD_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.R);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    if ((p.R <= 8 || cudaFuncSetAttribute(bwd_wgrad_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
                         cudaSuccess) &&
        cudaOccupancyMaxActiveClusters(&active, bwd_wgrad_kernel, &cfg) == cudaSuccess && active >= 1) {
      e = cudaLaunchKernelEx(&cfg, bwd_wgrad_kernel, tmA, tmG, q);
      if (e == cudaSuccess) *launches += 1;
      return e;
    }
    (void)cudaGetLastError();  // no cluster of that size fits: partials and the reduce kernel
  }
  WgradParams q = p;
  q.cluster = 0;
  bwd_wgrad_kernel<<<units < num_sms ? units : num_sms, BWD_THREADS, smem, s>>>(tmA, tmG, q);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int total = p.M * p.N;
  bwd_wgrad_reduce_kernel<<<(total + WG_RED_OUT - 1) / WG_RED_OUT, dim3(WG_RED_OUT, WG_RED_SPLIT), 0, s>>>(
      p.part, dW, p.M, p.N, p.R);
  e = cudaGetLastError();
  if (e == cudaSuccess) *launches += 2;
  return e;
}

}  // namespace ikbo
