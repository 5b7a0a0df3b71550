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
//   bwd_segsum_kernel / bwd_segsum_finish_kernel  S (HBM-bound reduction)
//   bwd_db_kernel                                 db from S
//   bwd_act_kernel     out[b][m][d] = sum_n W[m][n] X[b][n][d]   (dC, dU)
//   bwd_wgrad_kernel   split-K partials of sum_b sum_d A[b][m][d] G[b][n][d]
//   bwd_wgrad_reduce_kernel                       (dW_c, dW_u)
// The two GEMM kernels are persistent, one CTA per SM, warp-specialised like
// the forward: warp 0 TMA (elected lane issues), warp 1 tcgen05.mma (elected
// lane), warp 2 TMEM owner, warps 4-11 epilogue.  Every wait is bounded.
#include <cuda_bf16.h>

#include "ikbo_internal.h"
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

// Tiles q = dblk * B + b (D-block-major); each CTA takes one contiguous range.
__device__ __forceinline__ void act_range(const ActParams& p, int& q0, int& q1) {
  const long long nq = static_cast<long long>(p.B) * p.n_dblk;
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
    // ---- TMA producer: W once, then the X chunks of every tile
    if (elect_one()) {
      mbar_arrive_expect_tx(s.w_full, act_w_bytes(p.kc, p.m_rows));
      for (int kc = 0; kc < p.kc; ++kc)
        for (int r = 0; r < p.m_rows; r += 128)
          tma_load_2d(s.w + (static_cast<size_t>(kc) * p.m_rows + r) * 128, &tmW, s.w_full, kc * 64, r);
    }
    __syncwarp();
    int stage = 0;
    uint32_t phase = 0;
    for (int q = q0; q < q1; ++q) {
      const int dblk = q / p.B, b = q - dblk * p.B;
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
    const int nchunks = (p.M + 31) / 32;
    for (int q = q0, t = 0; q < q1; ++q, ++t) {
      const int dblk = q / p.B, b = q - dblk * p.B;
      const int buf = p.bufs == 2 ? (t & 1) : 0;
      const uint32_t use = static_cast<uint32_t>(p.bufs == 2 ? (t >> 1) : t);
      if (!warp_wait(&s.acc_full[buf], use & 1u, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      const int d = dblk * 128 + quarter * 32 + static_cast<int>(lane_id());
      const bool dok = d < p.D;
      __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(b) * p.M * p.D + d;
      for (int c = half; c < nchunks; c += 2) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + static_cast<uint32_t>(buf * 256 + c * 32), v);
        tmem_ld_wait(v);
        __nv_bfloat16* o = out + static_cast<size_t>(c * 32) * p.D;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (c * 32 + j < p.M && dok) *o = __float2bfloat16_rn(__uint_as_float(v[j]));
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
// See CandParams.  Per CTA (one per SM, 12 warps): warp 0 TMA producer,
// warp 1 MMA issuer, warp 2 TMEM owner, warps 4-11 epilogue (S sums).
// Tiles q = dblk * n_cand + pos (D-block-major over the plan's grouped
// order), one contiguous range per CTA, so a CTA's consecutive tiles share a
// user and its S sums stay in registers.
// TMEM columns: dW_c block 0 [0, n_mma), block 1 [n_mma, 2 n_mma) (lanes =
// K_c rows, columns = n), accumulated over the CTA's tiles.
// Shared memory: two dY tile slots, each [d half][n rows][64 d] (128-byte
// rows, 128-byte swizzle), read K-major as dW_c's B; then the ring of 16 KB
// C slots, per tile one per (128-row block of K_c, 64-d half).
constexpr uint32_t CB_SLOT = 128 * 64 * 2;  // 16 KB: 128 rows x 64 bf16
constexpr uint32_t CB_DYHALF = 3 * BOX;     // one d half of a dY tile (<= 192 n rows)
constexpr uint32_t CAND_TILES = 2 * BWD_CAND_DY_BYTES + BWD_CAND_SLOTS * CB_SLOT;
constexpr int CAND_BARS = 4 + 2 * BWD_CAND_SLOTS + 1;
constexpr size_t CAND_SMEM = 1024 + CAND_TILES + 8 * CAND_BARS + 8;
static_assert(CAND_SMEM <= 227 * 1024, "candidate pass does not fit in shared memory");

struct CandSmem {
  uint8_t* dy;
  uint8_t* ring;
  uint64_t* dy_full;   // [2]
  uint64_t* dy_empty;  // [2] MMA reads done (commit) and the S sums taken
  uint64_t* st_full;   // [SLOTS]
  uint64_t* st_empty;  // [SLOTS]
  uint64_t* w_full;    // the CTA's dW_c partial is complete in TMEM
  uint32_t* tmem_slot;
  uint32_t* abort;
};

__device__ __forceinline__ CandSmem cand_carve(uint8_t* base) {
  CandSmem s;
  s.dy = base;
  s.ring = base + 2 * BWD_CAND_DY_BYTES;
  uint64_t* b = reinterpret_cast<uint64_t*>(base + CAND_TILES);
  s.dy_full = b;
  s.dy_empty = b + 2;
  s.st_full = b + 4;
  s.st_empty = s.st_full + BWD_CAND_SLOTS;
  s.w_full = s.st_empty + BWD_CAND_SLOTS;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.w_full + 1);
  s.abort = s.tmem_slot + 1;
  return s;
}

__device__ __forceinline__ void cand_range(const CandParams& p, long long& q0, long long& q1) {
  const long long nq = static_cast<long long>(p.n_dblk) * p.n_cand;
  q0 = blockIdx.x * nq / gridDim.x;
  q1 = (blockIdx.x + 1) * nq / gridDim.x;
}

// The candidate (and its user, -1 if out of range) of tile q, looked up by
// the warp 32 tiles at a time: lane l holds tile wbase + l.
struct CandWin {
  long long base = -1;
  int b = 0, u = -1;
};
__device__ __forceinline__ void cand_tile(const CandParams& p, long long q, long long q1, CandWin& w, int& b, int& u) {
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
    }
  }
  const int k = static_cast<int>(q - w.base);
  b = __shfl_sync(0xffffffffu, w.b, k);
  u = __shfl_sync(0xffffffffu, w.u, k);
}

struct SlotRing {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == BWD_CAND_SLOTS) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// S sums of a run (user u, D block dblk) of this CTA: the run inside the
// CTA's range goes straight to S; the range's first run to partial slot 0,
// its last (when another) to slot 1.  Thread: d pair 2pd, 2pd+1 of the block,
// rows n = 64 j + 16 ng + i.
__device__ __forceinline__ void cand_flush(const CandParams& p, const float (&acc)[3][16][2], int u, int dblk,
                                           int slot, int pd, int ng) {
  const int d = 2 * pd;
  const bool dok = dblk * 128 + d < p.D;  // D is a multiple of 8: both of the pair or neither
#pragma unroll
  for (int j = 0; j < 3; ++j)
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int n = 64 * j + 16 * ng + i;
      if (n >= p.N || !dok) continue;
      float2* dst = slot < 0 ? reinterpret_cast<float2*>(p.S + (static_cast<size_t>(u) * p.N + n) * p.D + dblk * 128 + d)
                             : reinterpret_cast<float2*>(p.spart +
                                                         ((static_cast<size_t>(blockIdx.x) * 2 + slot) * p.N + n) * 128 + d);
      *dst = make_float2(acc[j][i][0], acc[j][i][1]);
    }
}

__global__ void __launch_bounds__(BWD_THREADS, 1)
    bwd_cand_kernel(const __grid_constant__ CUtensorMap tmDY, const __grid_constant__ CUtensorMap tmC,
                    const CandParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const CandSmem s = cand_carve(base);
  const int warp = threadIdx.x >> 5;
  const bool do_s = p.S != nullptr;
  const bool do_w = p.wpart != nullptr;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.dy_full[i], 1);
      mbar_init(&s.dy_empty[i], 1 + (do_s ? BWD_THREADS - 128 : 0));
    }
    for (int i = 0; i < BWD_CAND_SLOTS; ++i) {
      mbar_init(&s.st_full[i], 1);
      mbar_init(&s.st_empty[i], 1);
    }
    mbar_init(s.w_full, 1);
    *s.abort = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane_id() == 0) {
    tma_prefetch_desc(&tmDY);
    if (do_w) tma_prefetch_desc(&tmC);
  }
  if (warp == 2) {
    tmem_alloc(s.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s.tmem_slot;
  long long q0, q1;
  cand_range(p, q0, q1);
  if (threadIdx.x == 0 && do_s) {  // the range, for the S finish
    p.bounds[blockIdx.x] = q0;
    if (blockIdx.x + 1 == gridDim.x) p.bounds[gridDim.x] = q1;
  }
  const int nc = do_w ? 2 * p.n_mblk : 0;  // C slots per tile
  const uint32_t dy_bytes = static_cast<uint32_t>(2 * p.kcn) * BOX;

  if (warp == 0) {
    // ---- TMA producer: the dY tile into its slot, then the tile's C slots
    CandWin win;
    SlotRing ring;
    int t = 0;
    for (long long q = q0; q < q1; ++q, ++t) {
      int b, u;
      cand_tile(p, q, q1, win, b, u);
      const int dblk = static_cast<int>(q / p.n_cand);
      const int y = t & 1;
      if (!warp_wait(&s.dy_empty[y], ((t >> 1) & 1) ^ 1u, s.abort, p.timeout_ns)) goto done;
      if (elect_one()) {
        uint8_t* dst = s.dy + y * BWD_CAND_DY_BYTES;
        mbar_arrive_expect_tx(&s.dy_full[y], dy_bytes);
        for (int h = 0; h < 2; ++h)
          for (int j = 0; j < p.kcn; ++j)
            tma_load_3d(dst + h * CB_DYHALF + j * BOX, &tmDY, &s.dy_full[y], dblk * 128 + 64 * h, 64 * j, b);
      }
      __syncwarp();
      for (int c = 0; c < nc; ++c, ring.next()) {  // C block c / 2, d half c % 2
        if (!warp_wait(&s.st_empty[ring.slot], ring.phase ^ 1u, s.abort, p.timeout_ns)) goto done;
        if (elect_one()) {
          uint64_t* bar = &s.st_full[ring.slot];
          mbar_arrive_expect_tx(bar, CB_SLOT);
          tma_load_3d(s.ring + ring.slot * CB_SLOT, &tmC, bar, dblk * 128 + 64 * (c & 1), 128 * (c >> 1), b);
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer: dW_c[m][n] += C[b][m][d] dY[b][n][d]; A = the C slot
    // (K-major), B = a dY d half (K-major, n rows), 4 steps of 16 d per slot
    SlotRing ring;
    const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(p.n_mma), false, false);
    int t = 0;
    for (long long q = q0; q < q1; ++q, ++t) {
      const int y = t & 1;
      if (!warp_wait(&s.dy_full[y], (t >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      const uint32_t dy_base = smem_u32(s.dy + y * BWD_CAND_DY_BYTES);
      for (int c = 0; c < nc; ++c, ring.next()) {
        if (!warp_wait(&s.st_full[ring.slot], ring.phase, s.abort, p.timeout_ns)) goto done;
        tc_fence_after();
        if (elect_one()) {
          const uint64_t adesc = sdesc_sw128(smem_u32(s.ring + ring.slot * CB_SLOT), 16, 1024u);
          const uint64_t bdesc = sdesc_sw128(dy_base + (c & 1) * CB_DYHALF, 16, 1024u);
          const uint32_t d_tmem = tmem + static_cast<uint32_t>((c >> 1) * p.n_mma);
#pragma unroll
          for (int st = 0; st < 4; ++st)
            mma_bf16_ss(d_tmem, adesc + st * (32u >> 4), bdesc + st * (32u >> 4), idesc,
                        (t == 0 && (c & 1) == 0 && st == 0) ? 0u : 1u);
          mma_commit(&s.st_empty[ring.slot]);
        }
        __syncwarp();
      }
      if (elect_one()) mma_commit(&s.dy_empty[y]);  // every product of this tile has read dY
      __syncwarp();
    }
    if (elect_one()) mma_commit(s.w_full);
    __syncwarp();
  } else if (warp >= 4) {
    // ---- epilogue: the S sums, then the CTA's dW_c partial
    const int et = static_cast<int>(threadIdx.x) - 128;
    const int quarter = warp & 3, half = (warp - 4) >> 2;
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const int pd = et & 63, ng = et >> 6;  // S: d pair, group of 16 n rows in each 64-n chunk
    if (do_s) {
      float acc[3][16][2];
#pragma unroll
      for (int j = 0; j < 3; ++j)
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[j][i][0] = acc[j][i][1] = 0.f;
      // the open run of (user, D block); whether it holds the range's first
      // tile (its sums go to slot 0) and whether the last tile seen was in it
      int run_u = -2, run_dblk = -1;
      bool run_first = false, last_in_run = false, bad_seen = false;
      CandWin win;
      int t = 0;
      for (long long q = q0; q < q1; ++q, ++t) {
        int b, u;
        cand_tile(p, q, q1, win, b, u);
        const int dblk = static_cast<int>(q / p.n_cand);
        const int y = t & 1;
        if (!warp_wait(&s.dy_full[y], (t >> 1) & 1u, s.abort, p.timeout_ns)) goto done;
        if (u < 0) {  // out of range: in no user's sum (candidates after the valid ones in perm)
          bad_seen = true;
          last_in_run = false;
        } else {
          if (u != run_u || dblk != run_dblk) {
            if (run_u >= 0) {  // a run ends inside the range: slot 0 if it held the first tile, else S
              cand_flush(p, acc, run_u, run_dblk, run_first ? 0 : -1, pd, ng);
#pragma unroll
              for (int j = 0; j < 3; ++j)
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[j][i][0] = acc[j][i][1] = 0.f;
            }
            run_first = q == q0;
          }
          run_u = u;
          run_dblk = dblk;
          last_in_run = true;
          // this thread's 96 elements of the staged tile: d half pd / 32,
          // byte (2 pd % 64) * 2 of row n, 16-byte chunk swizzled by n % 8
          const uint8_t* tile = s.dy + y * BWD_CAND_DY_BYTES + (pd >> 5) * CB_DYHALF;
          const int dd = (2 * pd) & 63;
#pragma unroll
          for (int j = 0; j < 3; ++j) {
            if (j < p.kcn) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int n = 64 * j + 16 * ng + i;
                const uint32_t w = *reinterpret_cast<const uint32_t*>(
                    tile + n * 128 + ((((dd >> 3) ^ (n & 7)) << 4) | ((dd & 7) << 1)));
                acc[j][i][0] += __uint_as_float(w << 16);
                acc[j][i][1] += __uint_as_float(w & 0xffff0000u);
              }
            }
          }
        }
        mbar_arrive(&s.dy_empty[y]);
      }
      // the open run: slot 0 if it held the first tile; else slot 1 if it runs
      // past the range's end (its last tile was the range's), else S
      if (run_u >= 0) cand_flush(p, acc, run_u, run_dblk, run_first ? 0 : (last_in_run ? 1 : -1), pd, ng);
      if (bad_seen && et == 0) atomicOr(p.status, DEV_ERR_MAP_RANGE);
    }
    // the CTA's dW_c partial: TMEM lane = K_c row of a block, columns = n
    if (do_w && q1 > q0) {
      if (!warp_wait(s.w_full, 0, s.abort, p.timeout_ns)) goto done;
      tc_fence_after();
      const int row = quarter * 32 + static_cast<int>(lane_id());
      const int nchunks = (p.N + 31) / 32;
      for (int mb = 0; mb < p.n_mblk; ++mb) {
        float* out = p.wpart + (static_cast<size_t>(mb * gridDim.x + blockIdx.x) * 128 + row) * p.N;
        for (int c = half; c < nchunks; c += 2) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_base + static_cast<uint32_t>(mb * p.n_mma + c * 32), v);
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

// S of (user u, D block dblk, slice of N x 128 elements): the run's tiles
// [a, a + cnt) in q order; a run inside one CTA's range that is neither its
// first nor its last run was stored straight to S; otherwise the partial
// slots of the CTAs that share it are added in CTA order (slot 0 where the
// run holds the CTA's first tile, else slot 1).  Then the hi/lo pair.
constexpr int SF_THREADS = 256;
constexpr int SF_ELEMS = 4 * SF_THREADS;  // elements per block
constexpr int SF_MAX_CTAS = 1024;  // contributors a run may have (the grid never exceeds the SM count)
__global__ void __launch_bounds__(SF_THREADS) bwd_sfinish_kernel(const SFinishParams p) {
  __shared__ int c_lo, c_n, c_direct;
  __shared__ uint32_t c_slot[SF_MAX_CTAS / 32];  // bit k: contributor c_lo + k reads slot 1
  const int elems = p.N * 128;
  const int slices = (elems + SF_ELEMS - 1) / SF_ELEMS;
  const int sl = blockIdx.x % slices;
  const int ud = blockIdx.x / slices;
  const int u = ud / p.n_dblk, dblk = ud - u * p.n_dblk;
  if (u >= p.n_users) return;  // uniform over the block
  const long long a = static_cast<long long>(dblk) * p.n_cand + __ldg(p.offsets + u);
  const long long e = static_cast<long long>(dblk) * p.n_cand + __ldg(p.offsets + u + 1);
  // the run's contributing CTAs and the slot each holds it in, once per
  // block: every thread tests the ranges [bounds[k], bounds[k + 1]) at once
  if (threadIdx.x == 0) {
    c_lo = 0;
    c_n = 0;
    c_direct = 0;
  }
  __syncthreads();
  if (e > a) {
    int c1 = -1;
    for (int k = static_cast<int>(threadIdx.x); k < p.G; k += SF_THREADS) {
      const long long b0 = __ldg(p.bounds + k), b1 = __ldg(p.bounds + k + 1);
      if (b0 <= a && a < b1) {
        c_lo = k;
        if (a > b0 && e < b1) c_direct = 1;  // inside one range, neither its first nor its last run: S already
      }
      if (b0 <= e - 1 && e - 1 < b1) c1 = k;
    }
    __syncthreads();
    if (c1 >= 0) c_n = c1 - c_lo + 1;
  }
  __syncthreads();
  const int nc = c_n;
  for (int w = static_cast<int>(threadIdx.x); w < (nc + 31) / 32; w += SF_THREADS) c_slot[w] = 0;
  __syncthreads();
  for (int k = static_cast<int>(threadIdx.x); k < nc; k += SF_THREADS)
    if (a > __ldg(p.bounds + c_lo + k)) atomicOr(&c_slot[k >> 5], 1u << (k & 31));
  __syncthreads();
  for (int r = 0; r < SF_ELEMS / SF_THREADS; ++r) {
    const int idx = sl * SF_ELEMS + r * SF_THREADS + static_cast<int>(threadIdx.x);
    if (idx >= elems) break;
    const int n = idx >> 7, dl = idx & 127;
    const int d = dblk * 128 + dl;
    if (d >= p.D) continue;
    float* Sp = p.S + (static_cast<size_t>(u) * p.N + n) * p.D + d;
    float v = 0.f;
    if (c_direct) {
      v = *Sp;
    } else {
      // the contributors' values, loaded 8 at a time, then added in CTA order
      const float* base = p.spart + static_cast<size_t>(n) * 128 + dl;
      const size_t slot_stride = static_cast<size_t>(p.N) * 128;
      for (int k0 = 0; k0 < nc; k0 += 8) {
        float w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int k = k0 + j;
          const int slot = k < nc ? static_cast<int>((c_slot[k >> 5] >> (k & 31)) & 1u) : 0;
          w[j] = k < nc ? __ldg(base + (static_cast<size_t>(c_lo + k) * 2 + slot) * slot_stride) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (k0 + j < nc) v += w[j];
      }
      *Sp = v;  // 0 for a user without candidates
    }
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    uint16_t* s2 = p.S2 + static_cast<size_t>(u) * 2 * p.NPD + static_cast<size_t>(n) * p.D + d;
    s2[0] = __bfloat16_as_ushort(hi);
    s2[p.NPD] = __bfloat16_as_ushort(lo);
  }
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
  p->n_dblk = (p->D + 127) / 128;
  p->kcn = (p->N + 63) / 64;
  p->n_mblk = (p->K_c + 127) / 128;
  p->n_mma = (p->N + 15) / 16 * 16;
  return true;
}

int bwd_cand_grid(const CandParams& p, int num_sms) {
  const long long nq = static_cast<long long>(p.n_dblk) * p.n_cand;
  return static_cast<int>(nq < num_sms ? nq : num_sms);
}

cudaError_t launch_bwd_cand(const CUtensorMap& tmDY, const CUtensorMap& tmC, const CandParams& p, int grid,
                            cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(bwd_cand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(CAND_SMEM));
  if (e != cudaSuccess) return e;
  bwd_cand_kernel<<<grid, BWD_THREADS, CAND_SMEM, s>>>(tmDY, tmC, p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_sfinish(const SFinishParams& p, cudaStream_t s) {
  const int slices = (p.N * 128 + SF_ELEMS - 1) / SF_ELEMS;
  bwd_sfinish_kernel<<<p.n_users * p.n_dblk * slices, SF_THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

// The in-order reduce of split-K partials part[(mblk * R + r) * 128 + row][n] into dW.
cudaError_t launch_bwd_wreduce(const float* part, float* dW, int M, int N, int R, cudaStream_t s) {
  const int total = M * N;
  bwd_wgrad_reduce_kernel<<<(total + WG_RED_OUT - 1) / WG_RED_OUT, dim3(WG_RED_OUT, WG_RED_SPLIT), 0, s>>>(part, dW,
                                                                                                       M, N, R);
  return cudaGetLastError();
}

size_t bwd_act_smem(const ActParams& p) {
  return SMEM_ALIGN_PAD + act_w_bytes(p.kc, p.m_rows) + static_cast<size_t>(p.stages) * 2 * BOX +
         sizeof(uint64_t) * (2 * p.stages + 1 + 4) + 2 * sizeof(uint32_t);
}

// Fills the derived fields from B, M, D, N; `pair`: X holds a hi/lo pair
// (2 * kc chunks per b).  False for shapes it cannot run.
bool bwd_act_configure(ActParams* p, size_t max_smem, bool pair) {
  if (p->B < 1 || p->M < 1 || p->D < 1 || p->N < 1) return false;
  p->n_dblk = (p->D + 127) / 128;
  p->kc = (p->N + 63) / 64;
  p->m_pad = (p->M + 15) / 16 * 16;
  p->m_rows = (p->M + 127) / 128 * 128;
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
  const long long tiles = static_cast<long long>(p.B) * p.n_dblk;
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
  int R = num_sms / p->n_mgrp;
  if (R < 1) R = 1;
  if (R > p->B) R = p->B;
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
cudaError_t launch_bwd_wgrad(const CUtensorMap& tmA, const CUtensorMap& tmG, const WgradParams& p, float* dW,
                             int num_sms, cudaStream_t s, int* launches) {
  const size_t smem = bwd_wgrad_smem(p);
  cudaError_t e =
      cudaFuncSetAttribute(bwd_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int units = p.n_mgrp * p.R;
  bwd_wgrad_kernel<<<units < num_sms ? units : num_sms, BWD_THREADS, smem, s>>>(tmA, tmG, p);
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
