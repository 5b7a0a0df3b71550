/*
 * ikbo.h -- C ABI of the GB300 (sm_103a) In-Kernel Broadcast Optimization
 * (IKBO) hot path.
 *
 * IKBO ("Meta Optimizes Inference for Recommendation Systems", RO/NRO and
 * Type I / Type II paragraphs; aixai.ru, "Почему broadcast — это проблема
 * раскладки данных"): an interaction operator takes the request-only (user)
 * tensors at their own batch n_users, the per-candidate tensors at n_cand,
 * and a candidate->user map, and never materialises the user tensors
 * replicated to n_cand -- not in memory, not on the bus, not in cache.
 *
 * Two operators are provided:
 *   - Linear Compression Embedding (LCE, Type I, decomposable):
 *       Y[i] = W_u^T U[map[i]] + W_c^T C[i] + b
 *   - broadcast attention (Type II, broadcast inside the kernel):
 *       O[i,h] = softmax(Q[i,h] K[map[i],h]^T * scale) V[map[i],h]
 *
 * Conventions for every entry point:
 *   - All tensor arguments are DEVICE pointers to row-major, contiguous
 *     memory owned by the caller; bf16 tensors are passed as `const void*`
 *     (IEEE bfloat16 bit patterns), integer tensors as int32.  Every tensor
 *     pointer must be 16-byte aligned (TMA requirement).
 *   - Every call is asynchronous and ordered on the given CUDA stream; no
 *     call synchronises except ikbo_plan_get_status and ikbo_plan_destroy.
 *   - Arguments are validated before any launch; a rejected call launches
 *     nothing and returns an error code.  No exception crosses the ABI and
 *     no kernel traps: errors detected on the device (a map value out of
 *     range, a bounded wait that ran out) are recorded in the plan's status
 *     word and returned by ikbo_plan_get_status.
 *   - One plan must not be used by two streams at the same time.
 *   - Device: one GPU of compute capability 10.3 (sm_103a), the device that
 *     is current when the plan is created.
 */
#ifndef IKBO_H
#define IKBO_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  IKBO_OK = 0,
  IKBO_ERR_INVALID_ARG = 1,       /* null pointer, non-positive size, size above the plan's maximum, misalignment */
  IKBO_ERR_UNSUPPORTED = 2,       /* legal but not implemented: d != 128, D or N not a multiple of 8, ... */
  IKBO_ERR_CUDA = 3,              /* a CUDA runtime / driver call failed (launch, allocation, tensor map) */
  IKBO_ERR_MAP_OUT_OF_RANGE = 4,  /* device-detected: some map[i] outside [0, n_users) */
  IKBO_ERR_TIMEOUT = 5,           /* device-detected: a bounded wait inside a kernel gave up */
  IKBO_ERR_NOT_PLANNED = 6,       /* forward called before ikbo_plan */
  IKBO_ERR_INTERNAL = 7           /* device-detected: inconsistent work list */
} ikbo_status_t;

/* Opaque plan: owns the segment arrays, the attention work list, the fp32
 * user-partial workspace of LCE, its readiness flags and the status word. */
typedef struct ikbo_plan_s* ikbo_plan_t;

/* Create a plan for requests of at most max_cand candidates, max_users users
 * and max_heads attention heads (each >= 1; max_users <= 8192).  Allocates
 * the plan's device memory on the current device (synchronous allocation).
 * On success *out receives the plan; on failure *out is set to NULL. */
ikbo_status_t ikbo_plan_create(ikbo_plan_t* out, int max_cand, int max_users, int max_heads);

/* Bind a request to the plan and build its segments on `stream`
 * (the runtime "passes a candidate-to-user mapping", aibriefing RO/NRO
 * paragraph; grouping the candidates of one user is what lets their K/V be
 * loaded once, aixai.ru "Deep Dive: Flash Attention"):
 *   d_map     int32 [n_cand], values in [0, n_users); BORROWED: must stay
 *             valid and unchanged until the last call of this request (the
 *             forward and backward calls read it)
 *   n_cand    1..max_cand;  n_users 1..max_users
 *   H, Lq     attention heads (1..max_heads) and queries per candidate
 *             (multiple of 8, at most 128); they shape the work list.
 * Produces, stream-ordered and bit-exact:
 *   counts[u]  = #{i : map[i] = u}
 *   offsets[u] = sum_{v<u} counts[v]   (offsets[n_users] = n_cand)
 *   perm       = candidates grouped by user, ascending i within a user
 *   work       = for u, for h, for each run of <= cands_per_unit entries of
 *                u's segment: {u, h, first position in perm, run length}
 * A map value out of range is skipped and reported by ikbo_plan_get_status. */
ikbo_status_t ikbo_plan(ikbo_plan_t p, const int32_t* d_map, int n_cand, int n_users, int H, int Lq,
                        cudaStream_t stream);

/* Borrow the segment arrays of the last ikbo_plan (device pointers, valid
 * until the next ikbo_plan or ikbo_plan_destroy): counts [n_users], offsets
 * [n_users+1], perm [n_cand] (positions offsets[n_users] .. n_cand-1 hold
 * the candidates whose map value is out of range, ascending).  Any output
 * pointer may be NULL. */
ikbo_status_t ikbo_plan_segments(ikbo_plan_t p, const int32_t** d_counts, const int32_t** d_offsets,
                                 const int32_t** d_perm);

/* Borrow the attention work list: d_work int32 [max_units][4], d_n_units a
 * device int32 holding the number of units, *cands_per_unit and *max_units
 * host values.  Any output pointer may be NULL. */
ikbo_status_t ikbo_plan_worklist(ikbo_plan_t p, const int32_t** d_work, const int32_t** d_n_units,
                                 int* cands_per_unit, int* max_units);

/* Linear Compression Embedding with in-kernel broadcast (aixai.ru, "Deep
 * Dive: Linear Compression", stages 1-4; aibriefing, LCE deep dive):
 *   Y[i][n][d] = b[n] + sum_{k<K_u} Wu[k][n] U[map[i]][k][d]
 *                     + sum_{k<K_c} Wc[k][n] C[i][k][d]
 * with the map, n_cand and n_users of the last ikbo_plan.
 *   U  bf16 [n_users][K_u][D]     C  bf16 [n_cand][K_c][D]
 *   Wu bf16 [K_u][N]              Wc bf16 [K_c][N]
 *   b  bf16 [N] or NULL           Y  bf16 [n_cand][N][D] (written)
 * bf16 inputs, fp32 accumulation, round-to-nearest-even bf16 output.  The
 * user GEMM runs at n_users into a plan-owned fp32 workspace (grown on the
 * first call that needs more; that call allocates synchronously) and is
 * added in the candidate GEMM's epilogue by map lookup.  One launch.
 * Limits: K_u, K_c >= 1; D, N multiples of 8; N <= 256;
 * ceil(K_c/64) * ceil(roundup(N,16)/64) <= 16 (Wc stays in shared memory);
 * else IKBO_ERR_UNSUPPORTED. */
ikbo_status_t ikbo_lce_forward(ikbo_plan_t p, const void* U, const void* C, const void* Wu, const void* Wc,
                               const void* b, void* Y, int K_u, int K_c, int D, int N, cudaStream_t stream);

/* The same fused LCE as ikbo_lce_forward, for callers that cannot allocate
 * device memory.  (The IKBO write-ups have no counterpart to this entry
 * point: it exists for deployment, not for the method.)
 *
 * ikbo_lce_forward keeps its scratch (fp32 user partials, readiness flags)
 * in a plan that ikbo_plan_create allocates with cudaMalloc.  Callers whose
 * device memory is owned by another allocator (a framework's memory pool, a
 * fixed per-process budget), or whose request path may not call cudaMalloc
 * or cudaFree (both can synchronise the device), use this instead: it takes
 * the request directly and keeps its scratch in a 16 MiB array that the
 * library declares in device memory, so it allocates nothing.
 *   d_map   int32 [n_cand], values in [0, n_users)
 *   U, C, Wu, Wc, b, Y, K_u, K_c, D, N: exactly as ikbo_lce_forward
 * Limits: those of ikbo_lce_forward, and
 *   4 * n_users * N * D
 *   + 4 * n_users * ceil(D/128) * ceil(roundup(N,16)/64) (rounded up to 256)
 *   + 256  <=  16 MiB, else IKBO_ERR_UNSUPPORTED before any launch.
 * Notes:
 *   - every GPU that loads the library holds the 16 MiB until process exit;
 *   - the first call made with a given device current looks up the array's
 *     device address (cudaGetSymbolAddress) and the device's limits (host
 *     queries that later calls on that device do not repeat);
 *   - all calls share the array and it keeps the last call's contents; each
 *     call first clears, on its stream, the words that must start at zero
 *     (status and readiness flags); calls that overlap on the GPU (two
 *     streams, or two host threads on one device) race;
 *   - device-detected errors are not reported: a candidate whose map value
 *     is out of range keeps its rows of Y untouched, and a bounded wait that
 *     runs out (which makes the waiting tiles form the user partial on the
 *     CUDA cores, so Y stays right) goes unnoticed. */
ikbo_status_t ikbo_lce_forward_noalloc(const int32_t* d_map, int n_cand, int n_users, const void* U, const void* C,
                                       const void* Wu, const void* Wc, const void* b, void* Y, int K_u, int K_c,
                                       int D, int N, cudaStream_t stream);

/* The pages' LCE stage ladder as ablations of this kernel (aixai.ru IKBO
 * blog, "Deep Dive: Linear Compression": decompose, pad K, fuse the
 * broadcast add into the epilogue, warp-specialised persistent fusion; the
 * aibriefing LCE deep dive's per-stage latencies).  Same arguments, result
 * and errors as ikbo_lce_forward; `stage`:
 *   1  decomposed and unfused: user tiles -> fp32 partial; candidate tiles
 *      store bf16(C[i] W_c) without it; a separate broadcast-add launch adds
 *      P[map[i]] (Y rounded twice; within the LCE tolerance)
 *   3  broadcast add fused into the candidate epilogue, one TMEM
 *      accumulator (a tile's epilogue and the next tile's products do not
 *      overlap)
 *   4  the full kernel (= ikbo_lce_forward)
 * The pages' stage 2 (pad K) has no separate variant here: TMA's
 * out-of-bounds zero fill pads K in every stage.  Other values:
 * IKBO_ERR_INVALID_ARG. */
ikbo_status_t ikbo_lce_forward_staged(ikbo_plan_t p, const void* U, const void* C, const void* Wu, const void* Wc,
                                      const void* b, void* Y, int K_u, int K_c, int D, int N, int stage,
                                      cudaStream_t stream);

/* LCE backward for training (aibriefing, "Meta Optimizes Inference for
 * Recommendation Systems": the IKBO kernels serve training when the
 * candidate:user ratio exceeds 1; the pages give no backward formulas, so
 * these are the chain rule of ikbo_lce_forward's definition).  Given the
 * upstream gradient dY = dL/dY and the map of the last ikbo_plan:
 *   S[u]       = sum_{i : map[i] = u} dY[i]          (fp32 segment sum; the
 *                transpose of the broadcast, so the user side stays at n_users)
 *   dU[u][k][d] = sum_n Wu[k][n] S[u][n][d]            bf16 [n_users][K_u][D]
 *   dWu[k][n]   = sum_u sum_d U[u][k][d] S[u][n][d]    fp32 [K_u][N]
 *   dC[i][k][d] = sum_n Wc[k][n] dY[i][n][d]           bf16 [n_cand][K_c][D]
 *   dWc[k][n]   = sum_i sum_d C[i][k][d] dY[i][n][d]   fp32 [K_c][N]
 *   db[n]       = sum_u sum_d S[u][n][d]               fp32 [N]
 *   U, C, Wu, Wc: as ikbo_lce_forward; dY bf16 [n_cand][N][D].
 * Every output pointer may be NULL to skip that gradient; an input is only
 * required by the gradients that read it (Wu for dU, Wc for dC, U for dWu,
 * C for dWc), else IKBO_ERR_INVALID_ARG.  Outputs are overwritten, not
 * accumulated into.  bf16 operands, fp32 accumulation; S is rounded to bf16
 * for the two products that read it (dU, dWu).  The weight gradients are
 * summed over split-K partials in a fixed order, so results repeat bit for
 * bit.  Candidates whose map value is out of range are left out of S (so of
 * dU, dWu and db) and reported by the plan's status; they still enter dC and
 * dWc.  Workspaces (S, partial sums) are plan-owned and grown on first use
 * (that call allocates synchronously).  With both dU and dWu asked for, dWu
 * runs on a second stream the plan creates on first use, forked from and
 * joined back into `stream` through events: the call stays ordered on
 * `stream` like a single-stream one.  With K_c <= 256 and N <= 192 the
 * candidate side (dC, dWc, S, db) is one cooperative launch whose CTAs wait
 * for one another once (bounded by the plan's timeout); where a cooperative
 * launch is refused it is two launches.  Limits: D, N multiples of 8,
 * N <= 256; for dC / dU, K <= 512 and the weight, roundup(K, 128) *
 * ceil(N / 64) * 128 bytes, fits in shared memory beside two 16 KB stages
 * (about 190 KB); else IKBO_ERR_UNSUPPORTED. */
ikbo_status_t ikbo_lce_backward(ikbo_plan_t p, const void* U, const void* C, const void* Wu, const void* Wc,
                                const void* dY, void* dU, void* dC, float* dWu, float* dWc, float* db, int K_u,
                                int K_c, int D, int N, cudaStream_t stream);

/* Broadcast attention (aixai.ru, "Deep Dive: Flash Attention"; aibriefing,
 * Flash Attention case): for every candidate i and head h, with u = map[i],
 *   O[i,h,q,:] = sum_j softmax_j(scale * Q[i,h,q,:].K[u,h,j,:]) V[u,h,j,:]
 * with the map, n_cand, n_users, H and Lq of the last ikbo_plan.
 *   Q bf16 [n_cand][H][Lq][d]
 *   dense  (d_kv_offsets == NULL): K, V bf16 [n_users][H][Lkv][d], Lkv >= 1
 *   jagged (d_kv_offsets != NULL): K, V bf16 [Lkv][H][d] where Lkv is the
 *          total packed rows and user u owns rows d_kv_offsets[u] ..
 *          d_kv_offsets[u+1]-1 (int32 [n_users+1], offsets[0] = 0)
 *   O bf16 [n_cand][H][Lq][d] (written; rows whose user has no keys get 0)
 *   scale  > 0 (usually 1/sqrt(d)).  No mask.
 * Each user's K/V tile is read once per work unit and shared by up to
 * floor(128/Lq) candidates.  fp32 scores and softmax, P rounded to bf16
 * for P.V, fp32 accumulation, bf16 output.  Limits: d == 128. */
ikbo_status_t ikbo_attn_forward(ikbo_plan_t p, const void* Q, const void* K, const void* V,
                                const int32_t* d_kv_offsets, void* O, int Lkv, int d, float scale,
                                cudaStream_t stream);

/* Self + target attention in one launch (aixai.ru IKBO blog, section
 * "Self + Target Attention Fusion"): self-attention and target-attention
 * read the same per-user K/V and differ only in their queries -- the users'
 * own query set (self) and their candidates' queries (target) -- so both run
 * as work units of one launch of the broadcast attention kernel:
 *   O[i,h]      = softmax(Q[i,h] K[map[i],h]^T * scale) V[map[i],h]   (as ikbo_attn_forward)
 *   O_user[u,h] = softmax(Q_user[u,h] K[u,h]^T * scale) V[u,h]
 * The pages give no mask, causality or query length for the self part; it
 * is read here as the same unmasked attention over the user's whole key
 * range, with its own query length Lq_u.
 *   Q_user, O_user bf16 [n_users][H][Lq_u][d], 16-byte aligned; Lq_u >= 8,
 *   a multiple of 8 (else IKBO_ERR_UNSUPPORTED); users with no keys get
 *   O_user rows of 0.  Every other argument, limit and error as for
 *   ikbo_attn_forward (the plan's map, n_users, H and Lq; K/V dense or
 *   jagged).  The target rows of O are bit-identical to ikbo_attn_forward's.
 *   The self units (n_users * H * ceil(Lq_u / 128) tiles of up to 128 query
 *   rows) follow the plan's work list in the persistent launch.  Q and O both
 *   NULL: the self part alone (the plan's map is then not read by the launch,
 *   but n_users and H still come from the last ikbo_plan). */
ikbo_status_t ikbo_attn_self_target_forward(ikbo_plan_t p, const void* Q, const void* Q_user, const void* K,
                                            const void* V, const int32_t* d_kv_offsets, void* O, void* O_user,
                                            int Lq_u, int Lkv, int d, float scale, cudaStream_t stream);

/* ikbo_attn_forward for training: the same O (bit-identical), and also each
 * query row's softmax log-sum-exp, the statistic the backward needs to
 * recover every probability without a second pass over the keys:
 *   lse[i,h,q] = log( sum_j exp(scale Q[i,h,q] . K[map[i],h,j]) )   (natural log)
 * fp32 [n_cand][H][Lq], caller-owned, 4-byte aligned, overwritten; -inf for
 * the rows of a user with no keys.  Same inputs, limits and errors as
 * ikbo_attn_forward (lse NULL: IKBO_ERR_INVALID_ARG).  The definition is the
 * normaliser of the attention in aixai.ru, "Deep Dive: Flash Attention"
 * (ordinary attention with K/V from the candidate's user). */
ikbo_status_t ikbo_attn_forward_lse(ikbo_plan_t p, const void* Q, const void* K, const void* V,
                                    const int32_t* d_kv_offsets, void* O, float* lse, int Lkv, int d, float scale,
                                    cudaStream_t stream);

/* Broadcast attention backward for training (aibriefing, "Meta Optimizes
 * Inference for Recommendation Systems": the kernels serve training when
 * candidates outnumber users; the pages give no backward, so this is the
 * chain rule of ikbo_attn_forward's definition).  Given the forward's
 * inputs, its output O and the upstream gradient dO = dL/dO, with the plan's
 * map, H and Lq, for every candidate i, head h, query q (u = map[i]):
 *   p = softmax(scale Q K[u]^T), dP = dO V[u]^T, D = rowsum(dO * O),
 *   dS = p (dP - D)
 *   dQ[i,h]  = scale dS K[u,h]                          bf16, Q's layout
 *   dK[u,h]  = scale sum_{i : map[i] = u} dS_i^T Q[i,h]   bf16, K's layout
 *   dV[u,h]  = sum_{i : map[i] = u} p_i^T dO[i,h]         bf16, V's layout
 * so the K/V gradients sum over every candidate of a user, the transpose of
 * the forward's broadcast; keys of a user with no candidates get 0, queries
 * of a user with no keys get dQ = 0.
 *   Q, O, dO bf16 [n_cand][H][Lq][d]; K, V (and dK, dV) dense or jagged
 *   exactly as in ikbo_attn_forward; all 16-byte aligned, none NULL.
 *   lse: the forward's log-sum-exp (ikbo_attn_forward_lse on the same
 *   inputs), fp32 [n_cand][H][Lq], 4-byte aligned; or NULL, and the
 *   backward recomputes it with one more pass over each user's keys.
 * P and dS are rounded to bf16 for the tensor cores (as P is in the
 * forward); accumulation is fp32.  Gradients are overwritten.  Three
 * launches; the plan keeps per-row LSE and D (grown on first use, which
 * allocates synchronously).  Limits: d == 128 (else IKBO_ERR_UNSUPPORTED);
 * the plan's map values must be in range (a candidate outside is skipped by
 * the segments, so its dQ is left untouched). */
ikbo_status_t ikbo_attn_backward(ikbo_plan_t p, const void* Q, const void* K, const void* V, const void* O,
                                 const void* dO, const float* lse, const int32_t* d_kv_offsets, void* dQ, void* dK,
                                 void* dV, int Lkv, int d, float scale, cudaStream_t stream);

/* Synchronise `stream`, then return (and clear) the first device-detected
 * error recorded since the last call: IKBO_ERR_MAP_OUT_OF_RANGE,
 * IKBO_ERR_TIMEOUT, IKBO_ERR_INTERNAL, or IKBO_OK. */
ikbo_status_t ikbo_plan_get_status(ikbo_plan_t p, cudaStream_t stream);

/* Debug and robustness knobs.  flags: bit 0 = LCE user tiles compute but do
 * not publish their partials (candidate epilogues then wait, give up after
 * the timeout, form the partial themselves on the CUDA cores, still write a
 * correct Y, and the call reports IKBO_ERR_TIMEOUT); bit 1 = the LCE
 * backward's candidate pass does not end with its finish in the same
 * (cooperative) launch but is followed by a finish kernel, the path taken
 * where a cooperative launch is refused.  The timeout bounds every wait
 * inside the kernels (default 2 s). */
ikbo_status_t ikbo_plan_set_debug(ikbo_plan_t p, unsigned flags);
ikbo_status_t ikbo_plan_set_timeout_ns(ikbo_plan_t p, uint64_t timeout_ns);

/* Launch schedule of ikbo_lce_forward (plan-time kernel selection over the
 * shape range, the "compile for a range of shapes" idea of the pages done as
 * a runtime choice):
 *   0  chosen from the shape (default): 3 where it applies; otherwise 2 for
 *      a single user or when the request has fewer than 8 candidate tiles
 *      of 128 D-rows per SM, else 1
 *   1  two launches: user tiles (fp32 partials in the plan's workspace, with
 *      release flags), then candidate tiles
 *   2  one launch: user tiles first in every CTA's list.  Its candidate
 *      tiles wait for user tiles of other CTAs, so it is a cooperative
 *      launch (all CTAs resident at once); where the context cannot hold
 *      one CTA per SM of the device (fewer SMs available to it) it runs
 *      as 1
 *   3  local partials, one launch: each CTA computes, into TMEM, the partial
 *      of every (user, 128-row D block) its candidate tiles need and keeps it
 *      in registers; no workspace and no hand-off between CTAs.  Applies when
 *      N <= 192 and shared memory holds W_c plus two full-width W_u chunks;
 *      elsewhere a request for 3 runs as 0.
 * Results are identical; only the time differs.  Other values:
 * IKBO_ERR_INVALID_ARG. */
ikbo_status_t ikbo_plan_set_lce_schedule(ikbo_plan_t p, int schedule);

/* Number of kernel launches the forward calls and ikbo_plan have made
 * through this plan since it was created. */
uint64_t ikbo_plan_launch_count(ikbo_plan_t p);

const char* ikbo_status_string(ikbo_status_t s);

/* Synchronise the device and free the plan's memory.  NULL is a no-op. */
void ikbo_plan_destroy(ikbo_plan_t p);

/* ABI version (major * 100 + minor). */
int ikbo_version(void);

#ifdef __cplusplus
}
#endif

#endif /* IKBO_H */
