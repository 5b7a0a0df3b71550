/*
 * ikbo_oracle.c -- CPU oracle for the In-Kernel Broadcast Optimization (IKBO)
 * hot path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; no product code path may.
 *
 * It computes, plainly and slowly, in double precision, what the IKBO kernels
 * compute quickly: the MATERIALISED-broadcast definition.  IKBO's claim is that
 * it reaches the same result without ever building the replicated user tensor;
 * this file builds it, on purpose, so that nothing here resembles the GPU path.
 *
 * Sources (the IKBO write-ups):
 *   - "IKBO: recsys kernel optimization" (aixai.ru blog), section "Что такое
 *     broadcast-проблема": user features are the same for all candidates of a
 *     request and are replicated ~70x to match the candidate batch.
 *   - same page, "Deep Dive: Linear Compression": LCE is one batched matmul of
 *     the (replicated) input embeddings with a learned projection W; stage 1
 *     splits it by linearity into a user part and a candidate part.
 *   - "Meta Optimizes Inference for Recommendation Systems" (aibriefing), LCE
 *     deep dive: the split is along the K axis.
 *   - aixai.ru, "Deep Dive: Flash Attention": IKBO attention is ordinary
 *     attention whose K/V come from the candidate's user; nothing changes in
 *     the result, only in how K/V are fetched.
 *
 * Readings taken where the pages are silent (each repeated at its function):
 *   - LCE orientation: X[i] is [K, D] (K embeddings of width D), W is [K, N],
 *     Y[i] = W^T X[i] is [N, D]; user rows come first along K.
 *   - LCE bias b[N] is added once per output element, broadcast over D.
 *   - Attention: scale 1/sqrt(d) unless the caller passes another, no mask,
 *     heads independent; an empty key range gives output 0.
 *   - Segments: stable counting sort (ascending candidate index within a
 *     user); work units ordered by user, then head, then chunk.
 *
 * All inputs arrive as bf16 bit patterns (uint16) and are widened to double
 * exactly; every sum is formed in double in ascending index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_MAP_OUT_OF_RANGE 2
#define ORACLE_NO_MEMORY 3
#define ORACLE_WORK_OVERFLOW 4

/* Exact widening of a bf16 bit pattern: its bits are the top half of a float. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static void set_threads(int n_threads)
{
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
}

int ikbo_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Segments: counts[u] = #{i : map[i] = u}; offsets = exclusive prefix sum of
 * counts (offsets[n_users] = n_cand); perm lists the candidates grouped by
 * user, keeping ascending candidate order inside a user.  The attention work
 * list follows: for each user u, each head h, each run of at most
 * `cands_per_unit` consecutive entries of u's segment, one unit
 * (u, h, first position in perm, count).
 *
 * Grouping a user's candidates is what lets their K/V be fetched once ("K/V
 * accesses amortised across candidates sharing one user", aixai.ru, "Deep
 * Dive: Flash Attention").
 */
int ikbo_oracle_segments(const int32_t *map, int n_cand, int n_users, int H, int cands_per_unit,
                         int32_t *counts, int32_t *offsets, int32_t *perm,
                         int32_t *work, int64_t max_units, int64_t *n_units)
{
    if (n_cand < 0 || n_users < 1 || H < 1 || cands_per_unit < 1) return ORACLE_BAD_ARG;
    for (int i = 0; i < n_cand; ++i)
        if (map[i] < 0 || map[i] >= n_users) return ORACLE_MAP_OUT_OF_RANGE;

    for (int u = 0; u < n_users; ++u) counts[u] = 0;
    for (int i = 0; i < n_cand; ++i) counts[map[i]] += 1;

    offsets[0] = 0;
    for (int u = 0; u < n_users; ++u) offsets[u + 1] = offsets[u] + counts[u];

    int32_t *next = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_users);
    if (!next) return ORACLE_NO_MEMORY;
    for (int u = 0; u < n_users; ++u) next[u] = offsets[u];
    for (int i = 0; i < n_cand; ++i) {       /* ascending i: stable */
        int u = map[i];
        perm[next[u]] = i;
        next[u] += 1;
    }
    free(next);

    int64_t k = 0;
    for (int u = 0; u < n_users; ++u) {
        for (int h = 0; h < H; ++h) {
            for (int c = 0; c < counts[u]; c += cands_per_unit) {
                if (k >= max_units) return ORACLE_WORK_OVERFLOW;
                int cnt = counts[u] - c;
                if (cnt > cands_per_unit) cnt = cands_per_unit;
                work[4 * k + 0] = u;
                work[4 * k + 1] = h;
                work[4 * k + 2] = offsets[u] + c;
                work[4 * k + 3] = cnt;
                k += 1;
            }
        }
    }
    *n_units = k;
    return ORACLE_OK;
}

/*
 * Linear Compression Embedding, materialised form.
 *
 * For candidate i with user u = map[i]:
 *   X[i] = [ U[u] ; C[i] ]              ((K_u + K_c) x D, the replicated input)
 *   W    = [ W_u  ; W_c  ]              ((K_u + K_c) x N)
 *   Y[i][n][d] = b[n] + sum_k W[k][n] * X[i][k][d]
 *
 * This is the baseline "one batched matmul over all candidates" of aixai.ru,
 * "Deep Dive: Linear Compression"; the IKBO kernels reach the same Y through
 * the K-axis split (stage 1), which is exact in exact arithmetic.
 *
 * Layouts (row-major): map[n_cand]; U[n_users][K_u][D]; C[n_cand][K_c][D];
 * Wu[K_u][N]; Wc[K_c][N]; b[N] or NULL; output Y[n_sel][N][D] in double for
 * the selected candidates cands[0..n_sel) (all candidates, in order, when
 * cands is NULL and n_sel == n_cand).
 */
int ikbo_oracle_lce(const int32_t *map, const uint16_t *U, const uint16_t *C,
                    const uint16_t *Wu, const uint16_t *Wc, const uint16_t *b,
                    int n_cand, int n_users, int K_u, int K_c, int D, int N,
                    const int32_t *cands, int n_sel, double *Y, int n_threads)
{
    if (n_cand < 0 || n_users < 1 || K_u < 0 || K_c < 0 || D < 1 || N < 1 || n_sel < 0)
        return ORACLE_BAD_ARG;
    if (!cands && n_sel != n_cand) return ORACLE_BAD_ARG;
    const int K = K_u + K_c;

    for (int s = 0; s < n_sel; ++s) {
        int i = cands ? cands[s] : s;
        if (i < 0 || i >= n_cand) return ORACLE_BAD_ARG;
        if (map[i] < 0 || map[i] >= n_users) return ORACLE_MAP_OUT_OF_RANGE;
    }

    /* W = concat_rows(W_u, W_c) */
    double *W = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)N);
    if (!W) return ORACLE_NO_MEMORY;
    for (int k = 0; k < K_u; ++k)
        for (int n = 0; n < N; ++n) W[(size_t)k * N + n] = bf16_bits_to_double(Wu[(size_t)k * N + n]);
    for (int k = 0; k < K_c; ++k)
        for (int n = 0; n < N; ++n)
            W[(size_t)(K_u + k) * N + n] = bf16_bits_to_double(Wc[(size_t)k * N + n]);

    int status = ORACLE_OK;
    set_threads(n_threads);
#pragma omp parallel
    {
        double *X = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)D);
        if (!X) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        }
#pragma omp for schedule(dynamic, 1)
        for (int s = 0; s < n_sel; ++s) {
            if (!X) continue;
            int i = cands ? cands[s] : s;
            int u = map[i];
            /* the broadcast: copy user u's rows, then candidate i's rows */
            for (int k = 0; k < K_u; ++k)
                for (int d = 0; d < D; ++d)
                    X[(size_t)k * D + d] = bf16_bits_to_double(U[((size_t)u * K_u + k) * D + d]);
            for (int k = 0; k < K_c; ++k)
                for (int d = 0; d < D; ++d)
                    X[(size_t)(K_u + k) * D + d] = bf16_bits_to_double(C[((size_t)i * K_c + k) * D + d]);
            double *Yi = Y + (size_t)s * N * D;
            for (int n = 0; n < N; ++n) {
                double bias = b ? bf16_bits_to_double(b[n]) : 0.0;
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int k = 0; k < K; ++k) acc += W[(size_t)k * N + n] * X[(size_t)k * D + d];
                    Yi[(size_t)n * D + d] = bias + acc;
                }
            }
        }
        free(X);
    }
    free(W);
    return status;
}

/*
 * Broadcast attention, ordinary softmax attention per (candidate, head):
 *   u = map[i];  keys/values are user u's rows j in [0, L_u)
 *   s_j  = scale * sum_c Q[i,h,q,c] * K[u,h,j,c]
 *   m    = max_j s_j;   p_j = exp(s_j - m)
 *   O[i,h,q,:] = sum_j p_j V[u,h,j,:] / sum_j p_j        (0 when L_u = 0)
 *
 * aixai.ru, "Deep Dive: Flash Attention": IKBO FA reuses one user's K/V for
 * all of that user's candidates; the attention itself is unchanged.
 *
 * Layouts: Q[n_cand][H][Lq][d].  Dense K/V (kv_offsets NULL):
 * K[n_users][H][Lkv][d].  Jagged K/V: K[total][H][d], user u owning rows
 * kv_offsets[u] .. kv_offsets[u+1]-1.  Output O[n_sel][Lq][d] in double for
 * the selected (i, h) pairs pairs[2s], pairs[2s+1] (all pairs in (i, h) order
 * when pairs is NULL and n_sel == n_cand*H).
 */
int ikbo_oracle_attn(const int32_t *map, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     const int32_t *kv_offsets, int n_cand, int n_users, int H, int Lq, int Lkv,
                     int d, double scale, const int32_t *pairs, int n_sel, double *O, int n_threads)
{
    if (n_cand < 0 || n_users < 1 || H < 1 || Lq < 1 || d < 1 || n_sel < 0) return ORACLE_BAD_ARG;
    if (!kv_offsets && Lkv < 0) return ORACLE_BAD_ARG;
    if (!pairs && n_sel != n_cand * H) return ORACLE_BAD_ARG;
    for (int s = 0; s < n_sel; ++s) {
        int i = pairs ? pairs[2 * s] : s / H;
        int h = pairs ? pairs[2 * s + 1] : s % H;
        if (i < 0 || i >= n_cand || h < 0 || h >= H) return ORACLE_BAD_ARG;
        if (map[i] < 0 || map[i] >= n_users) return ORACLE_MAP_OUT_OF_RANGE;
    }
    int max_len = Lkv;
    if (kv_offsets) {
        max_len = 0;
        for (int u = 0; u < n_users; ++u) {
            int L = kv_offsets[u + 1] - kv_offsets[u];
            if (L < 0) return ORACLE_BAD_ARG;
            if (L > max_len) max_len = L;
        }
    }

    int status = ORACLE_OK;
    set_threads(n_threads);
#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        if (!sc) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        }
#pragma omp for schedule(dynamic, 1)
        for (int s = 0; s < n_sel; ++s) {
            if (!sc) continue;
            int i = pairs ? pairs[2 * s] : s / H;
            int h = pairs ? pairs[2 * s + 1] : s % H;
            int u = map[i];
            int L;
            size_t row0, row_stride; /* element offset of key row 0 and between key rows */
            if (kv_offsets) {
                L = kv_offsets[u + 1] - kv_offsets[u];
                row0 = ((size_t)kv_offsets[u] * H + h) * d;
                row_stride = (size_t)H * d;
            } else {
                L = Lkv;
                row0 = ((size_t)u * H + h) * (size_t)Lkv * d;
                row_stride = (size_t)d;
            }
            for (int q = 0; q < Lq; ++q) {
                const uint16_t *qrow = Q + (((size_t)i * H + h) * Lq + q) * d;
                double *orow = O + ((size_t)s * Lq + q) * d;
                for (int c = 0; c < d; ++c) orow[c] = 0.0;
                if (L == 0) continue;
                double m = -INFINITY;
                for (int j = 0; j < L; ++j) {
                    const uint16_t *krow = K + row0 + (size_t)j * row_stride;
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += bf16_bits_to_double(qrow[c]) * bf16_bits_to_double(krow[c]);
                    sc[j] = scale * dot;
                    if (sc[j] > m) m = sc[j];
                }
                double l = 0.0;
                for (int j = 0; j < L; ++j) {
                    sc[j] = exp(sc[j] - m);
                    l += sc[j];
                }
                for (int j = 0; j < L; ++j) {
                    const uint16_t *vrow = V + row0 + (size_t)j * row_stride;
                    double w = sc[j];
                    for (int c = 0; c < d; ++c) orow[c] += w * bf16_bits_to_double(vrow[c]);
                }
                for (int c = 0; c < d; ++c) orow[c] /= l;
            }
        }
        free(sc);
    }
    return status;
}

/*
 * Log-sum-exp of each query row's scores, the normaliser of the softmax in
 * ikbo_oracle_attn (aixai.ru, "Deep Dive: Flash Attention": IKBO attention is
 * ordinary attention whose K/V come from the candidate's user):
 *   LSE[i,h,q] = log( sum_{j in keys of map[i]} exp(scale * Q[i,h,q] . K[map[i],h,j]) )
 * in natural log, formed as m + log(sum exp(s_j - m)) with m the row maximum.
 * An empty key range gives -inf (the sum is empty).  Output double
 * [n_sel][Lq] for the (i, h) pairs (all, in (i, h) order, when pairs is NULL
 * and n_sel == n_cand * H).  This is the statistic a training forward keeps
 * so that its backward can recover every softmax probability as
 * exp(s_j - LSE) without a second pass over the keys.
 */
int ikbo_oracle_attn_lse(const int32_t *map, const uint16_t *Q, const uint16_t *K, const int32_t *kv_offsets,
                         int n_cand, int n_users, int H, int Lq, int Lkv, int d, double scale,
                         const int32_t *pairs, int n_sel, double *lse, int n_threads)
{
    if (n_cand < 0 || n_users < 1 || H < 1 || Lq < 1 || d < 1 || n_sel < 0) return ORACLE_BAD_ARG;
    if (!kv_offsets && Lkv < 0) return ORACLE_BAD_ARG;
    if (!pairs && n_sel != n_cand * H) return ORACLE_BAD_ARG;
    for (int s = 0; s < n_sel; ++s) {
        int i = pairs ? pairs[2 * s] : s / H;
        int h = pairs ? pairs[2 * s + 1] : s % H;
        if (i < 0 || i >= n_cand || h < 0 || h >= H) return ORACLE_BAD_ARG;
        if (map[i] < 0 || map[i] >= n_users) return ORACLE_MAP_OUT_OF_RANGE;
    }
    if (kv_offsets)
        for (int u = 0; u < n_users; ++u)
            if (kv_offsets[u + 1] < kv_offsets[u]) return ORACLE_BAD_ARG;
    set_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
    for (int s = 0; s < n_sel; ++s) {
        int i = pairs ? pairs[2 * s] : s / H;
        int h = pairs ? pairs[2 * s + 1] : s % H;
        int u = map[i];
        int L = kv_offsets ? kv_offsets[u + 1] - kv_offsets[u] : Lkv;
        for (int q = 0; q < Lq; ++q) {
            const uint16_t *qrow = Q + (((size_t)i * H + h) * Lq + q) * d;
            double m = -INFINITY, sum = 0.0;
            /* two sweeps over the keys: the maximum, then the shifted sum */
            for (int pass = 0; pass < 2; ++pass) {
                for (int j = 0; j < L; ++j) {
                    const uint16_t *krow = kv_offsets ? K + ((size_t)(kv_offsets[u] + j) * H + h) * d
                                                      : K + (((size_t)u * H + h) * (size_t)Lkv + j) * d;
                    double dot = 0.0;
                    for (int c = 0; c < d; ++c) dot += bf16_bits_to_double(qrow[c]) * bf16_bits_to_double(krow[c]);
                    double sj = scale * dot;
                    if (pass == 0) {
                        if (sj > m) m = sj;
                    } else {
                        sum += exp(sj - m);
                    }
                }
            }
            lse[(size_t)s * Lq + q] = L > 0 ? m + log(sum) : -INFINITY;
        }
    }
    return ORACLE_OK;
}

/*
 * LCE backward (training), from the materialised definition.  The pages say
 * the IKBO kernels serve training as they are when the candidate:user ratio
 * exceeds 1 ("Meta Optimizes Inference for Recommendation Systems",
 * aibriefing, the paragraph on kernels, compilation and runtime); they give
 * no backward formulas, so this is the chain rule of the forward above:
 *
 *   X[i] = [U[map[i]]; C[i]]  (the replicated input, K = K_u + K_c rows)
 *   Y[i] = W^T X[i] + b,  W = [W_u; W_c]
 *   given dY[i] = dL/dY[i]:
 *     dX[i][k][d] = sum_n W[k][n] dY[i][n][d]
 *     dW[k][n]    = sum_i sum_d X[i][k][d] dY[i][n][d]
 *     db[n]       = sum_i sum_d dY[i][n][d]
 *   and the broadcast's own rule: every copy of U[u] passes its gradient back,
 *     dU[u] = sum_{i : map[i] = u} dX[i][0 .. K_u)
 *     dC[i] = dX[i][K_u .. K)
 *   dW_u = dW[0 .. K_u), dW_c = dW[K_u .. K).
 *
 * Selections keep the cost bounded: dC for candidates csel[0..n_csel) (all,
 * in order, when csel is NULL and n_csel == n_cand), dU for users
 * usel[0..n_usel) (all when usel is NULL and n_usel == n_users), and dW_u,
 * dW_c, db only when want_w != 0.  Outputs in double: dC[n_csel][K_c][D],
 * dU[n_usel][K_u][D], dWu[K_u][N], dWc[K_c][N], db[N].  Every sum runs over
 * candidates in ascending order, then n (or d) ascending.
 */
int ikbo_oracle_lce_backward(const int32_t *map, const uint16_t *U, const uint16_t *C,
                             const uint16_t *Wu, const uint16_t *Wc, const uint16_t *dY,
                             int n_cand, int n_users, int K_u, int K_c, int D, int N,
                             const int32_t *csel, int n_csel, const int32_t *usel, int n_usel,
                             int want_w, double *dC, double *dU, double *dWu, double *dWc,
                             double *db, int n_threads)
{
    if (n_cand < 0 || n_users < 1 || K_u < 0 || K_c < 0 || D < 1 || N < 1 || n_csel < 0 || n_usel < 0)
        return ORACLE_BAD_ARG;
    if (!csel && n_csel != n_cand) return ORACLE_BAD_ARG;
    if (!usel && n_usel != n_users) return ORACLE_BAD_ARG;
    for (int i = 0; i < n_cand; ++i)
        if (map[i] < 0 || map[i] >= n_users) return ORACLE_MAP_OUT_OF_RANGE;
    for (int s = 0; s < n_csel; ++s)
        if ((csel ? csel[s] : s) < 0 || (csel ? csel[s] : s) >= n_cand) return ORACLE_BAD_ARG;
    for (int s = 0; s < n_usel; ++s)
        if ((usel ? usel[s] : s) < 0 || (usel ? usel[s] : s) >= n_users) return ORACLE_BAD_ARG;
    const int K = K_u + K_c;
    set_threads(n_threads);

    /* dX[i][K_u + k] for the selected candidates: their dC */
#pragma omp parallel for schedule(dynamic, 1)
    for (int s = 0; s < n_csel; ++s) {
        const int i = csel ? csel[s] : s;
        for (int k = 0; k < K_c; ++k)
            for (int d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int n = 0; n < N; ++n)
                    acc += bf16_bits_to_double(Wc[(size_t)k * N + n]) *
                           bf16_bits_to_double(dY[((size_t)i * N + n) * D + d]);
                dC[((size_t)s * K_c + k) * D + d] = acc;
            }
    }

    /* dU[u]: the user rows of dX[i], summed over every copy of U[u] */
#pragma omp parallel for schedule(dynamic, 1)
    for (int s = 0; s < n_usel; ++s) {
        const int u = usel ? usel[s] : s;
        double *out = dU + (size_t)s * K_u * D;
        for (size_t e = 0; e < (size_t)K_u * D; ++e) out[e] = 0.0;
        for (int i = 0; i < n_cand; ++i) {
            if (map[i] != u) continue;
            for (int k = 0; k < K_u; ++k)
                for (int d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int n = 0; n < N; ++n)
                        acc += bf16_bits_to_double(Wu[(size_t)k * N + n]) *
                               bf16_bits_to_double(dY[((size_t)i * N + n) * D + d]);
                    out[(size_t)k * D + d] += acc;
                }
        }
    }

    if (!want_w) return ORACLE_OK;

    /* dW[k][n] = sum_i sum_d X[i][k][d] dY[i][n][d], X[i] the replicated input */
#pragma omp parallel for schedule(dynamic, 1)
    for (int k = 0; k < K; ++k) {
        for (int n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int i = 0; i < n_cand; ++i) {
                const uint16_t *xrow = k < K_u ? U + ((size_t)map[i] * K_u + k) * D
                                               : C + ((size_t)i * K_c + (k - K_u)) * D;
                const uint16_t *grow = dY + ((size_t)i * N + n) * D;
                for (int d = 0; d < D; ++d) acc += bf16_bits_to_double(xrow[d]) * bf16_bits_to_double(grow[d]);
            }
            if (k < K_u)
                dWu[(size_t)k * N + n] = acc;
            else
                dWc[(size_t)(k - K_u) * N + n] = acc;
        }
    }
    for (int n = 0; n < N; ++n) {
        double acc = 0.0;
        for (int i = 0; i < n_cand; ++i)
            for (int d = 0; d < D; ++d) acc += bf16_bits_to_double(dY[((size_t)i * N + n) * D + d]);
        db[n] = acc;
    }
    return ORACLE_OK;
}

/* One query row: p_j = softmax_j(scale * q.k_j) and dS_j = p_j (dP_j - D)
 * with dP_j = g.v_j and D = sum_j p_j dP_j (= g.o), for the L keys starting
 * at element row0, row_stride elements apart (scale is applied by callers). */
static void attn_row(const uint16_t *qr, const uint16_t *gr, const uint16_t *K, const uint16_t *V, size_t row0,
                     size_t row_stride, int L, int d, double scale, double *p, double *ds)
{
    double m = -INFINITY;
    for (int j = 0; j < L; ++j) {
        const uint16_t *kr = K + row0 + (size_t)j * row_stride;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += bf16_bits_to_double(qr[c]) * bf16_bits_to_double(kr[c]);
        p[j] = scale * dot;
        if (p[j] > m) m = p[j];
    }
    double l = 0.0;
    for (int j = 0; j < L; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int j = 0; j < L; ++j) p[j] /= l;
    double D = 0.0;
    for (int j = 0; j < L; ++j) {
        const uint16_t *vr = V + row0 + (size_t)j * row_stride;
        double dp = 0.0;
        for (int c = 0; c < d; ++c) dp += bf16_bits_to_double(gr[c]) * bf16_bits_to_double(vr[c]);
        ds[j] = dp;
        D += p[j] * dp;
    }
    for (int j = 0; j < L; ++j) ds[j] = p[j] * (ds[j] - D);
}

/*
 * Broadcast attention backward (training), from the definition above (the
 * pages give no backward; the aibriefing paragraph on kernels, compilation
 * and runtime says the kernels serve training when candidates outnumber
 * users).  For every candidate i, head h, query q, with u = map[i] and keys
 * j of user u:
 *   s_j = scale * Q[i,h,q,:].K[u,h,j,:],  p = softmax(s),  o = sum_j p_j V[u,h,j,:]
 *   dP_j = dO[i,h,q,:].V[u,h,j,:],  D = dO[i,h,q,:].o,  dS_j = p_j (dP_j - D)
 *   dQ[i,h,q,:]  = scale * sum_j dS_j K[u,h,j,:]
 *   dK[u,h,j,:] += scale * dS_j Q[i,h,q,:]      (every candidate of u adds in:
 *   dV[u,h,j,:] += p_j dO[i,h,q,:]               the broadcast's transpose)
 * Selections: dQ for (i, h) pairs qpairs[2s], qpairs[2s+1] (all in (i, h)
 * order when qpairs is NULL and n_qsel == n_cand*H); dK, dV for (u, h) pairs
 * kvpairs (all in (u, h) order when NULL and n_kvsel == n_users*H).  Outputs
 * in double: dQ[n_qsel][Lq][d]; dK, dV[n_kvsel][max_len][d], rows past the
 * user's key count left 0 (max_len = Lkv dense, the longest user jagged).
 * Candidates and queries are summed in ascending order.
 */
int ikbo_oracle_attn_backward(const int32_t *map, const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                              const uint16_t *dO, const int32_t *kv_offsets, int n_cand, int n_users, int H,
                              int Lq, int Lkv, int d, double scale, const int32_t *qpairs, int n_qsel,
                              const int32_t *kvpairs, int n_kvsel, double *dQ, double *dK, double *dV,
                              int n_threads)
{
    if (n_cand < 0 || n_users < 1 || H < 1 || Lq < 1 || d < 1 || n_qsel < 0 || n_kvsel < 0) return ORACLE_BAD_ARG;
    if (!kv_offsets && Lkv < 0) return ORACLE_BAD_ARG;
    if (!qpairs && n_qsel != n_cand * H) return ORACLE_BAD_ARG;
    if (!kvpairs && n_kvsel != n_users * H) return ORACLE_BAD_ARG;
    for (int i = 0; i < n_cand; ++i)
        if (map[i] < 0 || map[i] >= n_users) return ORACLE_MAP_OUT_OF_RANGE;
    int max_len = Lkv;
    if (kv_offsets) {
        max_len = 0;
        for (int u = 0; u < n_users; ++u) {
            int L = kv_offsets[u + 1] - kv_offsets[u];
            if (L < 0) return ORACLE_BAD_ARG;
            if (L > max_len) max_len = L;
        }
    }
    for (int s = 0; s < n_qsel; ++s) {
        int i = qpairs ? qpairs[2 * s] : s / H, h = qpairs ? qpairs[2 * s + 1] : s % H;
        if (i < 0 || i >= n_cand || h < 0 || h >= H) return ORACLE_BAD_ARG;
    }
    for (int s = 0; s < n_kvsel; ++s) {
        int u = kvpairs ? kvpairs[2 * s] : s / H, h = kvpairs ? kvpairs[2 * s + 1] : s % H;
        if (u < 0 || u >= n_users || h < 0 || h >= H) return ORACLE_BAD_ARG;
    }
    set_threads(n_threads);
    int status = ORACLE_OK;

#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        double *ds = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        if (!p || !ds) {
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
        }
        /* dQ */
#pragma omp for schedule(dynamic, 1)
        for (int s = 0; s < n_qsel; ++s) {
            if (!p || !ds) continue;
            const int i = qpairs ? qpairs[2 * s] : s / H, h = qpairs ? qpairs[2 * s + 1] : s % H;
            const int u = map[i];
            int L;
            size_t row0, row_stride;
            if (kv_offsets) {
                L = kv_offsets[u + 1] - kv_offsets[u];
                row0 = ((size_t)kv_offsets[u] * H + h) * d;
                row_stride = (size_t)H * d;
            } else {
                L = Lkv;
                row0 = ((size_t)u * H + h) * (size_t)Lkv * d;
                row_stride = (size_t)d;
            }
            for (int q = 0; q < Lq; ++q) {
                double *out = dQ + ((size_t)s * Lq + q) * d;
                for (int c = 0; c < d; ++c) out[c] = 0.0;
                if (L == 0) continue;
                attn_row(Q + (((size_t)i * H + h) * Lq + q) * d, dO + (((size_t)i * H + h) * Lq + q) * d, K, V, row0,
                         row_stride, L, d, scale, p, ds);
                for (int j = 0; j < L; ++j) {
                    const uint16_t *kr = K + row0 + (size_t)j * row_stride;
                    for (int c = 0; c < d; ++c) out[c] += scale * ds[j] * bf16_bits_to_double(kr[c]);
                }
            }
        }
        /* dK, dV: every query of every candidate of u */
#pragma omp for schedule(dynamic, 1)
        for (int s = 0; s < n_kvsel; ++s) {
            if (!p || !ds) continue;
            const int u = kvpairs ? kvpairs[2 * s] : s / H, h = kvpairs ? kvpairs[2 * s + 1] : s % H;
            int L;
            size_t row0, row_stride;
            if (kv_offsets) {
                L = kv_offsets[u + 1] - kv_offsets[u];
                row0 = ((size_t)kv_offsets[u] * H + h) * d;
                row_stride = (size_t)H * d;
            } else {
                L = Lkv;
                row0 = ((size_t)u * H + h) * (size_t)Lkv * d;
                row_stride = (size_t)d;
            }
            double *gk = dK + (size_t)s * max_len * d, *gv = dV + (size_t)s * max_len * d;
            for (size_t e = 0; e < (size_t)max_len * d; ++e) gk[e] = gv[e] = 0.0;
            for (int i = 0; i < n_cand; ++i) {
                if (map[i] != u || L == 0) continue;
                for (int q = 0; q < Lq; ++q) {
                    attn_row(Q + (((size_t)i * H + h) * Lq + q) * d, dO + (((size_t)i * H + h) * Lq + q) * d, K, V,
                             row0, row_stride, L, d, scale, p, ds);
                    const uint16_t *qr = Q + (((size_t)i * H + h) * Lq + q) * d;
                    const uint16_t *gr = dO + (((size_t)i * H + h) * Lq + q) * d;
                    for (int j = 0; j < L; ++j)
                        for (int c = 0; c < d; ++c) {
                            gk[(size_t)j * d + c] += scale * ds[j] * bf16_bits_to_double(qr[c]);
                            gv[(size_t)j * d + c] += p[j] * bf16_bits_to_double(gr[c]);
                        }
                }
            }
        }
        free(p);
        free(ds);
    }
    return status;
}
