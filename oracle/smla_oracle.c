/*
 * smla_oracle.c -- plain, slow, fp64 CPU oracle for DeepSeek-V4-style sparse
 * MLA attention (forward and training backward).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline do. It shares no code, header, table or helper with the CUDA
 * library; the two meet only at the seeded inputs.
 *
 * Source of the definitions: the aiter pull request "[WIP][TRITON][GLUON]
 * [GFX950][DSV4] Sparse MLA training backward", sections "Contract" and
 * "Structure":
 *   - shared-KV GQA: K == V == kv, one dense [num_kv, D] tensor (D = 512 in
 *     the contract; the oracle takes D as a parameter so finite-difference
 *     checks can run at small D);
 *   - scale 1/sqrt(512) in the scores;
 *   - attn_sink folded into the softmax denominator only;
 *   - topk_indices == -1 masked out;
 *   - lse is sink-inclusive: lse = e_max + log(e_sum) with the sink folded
 *     into e_max / e_sum;
 *   - delta = rowsum(O * dO) from the given O;
 *   - dKV is the scatter of the per-(t, rank) intermediate
 *     sum_h P*dO + dS*q, inverted into a per-kv-row CSR and gathered.
 * Readings where the page is silent:
 *   sink is a logit in the scaled score domain; lse uses the natural log;
 *   no sink means no denominator term and no d_sink; a row with no valid rank
 *   gets O = 0, lse = sink (or -inf) and contributes no gradient; duplicate
 *   indices count once per slot; indices outside [-1, num_kv) are an error.
 *
 * Every accumulation is in double. Inputs are given as double arrays (the
 * Python wrapper converts bf16 / fp32 bit patterns exactly); outputs are
 * double. Loops follow the definitions directly: no tiling, no fusion, no
 * reordering beyond splitting independent outputs across OpenMP threads.
 */

#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_INDEX 2
#define OR_ERR_NOMEM 3

typedef int64_t i64;

int smla_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static double dot(const double* a, const double* b, i64 n) {
    double s = 0.0;
    for (i64 i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* Every index must be -1 (masked) or a row of kv. */
static int check_indices(const int32_t* topk, i64 count, i64 N) {
    for (i64 i = 0; i < count; ++i)
        if (topk[i] < -1 || topk[i] >= N) return OR_ERR_INDEX;
    return OR_OK;
}

/*
 * Forward ("Contract" section; lse convention in the paragraph under the
 * usage example). For each token t and head h, over the valid ranks r:
 *   s_r   = scale * <q[t,h,:], kv[idx_r,:]>
 *   m     = max(sink_h, max_r s_r)
 *   e     = exp(sink_h - m) + sum_r exp(s_r - m)
 *   lse   = m + log(e)
 *   O     = sum_r exp(s_r - lse) * kv[idx_r,:]
 * The sink has no value row. sink == NULL means no sink term at all.
 */
int smla_oracle_fwd(i64 T, i64 H, i64 D, i64 K, i64 N,
                    const double* q, const double* kv, const int32_t* topk,
                    const double* sink, double scale,
                    double* o, double* lse) {
    if (T < 0 || H <= 0 || D <= 0 || K < 0 || N <= 0) return OR_ERR_ARG;
    if (check_indices(topk, T * K, N)) return OR_ERR_INDEX;
    int fail = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 th = 0; th < T * H; ++th) {
        const i64 t = th / H, h = th % H;
        const double* qv = q + (t * H + h) * D;
        const int32_t* row = topk + t * K;
        double* s = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!s) { fail = 1; continue; }
        double m = sink ? sink[h] : -INFINITY;
        for (i64 r = 0; r < K; ++r) {
            if (row[r] < 0) continue;
            s[r] = scale * dot(qv, kv + (i64)row[r] * D, D);
            if (s[r] > m) m = s[r];
        }
        double* out = o + (t * H + h) * D;
        memset(out, 0, sizeof(double) * (size_t)D);
        if (m == -INFINITY) {              /* no valid rank and no sink */
            lse[t * H + h] = -INFINITY;
            free(s);
            continue;
        }
        double e = sink ? exp(sink[h] - m) : 0.0;
        for (i64 r = 0; r < K; ++r)
            if (row[r] >= 0) e += exp(s[r] - m);
        const double l = m + log(e);
        lse[t * H + h] = l;
        for (i64 r = 0; r < K; ++r) {
            if (row[r] < 0) continue;
            const double p = exp(s[r] - l);
            const double* kr = kv + (i64)row[r] * D;
            for (i64 d = 0; d < D; ++d) out[d] += p * kr[d];
        }
        free(s);
    }
    return fail ? OR_ERR_NOMEM : OR_OK;
}

/*
 * Per-(t, h, r) backward quantities from the given inputs ("Structure"
 * table: the delta phase, then the dQ phase):
 *   delta = sum_d O[t,h,d] * dO[t,h,d]
 *   P     = exp(s - lse[t,h])              (s as in the forward)
 *   dP    = <dO[t,h,:], kv[idx,:]>          (V == kv)
 *   dS    = P * (dP - delta)
 */
static void rank_grads(i64 D, const double* qv, const double* dov,
                       const double* kr, double scale, double lse_th,
                       double delta_th, double* P, double* dS) {
    const double s = scale * dot(qv, kr, D);
    const double p = exp(s - lse_th);
    const double dp = dot(dov, kr, D);
    *P = p;
    *dS = p * (dp - delta_th);
}

/*
 * Full backward on small problems.
 *   dq[t,h,:]  = scale * sum_r dS * kv[idx_r,:]
 *   dkv[j,:]   = sum over (t,h,r) with idx = j of P*dO[t,h,:] + scale*dS*q[t,h,:]
 *                (K-path plus V-path gradient, K == V == kv), summed in
 *                ascending (t, r) order with h innermost -- the scatter form
 *   d_sink[h]  = -sum_t exp(sink_h - lse[t,h]) * delta[t,h]
 *                (the sink's softmax weight times (0 - delta): the sink has
 *                no value row)
 * Any of dq, dkv, dsink, delta_out may be NULL. dsink must be NULL when
 * sink is NULL.
 */
int smla_oracle_bwd(i64 T, i64 H, i64 D, i64 K, i64 N,
                    const double* q, const double* kv, const double* dout,
                    const double* o, const double* lse, const int32_t* topk,
                    const double* sink, double scale,
                    double* dq, double* dkv, double* dsink, double* delta_out) {
    if (T < 0 || H <= 0 || D <= 0 || K < 0 || N <= 0) return OR_ERR_ARG;
    if (dsink && !sink) return OR_ERR_ARG;
    if (check_indices(topk, T * K, N)) return OR_ERR_INDEX;

    double* delta = (double*)malloc(sizeof(double) * (size_t)(T * H > 0 ? T * H : 1));
    double* P = (double*)malloc(sizeof(double) * (size_t)(T * H * K > 0 ? T * H * K : 1));
    double* dS = (double*)malloc(sizeof(double) * (size_t)(T * H * K > 0 ? T * H * K : 1));
    if (!delta || !P || !dS) { free(delta); free(P); free(dS); return OR_ERR_NOMEM; }

#pragma omp parallel for schedule(static)
    for (i64 th = 0; th < T * H; ++th)
        delta[th] = dot(o + th * D, dout + th * D, D);

#pragma omp parallel for schedule(dynamic, 1)
    for (i64 th = 0; th < T * H; ++th) {
        const i64 t = th / H;
        const int32_t* row = topk + t * K;
        for (i64 r = 0; r < K; ++r) {
            double p = 0.0, ds = 0.0;
            if (row[r] >= 0)
                rank_grads(D, q + th * D, dout + th * D, kv + (i64)row[r] * D,
                           scale, lse[th], delta[th], &p, &ds);
            P[th * K + r] = p;
            dS[th * K + r] = ds;
        }
        if (dq) {
            double* g = dq + th * D;
            memset(g, 0, sizeof(double) * (size_t)D);
            for (i64 r = 0; r < K; ++r) {
                if (row[r] < 0) continue;
                const double c = scale * dS[th * K + r];
                const double* kr = kv + (i64)row[r] * D;
                for (i64 d = 0; d < D; ++d) g[d] += c * kr[d];
            }
        }
    }

    if (dkv) {
        memset(dkv, 0, sizeof(double) * (size_t)(N * D));
        /* Scatter in (t, r, h) order; threads own disjoint column ranges of
         * dkv, so each element still sees that exact order. */
        const i64 DB = 16;
#pragma omp parallel for schedule(dynamic, 1)
        for (i64 d0 = 0; d0 < D; d0 += DB) {
            const i64 d1 = d0 + DB < D ? d0 + DB : D;
            for (i64 t = 0; t < T; ++t)
                for (i64 r = 0; r < K; ++r) {
                    const int32_t j = topk[t * K + r];
                    if (j < 0) continue;
                    double* g = dkv + (i64)j * D;
                    for (i64 h = 0; h < H; ++h) {
                        const i64 th = t * H + h;
                        const double p = P[th * K + r];
                        const double c = scale * dS[th * K + r];
                        for (i64 d = d0; d < d1; ++d)
                            g[d] += p * dout[th * D + d] + c * q[th * D + d];
                    }
                }
        }
    }

    if (dsink) {
        for (i64 h = 0; h < H; ++h) {
            double acc = 0.0;
            for (i64 t = 0; t < T; ++t) {
                const i64 th = t * H + h;
                acc -= exp(sink[h] - lse[th]) * delta[th];
            }
            dsink[h] = acc;
        }
    }
    if (delta_out) memcpy(delta_out, delta, sizeof(double) * (size_t)(T * H));
    free(delta); free(P); free(dS);
    return OR_OK;
}

/*
 * Inverted top-k CSR over the ranks [r0, r0 + R) of each row ("Structure":
 * CSR build; the flat position p = t*R + (r - r0) indexes the [T, R, D]
 * intermediate of the dKV gather). For every kv row j:
 *   row_ptr[j]                      = number of valid entries with key < j
 *   col[row_ptr[j] .. row_ptr[j+1]) = the positions p with key j, ascending
 * Entries equal to -1 are dropped. The page sorts with torch.sort on int16
 * keys and leaves the order inside a row unspecified; ascending p (a stable
 * counting sort) is the reading fixed here.
 */
int smla_oracle_csr(const int32_t* topk, i64 T, i64 Kw, i64 r0, i64 R, i64 N,
                    int32_t* row_ptr, int32_t* col) {
    if (T < 0 || Kw < 0 || R < 0 || r0 < 0 || r0 + R > Kw || N <= 0) return OR_ERR_ARG;
    for (i64 t = 0; t < T; ++t)
        if (check_indices(topk + t * Kw + r0, R, N)) return OR_ERR_INDEX;
    i64* count = (i64*)calloc((size_t)N + 1, sizeof(i64));
    if (!count) return OR_ERR_NOMEM;
    for (i64 t = 0; t < T; ++t)
        for (i64 r = 0; r < R; ++r) {
            const int32_t j = topk[t * Kw + r0 + r];
            if (j >= 0) count[j + 1] += 1;
        }
    row_ptr[0] = 0;
    for (i64 j = 0; j < N; ++j) {
        count[j + 1] += count[j];
        row_ptr[j + 1] = (int32_t)count[j + 1];
    }
    /* count[j] is now the next free slot of row j; walking p upward keeps
     * each row ascending. */
    for (i64 t = 0; t < T; ++t)
        for (i64 r = 0; r < R; ++r) {
            const int32_t j = topk[t * Kw + r0 + r];
            if (j < 0) continue;
            col[count[j]++] = (int32_t)(t * R + r);
        }
    free(count);
    return OR_OK;
}

/*
 * dkv for selected kv rows by the CSR-gather form ("Structure": dKV-interm
 * then the atomic-free dKV gather): for row j, walk its CSR entries p in
 * order; p = t*R + (r - r0) names token t and rank r; form
 *   interm[p,:] = sum_h P[t,h,r]*dO[t,h,:] + scale*dS[t,h,r]*q[t,h,:]
 * and add it to the row. Only the chunk [r0, r0+R) of ranks is covered; a
 * caller sums the chunks in order for the whole result.
 * out is [nrows, D].
 */
int smla_oracle_dkv_rows(i64 T, i64 H, i64 D, i64 K, i64 N,
                         const double* q, const double* kv, const double* dout,
                         const double* o, const double* lse, const int32_t* topk,
                         double scale, i64 r0, i64 R,
                         const int32_t* row_ptr, const int32_t* col,
                         const int64_t* rows, i64 nrows, double* out) {
    if (T < 0 || H <= 0 || D <= 0 || K < 0 || N <= 0 || r0 < 0 || R <= 0 || r0 + R > K)
        return OR_ERR_ARG;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 i = 0; i < nrows; ++i) {
        const i64 j = rows[i];
        double* g = out + i * D;
        memset(g, 0, sizeof(double) * (size_t)D);
        if (j < 0 || j >= N) { bad = 1; continue; }
        double* interm = (double*)malloc(sizeof(double) * (size_t)D);
        if (!interm) { bad = 1; continue; }
        for (i64 e = row_ptr[j]; e < row_ptr[j + 1]; ++e) {
            const i64 p = col[e];
            const i64 t = p / R, r = r0 + p % R;
            if (topk[t * K + r] != j) { bad = 1; break; }
            memset(interm, 0, sizeof(double) * (size_t)D);
            for (i64 h = 0; h < H; ++h) {
                const i64 th = t * H + h;
                const double delta = dot(o + th * D, dout + th * D, D);
                double pr, ds;
                rank_grads(D, q + th * D, dout + th * D, kv + j * D, scale,
                           lse[th], delta, &pr, &ds);
                const double c = scale * ds;
                for (i64 d = 0; d < D; ++d)
                    interm[d] += pr * dout[th * D + d] + c * q[th * D + d];
            }
            for (i64 d = 0; d < D; ++d) g[d] += interm[d];
        }
        free(interm);
    }
    return bad ? OR_ERR_ARG : OR_OK;
}

/*
 * dq for selected tokens (the dQ phase): for token t and head h,
 *   dq[t,h,:] = scale * sum_r dS[t,h,r] * kv[idx_r,:].
 * out is [ntok, H, D].
 */
int smla_oracle_dq_tokens(i64 T, i64 H, i64 D, i64 K, i64 N,
                          const double* q, const double* kv, const double* dout,
                          const double* o, const double* lse, const int32_t* topk,
                          double scale, const int64_t* tokens, i64 ntok,
                          double* out) {
    if (T < 0 || H <= 0 || D <= 0 || K < 0 || N <= 0) return OR_ERR_ARG;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (i64 ih = 0; ih < ntok * H; ++ih) {
        const i64 i = ih / H, h = ih % H;
        const i64 t = tokens[i];
        double* g = out + ih * D;
        memset(g, 0, sizeof(double) * (size_t)D);
        if (t < 0 || t >= T) { bad = 1; continue; }
        const i64 th = t * H + h;
        const double delta = dot(o + th * D, dout + th * D, D);
        for (i64 r = 0; r < K; ++r) {
            const int32_t j = topk[t * K + r];
            if (j < 0) continue;
            if (j >= N) { bad = 1; break; }
            double p, ds;
            rank_grads(D, q + th * D, dout + th * D, kv + (i64)j * D, scale,
                       lse[th], delta, &p, &ds);
            const double c = scale * ds;
            for (i64 d = 0; d < D; ++d) g[d] += c * kv[(i64)j * D + d];
        }
    }
    return bad ? OR_ERR_ARG : OR_OK;
}

/*
 * d_sink and delta alone: d_sink[h] = -sum_t exp(sink_h - lse[t,h]) * delta[t,h]
 * with delta = rowsum(O * dO).
 */
int smla_oracle_dsink(i64 T, i64 H, i64 D, const double* dout, const double* o,
                      const double* lse, const double* sink, double* dsink,
                      double* delta_out) {
    if (T < 0 || H <= 0 || D <= 0 || !sink) return OR_ERR_ARG;
    for (i64 h = 0; h < H; ++h) dsink[h] = 0.0;
    for (i64 t = 0; t < T; ++t)
        for (i64 h = 0; h < H; ++h) {
            const i64 th = t * H + h;
            const double delta = dot(o + th * D, dout + th * D, D);
            if (delta_out) delta_out[th] = delta;
            dsink[h] -= exp(sink[h] - lse[th]) * delta;
        }
    return OR_OK;
}
