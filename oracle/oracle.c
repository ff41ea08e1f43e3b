/*
 * oracle.c -- float64 CPU oracle for exact softmax attention and for the
 * split-KV (partial-state) form of it.
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the package's smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  The CUDA library never
 * loads this code, and the two share no source, header, table or helper.
 *
 * Sources (web pages, cited by title and section):
 *   [T1] "FlashAttention 简化版：Tiling + Online Softmax" (forceinjection.github.io)
 *   [T2] "Flash Attention 代码填空 (Level 2-3)" (boots-coder.github.io, LLM-101-CN)
 *   [T3] "CS349E 第 11 讲 01_online_softmax.py" (semidirectx.com)
 *   [T4] "从零手写 FlashAttention（PyTorch实现 + 原理推导）" (mokono.cn)
 *
 * What is computed.  Attention is the plain three-step definition
 *   S = Q K^T * scale,   P = softmax(S) along each row,   O = P V
 * ([T1] §1.1; [T2] Exercise 1; [T3] attn_row_3pass), with the numerically
 * stable softmax that subtracts the row maximum before exponentiating
 * ([T1] §2.1; [T2] Exercise 2 safe_softmax; [T4] §3).  For each query row this
 * file stores the whole score row and walks it three times: once for the
 * maximum, once for exp and the sum, once to weight V ([T3] attn_row_3pass,
 * "3 遍").  The log-sum-exp of a row is m + ln(l) in natural log and in units
 * of the scaled score ([T3] demo 2, the remark on the (o_s, lse_s) encoding).
 *
 * Partial states.  For a segment of keys the state (m, l, o) is the segment's
 * score maximum m, l = sum exp(s - m), and the UNNORMALISED o = sum exp(s - m) v;
 * finishing a state divides o by l ([T3] demo 2 and attn_row_1pass).  Two
 * states merge by rescaling both to the larger maximum ([T3] demo 2, the
 * merge rule; [T1] §2.2 correction = exp(m_old - m_new)).  A state over zero
 * keys is (m = -inf, l = 0, o = 0); it is the identity of the merge, and
 * merging two empty states yields an empty state (reading: the pages do not
 * treat empty segments; this is the only value that keeps the merge
 * associative).
 *
 * Arithmetic is IEEE double throughout; inputs are given as doubles (the
 * caller up-casts the exact stored bf16/fp32 values).  exp/log come from libm.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define FAO_OK 0
#define FAO_BAD_ARG (-1)
#define FAO_NO_MEM (-2)

/* One query row against nk keys: the three passes over a stored score row. */
static void attention_row_3pass(const double* qrow, const double* k,
                                const double* v, double* orow, double* lse,
                                long nk, long d, double scale, double* s)
{
    /* scores s_j = scale * <q, k_j> */
    for (long j = 0; j < nk; ++j) {
        double acc = 0.0;
        const double* kj = k + j * d;
        for (long c = 0; c < d; ++c) acc += qrow[c] * kj[c];
        s[j] = scale * acc;
    }
    /* pass 1: the row maximum */
    double m = s[0];
    for (long j = 1; j < nk; ++j)
        if (s[j] > m) m = s[j];
    /* pass 2: exponentiate relative to the maximum, and sum */
    double l = 0.0;
    for (long j = 0; j < nk; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    /* pass 3: normalise the probabilities and weight the value rows */
    for (long c = 0; c < d; ++c) orow[c] = 0.0;
    for (long j = 0; j < nk; ++j) {
        const double p = s[j] / l;
        const double* vj = v + j * d;
        for (long c = 0; c < d; ++c) orow[c] += p * vj[c];
    }
    if (lse) *lse = m + log(l);
}

/*
 * Exact attention for one head.
 *   q [nq, d], k [nk, d], v [nk, d] row-major; o [nq, d]; lse [nq] or NULL.
 * Returns FAO_OK, FAO_BAD_ARG (nq < 0, nk < 1, d < 1, NULL buffers) or
 * FAO_NO_MEM.
 */
int fao_attention_head(const double* q, const double* k, const double* v,
                       double* o, double* lse, long nq, long nk, long d,
                       double scale)
{
    if (nq < 0 || nk < 1 || d < 1) return FAO_BAD_ARG;
    if (nq == 0) return FAO_OK;
    if (!q || !k || !v || !o) return FAO_BAD_ARG;
    double* s = (double*)malloc((size_t)nk * sizeof(double));
    if (!s) return FAO_NO_MEM;
    for (long i = 0; i < nq; ++i)
        attention_row_3pass(q + i * d, k, v, o + i * d, lse ? lse + i : NULL,
                            nk, d, scale, s);
    free(s);
    return FAO_OK;
}

/*
 * Exact attention for one head where query row i sees only its first
 * limits[i] keys (1 <= limits[i] <= nk): the softmax runs over keys
 * 0 .. limits[i]-1 only.  A causal mask is one choice of limits.
 */
int fao_attention_head_limits(const double* q, const double* k, const double* v,
                              double* o, double* lse, long nq, long nk, long d,
                              double scale, const long* limits)
{
    if (nq < 0 || nk < 1 || d < 1 || !limits) return FAO_BAD_ARG;
    if (nq == 0) return FAO_OK;
    if (!q || !k || !v || !o) return FAO_BAD_ARG;
    for (long i = 0; i < nq; ++i)
        if (limits[i] < 1 || limits[i] > nk) return FAO_BAD_ARG;
    double* s = (double*)malloc((size_t)nk * sizeof(double));
    if (!s) return FAO_NO_MEM;
    for (long i = 0; i < nq; ++i)
        attention_row_3pass(q + i * d, k, v, o + i * d, lse ? lse + i : NULL,
                            limits[i], d, scale, s);
    free(s);
    return FAO_OK;
}

/*
 * Exact attention over [B, H, N, d] contiguous tensors (each head on its own).
 * lse is [B, H, nq] or NULL.
 */
int fao_attention(const double* q, const double* k, const double* v, double* o,
                  double* lse, long B, long H, long nq, long nk, long d,
                  double scale)
{
    if (B < 0 || H < 0) return FAO_BAD_ARG;
    for (long bh = 0; bh < B * H; ++bh) {
        int rc = fao_attention_head(q + bh * nq * d, k + bh * nk * d,
                                    v + bh * nk * d, o + bh * nq * d,
                                    lse ? lse + bh * nq : NULL, nq, nk, d, scale);
        if (rc != FAO_OK) return rc;
    }
    return FAO_OK;
}

/*
 * Partial state (m, l, o) of one query against a segment of nk >= 0 keys.
 * o [d] receives the unnormalised weighted sum.  nk == 0 gives the empty state.
 */
int fao_partial_state(const double* q, const double* k, const double* v,
                      long nk, long d, double scale, double* m, double* l,
                      double* o)
{
    if (nk < 0 || d < 1 || !m || !l || !o) return FAO_BAD_ARG;
    for (long c = 0; c < d; ++c) o[c] = 0.0;
    if (nk == 0) {
        *m = -INFINITY;
        *l = 0.0;
        return FAO_OK;
    }
    double* s = (double*)malloc((size_t)nk * sizeof(double));
    if (!s) return FAO_NO_MEM;
    for (long j = 0; j < nk; ++j) {
        double acc = 0.0;
        for (long c = 0; c < d; ++c) acc += q[c] * k[j * d + c];
        s[j] = scale * acc;
    }
    double mx = s[0];
    for (long j = 1; j < nk; ++j)
        if (s[j] > mx) mx = s[j];
    double sum = 0.0;
    for (long j = 0; j < nk; ++j) {
        const double e = exp(s[j] - mx);
        sum += e;
        for (long c = 0; c < d; ++c) o[c] += e * v[j * d + c];
    }
    free(s);
    *m = mx;
    *l = sum;
    return FAO_OK;
}

/*
 * Merge two partial states into (m, l, o).  o may alias oa or ob.
 *   M = max(ma, mb);  l = la e^{ma-M} + lb e^{mb-M};  o = oa e^{ma-M} + ob e^{mb-M}
 */
void fao_merge_states(double ma, double la, const double* oa, double mb,
                      double lb, const double* ob, long d, double* m,
                      double* l, double* o)
{
    const double M = ma > mb ? ma : mb;
    if (M == -INFINITY) { /* both empty */
        for (long c = 0; c < d; ++c) o[c] = 0.0;
        *m = -INFINITY;
        *l = 0.0;
        return;
    }
    const double wa = (ma == -INFINITY) ? 0.0 : exp(ma - M);
    const double wb = (mb == -INFINITY) ? 0.0 : exp(mb - M);
    for (long c = 0; c < d; ++c) o[c] = oa[c] * wa + ob[c] * wb;
    *l = la * wa + lb * wb;
    *m = M;
}

/*
 * Split-KV attention for one query per head.
 *   q [B*H, d], k/v [B*H, nk, d], o [B*H, d], lse [B*H] or NULL.
 * Keys are cut into `splits` chunks of L = ceil(nk / splits) keys (the last
 * chunks may be shorter or empty).  Each chunk yields a partial state; the
 * states are merged one after another in the order given by `order` (a
 * permutation of 0..splits-1; NULL means index order), and the merged state
 * is finished as o / l.
 */
int fao_decode_splitkv(const double* q, const double* k, const double* v,
                       double* o, double* lse, long BH, long nk, long d,
                       long splits, double scale, const int* order)
{
    if (BH < 0 || nk < 1 || d < 1 || splits < 1 || splits > nk) return FAO_BAD_ARG;
    if (order) { /* must be a permutation */
        char* seen = (char*)calloc((size_t)splits, 1);
        if (!seen) return FAO_NO_MEM;
        for (long i = 0; i < splits; ++i) {
            if (order[i] < 0 || order[i] >= splits || seen[order[i]]) {
                free(seen);
                return FAO_BAD_ARG;
            }
            seen[order[i]] = 1;
        }
        free(seen);
    }
    const long L = (nk + splits - 1) / splits;
    double* st_o = (double*)malloc((size_t)d * sizeof(double));
    double* acc_o = (double*)malloc((size_t)d * sizeof(double));
    if (!st_o || !acc_o) {
        free(st_o);
        free(acc_o);
        return FAO_NO_MEM;
    }
    int rc = FAO_OK;
    for (long bh = 0; bh < BH && rc == FAO_OK; ++bh) {
        const double* qh = q + bh * d;
        const double* kh = k + bh * nk * d;
        const double* vh = v + bh * nk * d;
        double acc_m = -INFINITY, acc_l = 0.0;
        for (long c = 0; c < d; ++c) acc_o[c] = 0.0;
        for (long i = 0; i < splits; ++i) {
            const long c = order ? order[i] : i;
            long a = c * L, b = a + L;
            if (a > nk) a = nk;
            if (b > nk) b = nk;
            double sm, sl;
            rc = fao_partial_state(qh, kh + a * d, vh + a * d, b - a, d, scale,
                                   &sm, &sl, st_o);
            if (rc != FAO_OK) break;
            fao_merge_states(acc_m, acc_l, acc_o, sm, sl, st_o, d, &acc_m,
                             &acc_l, acc_o);
        }
        for (long c = 0; c < d; ++c) o[bh * d + c] = acc_o[c] / acc_l;
        if (lse) lse[bh] = acc_m + log(acc_l);
    }
    free(st_o);
    free(acc_o);
    return rc;
}

/*
 * Gradients of exact attention for one head, from the plain definition.
 *   Forward:  S = scale Q K^T,  P = row-softmax(S),  O = P V.
 *   Given dO (the gradient of a loss with respect to O):
 *     dV = P^T dO                                  ([T2] Exercise 5: dV_j = sum_i P_ij^T dO_i)
 *     dP = dO V^T
 *     dS_ij = P_ij (dP_ij - D_i),  D_i = sum_c dO_ic O_ic   (softmax Jacobian, row by row)
 *     dQ = scale dS K,   dK = scale dS^T Q
 *   (the chain rule through S = scale Q K^T; the pages give only dV, the rest is calculus).
 *   q, dq [nq, d]; k, v, dk, dv [nk, d]; dout [nq, d].  Plain loops, O(nq nk d).
 *   limits[i], if not NULL, is the number of leading keys row i sees (1 .. nk): the other
 *   keys get P_ij = 0, so they receive no gradient from row i.
 */
int fao_attention_bwd_head_limits(const double* q, const double* k, const double* v,
                                  const double* dout, double* dq, double* dk, double* dv,
                                  long nq, long nk, long d, double scale, const long* limits)
{
    if (nq < 1 || nk < 1 || d < 1) return FAO_BAD_ARG;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return FAO_BAD_ARG;
    if (limits)
        for (long i = 0; i < nq; ++i)
            if (limits[i] < 1 || limits[i] > nk) return FAO_BAD_ARG;
    double* P = (double*)malloc((size_t)nq * nk * sizeof(double));
    double* orow = (double*)malloc((size_t)d * sizeof(double));
    if (!P || !orow) {
        free(P);
        free(orow);
        return FAO_NO_MEM;
    }
    for (long i = 0; i < nq; ++i) { /* P row by row: scores, max, exp, normalise; masked keys get P = 0 */
        double* p = P + i * nk;
        const long n_i = limits ? limits[i] : nk;
        for (long j = 0; j < n_i; ++j) {
            double acc = 0.0;
            for (long c = 0; c < d; ++c) acc += q[i * d + c] * k[j * d + c];
            p[j] = scale * acc;
        }
        double m = p[0];
        for (long j = 1; j < n_i; ++j)
            if (p[j] > m) m = p[j];
        double l = 0.0;
        for (long j = 0; j < n_i; ++j) {
            p[j] = exp(p[j] - m);
            l += p[j];
        }
        for (long j = 0; j < n_i; ++j) p[j] /= l;
        for (long j = n_i; j < nk; ++j) p[j] = 0.0;
    }
    for (long x = 0; x < nq * d; ++x) dq[x] = 0.0;
    for (long x = 0; x < nk * d; ++x) dk[x] = dv[x] = 0.0;
    for (long i = 0; i < nq; ++i) {
        const double* p = P + i * nk;
        const double* go = dout + i * d;
        /* O_i and D_i = <dO_i, O_i> */
        for (long c = 0; c < d; ++c) orow[c] = 0.0;
        for (long j = 0; j < nk; ++j)
            for (long c = 0; c < d; ++c) orow[c] += p[j] * v[j * d + c];
        double Di = 0.0;
        for (long c = 0; c < d; ++c) Di += go[c] * orow[c];
        for (long j = 0; j < nk; ++j) {
            /* dV_j += P_ij dO_i */
            for (long c = 0; c < d; ++c) dv[j * d + c] += p[j] * go[c];
            /* dP_ij = <dO_i, V_j>,  dS_ij = P_ij (dP_ij - D_i) */
            double dp = 0.0;
            for (long c = 0; c < d; ++c) dp += go[c] * v[j * d + c];
            const double ds = p[j] * (dp - Di);
            for (long c = 0; c < d; ++c) {
                dq[i * d + c] += scale * ds * k[j * d + c];
                dk[j * d + c] += scale * ds * q[i * d + c];
            }
        }
    }
    free(P);
    free(orow);
    return FAO_OK;
}

/* Unmasked gradients: every query row sees all nk keys. */
int fao_attention_bwd_head(const double* q, const double* k, const double* v,
                           const double* dout, double* dq, double* dk, double* dv,
                           long nq, long nk, long d, double scale)
{
    return fao_attention_bwd_head_limits(q, k, v, dout, dq, dk, dv, nq, nk, d, scale, NULL);
}
