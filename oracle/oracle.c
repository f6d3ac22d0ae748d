/*
 * oracle.c -- plain, slow, fp64 CPU oracle for blockwise ring attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or helper
 * with the CUDA path.
 *
 * Every floating-point step is done in double precision.  Inputs arrive as
 * float64 arrays; the Python wrapper widens bfloat16 tensors to them exactly.
 *
 * Sources restated here (page title, then section / equation):
 *  [P1] "Ring Attention with Blockwise Transformers: Mathematical Foundations,
 *       Circular KV Passing, Overlapped Communication-Computation, and Linear
 *       Context Scaling" -- "The Memory and Communication Bottlenecks" (the
 *       attention definition O = softmax(QK^T/sqrt(d))V), "Blockwise Attention
 *       and Online Softmax Formulations" (running max m, normaliser l,
 *       unnormalised O and their update; final division by l), "Causal Masking
 *       Dynamics" (token i sees tokens j <= i; striped assignment t -> t mod N).
 *  [P2] "Ring Attention for Infinite Context" -- "FlashAttention Integration"
 *       (rescale-merge of two partial outputs by e^(m_old-m_new), e^(m_blk-m_new)).
 *  [P3] the magicnetworld.com article on ring attention's communication
 *       budget, causal triangle and load imbalance -- section 6 (causal mask,
 *       contiguous vs striped token placement, 8-token / 4-device example).
 *  [P4] summary of "Ring Attention with Blockwise Transformers for
 *       Near-Infinite Context" -- "Incremental Blockwise Attention" (steps 1-5
 *       of the statistics update), "The Ring Communication Protocol"
 *       (k_block_idx = (axis_index - idx) mod N), "The Backward Pass".
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): the log-sum-exp is in natural-log units, LSE = m + ln l; GQA maps
 * query head hq to KV head hq / (h / n_kv); the causal rule is inclusive
 * (key position <= query position); a row that sees no key has O = 0 and
 * LSE = -inf.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_API __attribute__((visibility("default")))

static double dot(const double *a, const double *b, int d)
{
    double acc = 0.0;
    for (int e = 0; e < d; ++e)
        acc += a[e] * b[e];
    return acc;
}

/* ------------------------------------------------------------------------ */
/* Token placement.  [P3 section 6] contiguous: [0,1][2,3][4,5][6,7];
 * striped (stride N): [0,4][1,5][2,6][3,7].  [P1 "Striped Attention"]: token
 * t goes to device t mod N.  [P1 "Zig-Zag Ring Attention"]: the sequence is
 * cut into 2N half-blocks of C = S / 2N tokens and device p holds half-blocks
 * p and 2N-1-p; reading (recorded in the design notes): the early half-block
 * comes first in local order, so local rows [0, C) are tokens [pC, pC+C) and
 * rows [C, 2C) are tokens [(2N-1-p)C, (2N-p)C).
 * layout 0 = contiguous, 1 = striped, 2 = zig-zag.
 * shard_of[t], local_of[t] for every token; token_of[p*L + r] inverse map.  */
ORC_API int orc_position_map(int layout, int64_t S, int N, int32_t *shard_of,
                             int32_t *local_of, int32_t *token_of)
{
    if (N <= 0 || S < 0 || S % N != 0 || layout < 0 || layout > 2)
        return 1;
    if (layout == 2 && S % (2 * (int64_t)N) != 0)
        return 1;
    int64_t L = S / N;
    for (int64_t t = 0; t < S; ++t) {
        int64_t p, r;
        if (layout == 0) {
            p = t / L;
            r = t % L;
        } else if (layout == 1) {
            p = t % N;
            r = t / N;
        } else {
            int64_t C = L / 2;
            int64_t half = t / C;              /* which of the 2N half-blocks */
            if (half < N) {
                p = half;
                r = t % C;
            } else {
                p = 2 * (int64_t)N - 1 - half;
                r = C + t % C;
            }
        }
        shard_of[t] = (int32_t)p;
        local_of[t] = (int32_t)r;
        token_of[p * L + r] = (int32_t)t;
    }
    return 0;
}

/* [P4 "The Ring Communication Protocol"]: on scan iteration idx, host i holds
 * the key/value block that started on host (i - idx) mod N.  order[i*N + s]. */
ORC_API void orc_ring_order(int N, int32_t *order)
{
    for (int i = 0; i < N; ++i)
        for (int s = 0; s < N; ++s)
            order[i * N + s] = (int32_t)(((i - s) % N + N) % N);
}

/* ------------------------------------------------------------------------ */
/* Thread control for timing the oracle (no arithmetic): the number of
 * OpenMP threads a parallel region uses, and a way to set it.             */
ORC_API int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

ORC_API void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* Keys query token t sees, as the interval [j0, j1).  Without documents all
 * S keys, or under the causal rule keys 0..t.  Packed documents ([P3 section
 * 5], "packing" with a block-diagonal mask): doc_start / doc_end [b, S] give
 * the first token and one past the last token of t's document, and t sees
 * only keys of its own document (and, causal, not after t).               */
static void visible_keys(int64_t t, int64_t S, int causal, const int64_t *doc_start,
                         const int64_t *doc_end, int bb, int64_t *j0, int64_t *j1)
{
    int64_t lo = 0, hi = S;
    if (doc_start) {
        lo = doc_start[(int64_t)bb * S + t];
        hi = doc_end[(int64_t)bb * S + t];
    }
    if (causal && t + 1 < hi)
        hi = t + 1;
    *j0 = lo;
    *j1 = hi;
}

/* ------------------------------------------------------------------------ */
/* Direct definition, [P1 "The Memory and Communication Bottlenecks"] with the
 * causal rule of [P3 section 6] and GQA head sharing of [P3 section 2]:
 *   s_tj  = scale * <q_t, k_j>          for visible keys j
 *   LSE_t = ln sum_j exp(s_tj)           (max-subtracted, fp64)
 *   O_t   = sum_j exp(s_tj - LSE_t) v_j
 * Tokens are in natural order; key j is visible to query token t when not
 * causal, or when j <= t.  k, v [b,S,n_kv,d]; q_rows [b,R,h,d] holds the
 * queries of the R tokens rows[0..R).  out [b,R,h,d], lse [b,h,R].          */
ORC_API void orc_attn_fwd_rows(const double *q_rows, const double *k,
                               const double *v, int b, int64_t S, int h,
                               int n_kv, int d, int causal, double scale,
                               const int64_t *rows, int64_t R, double *out,
                               double *lse, const int64_t *doc_start,
                               const int64_t *doc_end)
{
    const int g = h / n_kv;
    const int64_t total = (int64_t)b * R * h;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
#pragma omp for schedule(dynamic, 4)
        for (int64_t w = 0; w < total; ++w) {
            const int hq = (int)(w % h);
            const int64_t ri = (w / h) % R;
            const int bb = (int)(w / ((int64_t)h * R));
            const int64_t t = rows[ri];
            const int kh = hq / g;
            const double *qt = q_rows + (((int64_t)bb * R + ri) * h + hq) * d;
            int64_t j0, nvis;
            visible_keys(t, S, causal, doc_start, doc_end, bb, &j0, &nvis);
            double *o = out + (((int64_t)bb * R + ri) * h + hq) * d;
            double *ls = lse + ((int64_t)bb * h + hq) * R + ri;
            for (int e = 0; e < d; ++e)
                o[e] = 0.0;
            if (nvis <= j0) {
                *ls = -INFINITY;
                continue;
            }
            double mx = -INFINITY;
            for (int64_t j = j0; j < nvis; ++j) {
                s[j] = scale * dot(qt, k + (((int64_t)bb * S + j) * n_kv + kh) * d, d);
                if (s[j] > mx)
                    mx = s[j];
            }
            double sum = 0.0;
            for (int64_t j = j0; j < nvis; ++j)
                sum += exp(s[j] - mx);
            const double lse_t = mx + log(sum);
            *ls = lse_t;
            for (int64_t j = j0; j < nvis; ++j) {
                const double p = exp(s[j] - lse_t);
                const double *vj = v + (((int64_t)bb * S + j) * n_kv + kh) * d;
                for (int e = 0; e < d; ++e)
                    o[e] += p * vj[e];
            }
        }
        free(s);
    }
}

/* ------------------------------------------------------------------------ */
/* Analytic gradient of the direct definition ([P4 "The Backward Pass"]: dV
 * from the attention weights and dO, dQ from the values, dK from the queries;
 * weights recomputed from the saved statistics):
 *   P_tj  = exp(s_tj - LSE_t),  O_t = sum_j P_tj v_j,  D_t = <dO_t, O_t>
 *   dV_j += P_tj dO_t
 *   dS_tj = P_tj (<dO_t, v_j> - D_t)
 *   dQ_t  = scale * sum_j dS_tj k_j
 *   dK_j += scale * dS_tj q_t
 * The upstream gradient dO is taken to be zero outside the listed rows, so dK
 * and dV are exactly the contributions of those rows (summed over the g query
 * heads sharing each KV head).  q_rows, dout_rows [b,R,h,d] hold those rows;
 * dq_rows [b,R,h,d]; dk, dv [b,S,n_kv,d] are overwritten.                   */
ORC_API void orc_attn_bwd_rows(const double *q_rows, const double *k,
                               const double *v, const double *dout_rows, int b,
                               int64_t S, int h, int n_kv, int d, int causal,
                               double scale, const int64_t *rows, int64_t R,
                               double *dq_rows, double *dk, double *dv,
                               const int64_t *doc_start, const int64_t *doc_end)
{
    const int g = h / n_kv;
    memset(dk, 0, sizeof(double) * (size_t)b * (size_t)S * n_kv * d);
    memset(dv, 0, sizeof(double) * (size_t)b * (size_t)S * n_kv * d);
    memset(dq_rows, 0, sizeof(double) * (size_t)b * (size_t)R * h * d);
    /* one (batch, kv head) per task: no two tasks touch the same dk/dv rows */
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
        double *o = (double *)malloc(sizeof(double) * (size_t)d);
#pragma omp for collapse(2) schedule(dynamic, 1)
        for (int bb = 0; bb < b; ++bb)
            for (int kh = 0; kh < n_kv; ++kh)
                for (int hq = kh * g; hq < (kh + 1) * g; ++hq)
                    for (int64_t ri = 0; ri < R; ++ri) {
                        const int64_t t = rows[ri];
                        int64_t j0, nvis;
                        visible_keys(t, S, causal, doc_start, doc_end, bb, &j0, &nvis);
                        if (nvis <= j0)
                            continue;
                        const double *qt = q_rows + (((int64_t)bb * R + ri) * h + hq) * d;
                        const double *gt = dout_rows + (((int64_t)bb * R + ri) * h + hq) * d;
                        double *dq = dq_rows + (((int64_t)bb * R + ri) * h + hq) * d;
                        double mx = -INFINITY;
                        for (int64_t j = j0; j < nvis; ++j) {
                            p[j] = scale * dot(qt, k + (((int64_t)bb * S + j) * n_kv + kh) * d, d);
                            if (p[j] > mx)
                                mx = p[j];
                        }
                        double sum = 0.0;
                        for (int64_t j = j0; j < nvis; ++j)
                            sum += exp(p[j] - mx);
                        const double lse_t = mx + log(sum);
                        for (int e = 0; e < d; ++e)
                            o[e] = 0.0;
                        for (int64_t j = j0; j < nvis; ++j) {
                            p[j] = exp(p[j] - lse_t); /* scores -> weights P_tj */
                            const double *vj = v + (((int64_t)bb * S + j) * n_kv + kh) * d;
                            for (int e = 0; e < d; ++e)
                                o[e] += p[j] * vj[e];
                        }
                        const double D = dot(gt, o, d);
                        for (int64_t j = j0; j < nvis; ++j) {
                            const int64_t kv_off = (((int64_t)bb * S + j) * n_kv + kh) * d;
                            const double ds = p[j] * (dot(gt, v + kv_off, d) - D);
                            const double *kj = k + kv_off;
                            double *dkj = dk + kv_off;
                            double *dvj = dv + kv_off;
                            for (int e = 0; e < d; ++e) {
                                dvj[e] += p[j] * gt[e];
                                dkj[e] += scale * ds * qt[e];
                                dq[e] += scale * ds * kj[e];
                            }
                        }
                    }
        free(o);
        free(p);
    }
}

/* ------------------------------------------------------------------------ */
/* One blockwise update, the recurrence of [P1 "Blockwise Attention and Online
 * Softmax Formulations"] / [P4 "Incremental Blockwise Attention" steps 1-5],
 * applied to one key/value block with explicit token positions:
 *   m~  = rowmax over visible keys of S = scale * Q K^T
 *   m'  = max(m, m~)
 *   P   = exp(S - m')                (masked entries contribute 0)
 *   l'  = exp(m - m') l + rowsum(P)
 *   O'  = exp(m - m') O + P V
 * A row with no visible key in this block is left unchanged.  The state
 * starts at m = -inf, l = 0, O = 0.
 * q [b,Lq,h,d]; k, v [b,Lk,n_kv,d]; q_pos [Lq]; k_pos [Lk];
 * m, l [b,h,Lq]; o [b,Lq,h,d] (unnormalised).                                */
ORC_API void orc_block_update(const double *q, const double *k, const double *v,
                              const int32_t *q_pos, const int32_t *k_pos, int b,
                              int64_t Lq, int64_t Lk, int h, int n_kv, int d,
                              int causal, double scale, double *m, double *l,
                              double *o)
{
    const int g = h / n_kv;
    const int64_t total = (int64_t)b * Lq * h;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Lk > 0 ? Lk : 1));
        unsigned char *vis = (unsigned char *)malloc((size_t)(Lk > 0 ? Lk : 1));
#pragma omp for schedule(dynamic, 8)
        for (int64_t w = 0; w < total; ++w) {
            const int hq = (int)(w % h);
            const int64_t r = (w / h) % Lq;
            const int bb = (int)(w / ((int64_t)h * Lq));
            const int kh = hq / g;
            const double *qr = q + (((int64_t)bb * Lq + r) * h + hq) * d;
            double mt = -INFINITY;
            int any = 0;
            for (int64_t j = 0; j < Lk; ++j) {
                vis[j] = (unsigned char)(!causal || k_pos[j] <= q_pos[r]);
                if (!vis[j])
                    continue;
                s[j] = scale * dot(qr, k + (((int64_t)bb * Lk + j) * n_kv + kh) * d, d);
                if (s[j] > mt)
                    mt = s[j];
                any = 1;
            }
            if (!any)
                continue;
            double *mr = m + ((int64_t)bb * h + hq) * Lq + r;
            double *lr = l + ((int64_t)bb * h + hq) * Lq + r;
            double *orow = o + (((int64_t)bb * Lq + r) * h + hq) * d;
            const double m_new = (*mr > mt) ? *mr : mt;
            const double alpha = exp(*mr - m_new); /* exp(-inf) = 0 */
            double rowsum = 0.0;
            for (int e = 0; e < d; ++e)
                orow[e] *= alpha;
            for (int64_t j = 0; j < Lk; ++j) {
                if (!vis[j])
                    continue;
                const double p = exp(s[j] - m_new);
                rowsum += p;
                const double *vj = v + (((int64_t)bb * Lk + j) * n_kv + kh) * d;
                for (int e = 0; e < d; ++e)
                    orow[e] += p * vj[e];
            }
            *lr = alpha * (*lr) + rowsum;
            *mr = m_new;
        }
        free(vis);
        free(s);
    }
}

/* Final division [P1 "Blockwise Attention ..."]: O* = diag(l)^-1 O, and
 * LSE = m + ln l.  A row with l = 0 saw no key: O* = 0, LSE = -inf.          */
ORC_API void orc_finalize(const double *o, const double *l, const double *m,
                          int b, int64_t Lq, int h, int d, double *out,
                          double *lse)
{
    for (int bb = 0; bb < b; ++bb)
        for (int hq = 0; hq < h; ++hq)
            for (int64_t r = 0; r < Lq; ++r) {
                const int64_t si = ((int64_t)bb * h + hq) * Lq + r;
                const int64_t oi = (((int64_t)bb * Lq + r) * h + hq) * d;
                const double lr = l[si];
                if (lr > 0.0) {
                    lse[si] = m[si] + log(lr);
                    for (int e = 0; e < d; ++e)
                        out[oi + e] = o[oi + e] / lr;
                } else {
                    lse[si] = -INFINITY;
                    for (int e = 0; e < d; ++e)
                        out[oi + e] = 0.0;
                }
            }
}

/* Merge of two partial results over disjoint key sets, [P2 "FlashAttention
 * Integration"]: O_new = O_old e^(m_old - m_new) + O_blk e^(m_blk - m_new).
 * Here each side is already normalised (O = numerator / l), so its reference
 * value is its own LSE and its normaliser is 1:
 *   m = max(lse_a, lse_b);  w_x = e^(lse_x - m)
 *   O = (w_a O_a + w_b O_b) / (w_a + w_b);   lse = m + ln(w_a + w_b).
 * A side with lse = -inf carries no keys; both -inf gives O = 0, lse = -inf.
 * o_* [b,Lq,h,d], lse_* [b,h,Lq].                                            */
ORC_API void orc_merge(const double *o_a, const double *lse_a,
                       const double *o_b, const double *lse_b, int b,
                       int64_t Lq, int h, int d, double *o, double *lse)
{
    for (int bb = 0; bb < b; ++bb)
        for (int hq = 0; hq < h; ++hq)
            for (int64_t r = 0; r < Lq; ++r) {
                const int64_t si = ((int64_t)bb * h + hq) * Lq + r;
                const int64_t oi = (((int64_t)bb * Lq + r) * h + hq) * d;
                const double a = lse_a[si], c = lse_b[si];
                const double mm = a > c ? a : c;
                if (mm == -INFINITY) {
                    lse[si] = -INFINITY;
                    for (int e = 0; e < d; ++e)
                        o[oi + e] = 0.0;
                    continue;
                }
                const double wa = exp(a - mm), wb = exp(c - mm);
                const double den = wa + wb;
                lse[si] = mm + log(den);
                for (int e = 0; e < d; ++e)
                    o[oi + e] = (wa * o_a[oi + e] + wb * o_b[oi + e]) / den;
            }
}
