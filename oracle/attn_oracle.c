/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64, two-pass CPU oracle for bottom-right-causal grouped-query
 * attention.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline leg call it; the product library never links it, and it shares no
 * code, header or table with the CUDA kernels.
 *
 * What it computes (restated from the pages, not copied):
 *   "Attention execution mapping: 现状、缺口与有界实验" (LuisaCompute), §1:
 *     the fixture is bottom-right-causal GQA; query head h reads KV head
 *     kh = h / (Hq / Hkv); a key k is legal for query row q iff
 *     k <= q + K - Q; one online-softmax program covers prefill and decode.
 *   Same page, §2 (phase graph): QK contracts over d, a mask, then
 *     max -> exp -> sum, then PV contracts over the key axis.
 *   "快速後端" (Laya fast backends), "數值校驗": sliding window, per-sequence
 *     (int32) lengths, empty sequences and finite padded output are covered.
 *
 * The online method (running max / sum / accumulator carried across KV
 * blocks) reaches, in exact arithmetic, the plain softmax definition below, so
 * the oracle is that definition written out -- no blocking, no online update:
 *
 *   for every sequence b, query head h, valid query row q < Qb:
 *     kh  = h / (Hq / Hkv)
 *     L   = { k : 0 <= k < Kb, k <= q + Kb - Qb,
 *                 and (window <= 0 or k >= q + Kb - Qb - window + 1) }
 *     if L is empty:   O[q,h,:] = +0,  LSE[q,h] = -inf
 *     else:  s_k = scale * sum_d Q[q,h,d] * K[k,kh,d]        (fp64)
 *            pass 1: m = max_{k in L} s_k
 *            pass 2: l = sum_{k in L} exp(s_k - m)
 *                    O[q,h,j] = sum_{k in L} exp(s_k - m) * V[k,kh,j] / l
 *            LSE[q,h] = m + log(l)                         (natural log)
 *   padded rows q >= Qb: O = +0, LSE = -inf.
 *
 * Readings where the pages are silent: a window w > 0 keeps the w most recent
 * keys including the diagonal one; rows with no legal key give +0 / -inf; the
 * LSE is in natural log.
 *
 * Two masks beyond the pages' bottom-right rule, selected by `mask` (the
 * library's extensions; the definition above is otherwise unchanged):
 *   mask 1, top-left causal: the diagonal is k = q (L = { k < Kb : k <= q },
 *           with the window counted back from that diagonal);
 *   mask 2, no mask: L = { k : 0 <= k < Kb } (no window).
 * mask 0 is the pages' bottom-right causal rule.
 *
 * Inputs are float32 arrays holding exactly the values the device sees
 * (bf16 / fp16 / fp32 values are all exact in float32); every product and sum
 * is taken in double.  Layouts:
 *   padded: q [B,Q,Hq,D]  k [B,K,Hkv,D]  v [B,K,Hkv,Dv]  o [B,Q,Hq,Dv]  lse [B,Q,Hq]
 *   packed: q [Tq,Hq,D]   k [Tk,Hkv,D]   v [Tk,Hkv,Dv]   o [Tq,Hq,Dv]   lse [Tq,Hq]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One (sequence, head, query-row) of the definition above.  qrow points at
 * Q[q,h,0]; kbase/vbase point at key row 0 of this sequence and KV head; the
 * key stride is the element distance between consecutive key rows. */
/* The legal keys of query row q as inclusive bounds [*lo, *hi]. */
static void legal_keys(int q, int Qb, int Kb, int window, int mask, long *lo, long *hi)
{
    *lo = 0;
    if (mask == 2) {                                   /* no mask: every key */
        *hi = (long)Kb - 1;
        return;
    }
    const long diag = mask == 1 ? (long)q : (long)q + Kb - Qb;   /* last legal key */
    *hi = diag;
    if (window > 0 && diag - window + 1 > *lo) *lo = diag - window + 1;
    if (*hi > (long)Kb - 1) *hi = (long)Kb - 1;
}

static void oracle_row(const float *qrow, const float *kbase, const float *vbase,
                       long kstride, long vstride, int D, int Dv, int q, int Qb,
                       int Kb, int window, int mask, double scale, double *s_scratch,
                       double *orow, double *lse_out)
{
    long lo, hi;                                       /* inclusive bounds */
    legal_keys(q, Qb, Kb, window, mask, &lo, &hi);
    for (int j = 0; j < Dv; ++j) orow[j] = 0.0;
    if (hi < lo) { *lse_out = -INFINITY; return; }

    /* scores of the legal keys, and pass 1: their maximum */
    double m = -INFINITY;
    for (long k = lo; k <= hi; ++k) {
        const float *krow = kbase + k * kstride;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += (double)qrow[d] * (double)krow[d];
        const double s = scale * acc;
        s_scratch[k - lo] = s;
        if (s > m) m = s;
    }
    /* pass 2: normaliser and weighted sum of V rows */
    double l = 0.0;
    for (long k = lo; k <= hi; ++k) {
        const double p = exp(s_scratch[k - lo] - m);
        l += p;
        const float *vrow = vbase + k * vstride;
        for (int j = 0; j < Dv; ++j) orow[j] += p * (double)vrow[j];
    }
    for (int j = 0; j < Dv; ++j) orow[j] /= l;
    *lse_out = m + log(l);
}

/* A per-sequence length outside [0, cap] is clamped into it (the padded
 * layout holds at most cap rows per sequence). */
static int clamp_len(int n, int cap)
{
    return n < 0 ? 0 : (n > cap ? cap : n);
}

static int check_dims(int B, int Hq, int Hkv, int D, int Dv)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Dv <= 0) return 1;
    if (Hq % Hkv != 0) return 1;
    return 0;
}

/* Padded layout.  seqlens_q / seqlens_k may be NULL (= all Q / all K). */
int oracle_attn_padded(const float *q, const float *k, const float *v, double *o,
                       double *lse, int B, int Hq, int Hkv, int Q, int K, int D,
                       int Dv, const int32_t *seqlens_q, const int32_t *seqlens_k,
                       int window, int mask, double scale, int nthreads)
{
    if (check_dims(B, Hq, Hkv, D, Dv) || Q < 0 || K < 0) return 1;
    if (mask < 0 || mask > 2 || (mask == 2 && window > 0)) return 1;
    const int G = Hq / Hkv;
    const long nrows = (long)B * Q * Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < nrows; ++r) {
            if (!s) continue;
            const int h = (int)(r % Hq);
            const int qi = (int)((r / Hq) % Q);
            const int b = (int)(r / ((long)Hq * Q));
            const int Qb = clamp_len(seqlens_q ? seqlens_q[b] : Q, Q);
            const int Kb = clamp_len(seqlens_k ? seqlens_k[b] : K, K);
            double *orow = o + r * Dv;
            if (qi >= Qb) {
                for (int j = 0; j < Dv; ++j) orow[j] = 0.0;
                lse[r] = -INFINITY;
                continue;
            }
            const int kh = h / G;
            oracle_row(q + r * D, k + ((long)b * K * Hkv + kh) * D,
                       v + ((long)b * K * Hkv + kh) * Dv, (long)Hkv * D,
                       (long)Hkv * Dv, D, Dv, qi, Qb, Kb, window, mask, scale, s, orow,
                       &lse[r]);
        }
        free(s);
    }
    return bad ? 3 : 0;
}

/* Packed (varlen) layout: sequence b owns query rows [cu_q[b], cu_q[b+1]) and
 * key rows [cu_k[b], cu_k[b+1]). */
int oracle_attn_packed(const float *q, const float *k, const float *v, double *o,
                       double *lse, int B, int Hq, int Hkv, int D, int Dv,
                       const int32_t *cu_q, const int32_t *cu_k, int window,
                       int mask, double scale, int nthreads)
{
    if (check_dims(B, Hq, Hkv, D, Dv) || !cu_q || !cu_k) return 1;
    if (mask < 0 || mask > 2 || (mask == 2 && window > 0)) return 1;
    if (cu_q[0] != 0 || cu_k[0] != 0) return 1;
    for (int b = 0; b < B; ++b)
        if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b]) return 1;
    const int G = Hq / Hkv;
    const long Tq = cu_q[B];
    long maxK = 1;
    for (int b = 0; b < B; ++b)
        if (cu_k[b + 1] - cu_k[b] > maxK) maxK = cu_k[b + 1] - cu_k[b];
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)maxK);
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < Tq * Hq; ++r) {
            if (!s) continue;
            const int h = (int)(r % Hq);
            const long t = r / Hq;
            int b = 0;
            while (b + 1 < B && cu_q[b + 1] <= t) ++b;
            const int Qb = cu_q[b + 1] - cu_q[b];
            const int Kb = cu_k[b + 1] - cu_k[b];
            const int qi = (int)(t - cu_q[b]);
            const int kh = h / G;
            oracle_row(q + r * D, k + ((long)cu_k[b] * Hkv + kh) * D,
                       v + ((long)cu_k[b] * Hkv + kh) * Dv, (long)Hkv * D,
                       (long)Hkv * Dv, D, Dv, qi, Qb, Kb, window, mask, scale, s,
                       o + r * Dv, &lse[r]);
        }
        free(s);
    }
    return bad ? 3 : 0;
}

/* Selected rows of the padded layout, for sampled checks at full size:
 * row i is (rb[i], rq[i], rh[i]); o_rows is [n, Dv], lse_rows [n]. */
int oracle_attn_padded_rows(const float *q, const float *k, const float *v,
                            int B, int Hq, int Hkv, int Q, int K, int D, int Dv,
                            const int32_t *seqlens_q, const int32_t *seqlens_k,
                            int window, int mask, double scale, const int32_t *rb,
                            const int32_t *rq, const int32_t *rh, long n,
                            double *o_rows, double *lse_rows, int nthreads)
{
    if (check_dims(B, Hq, Hkv, D, Dv) || Q < 0 || K < 0) return 1;
    if (mask < 0 || mask > 2 || (mask == 2 && window > 0)) return 1;
    for (long i = 0; i < n; ++i)
        if (rb[i] < 0 || rb[i] >= B || rq[i] < 0 || rq[i] >= Q || rh[i] < 0 ||
            rh[i] >= Hq)
            return 1;
    const int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!s) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long i = 0; i < n; ++i) {
            if (!s) continue;
            const int b = rb[i], qi = rq[i], h = rh[i];
            const int Qb = clamp_len(seqlens_q ? seqlens_q[b] : Q, Q);
            const int Kb = clamp_len(seqlens_k ? seqlens_k[b] : K, K);
            double *orow = o_rows + i * Dv;
            if (qi >= Qb) {
                for (int j = 0; j < Dv; ++j) orow[j] = 0.0;
                lse_rows[i] = -INFINITY;
                continue;
            }
            const long r = ((long)b * Q + qi) * Hq + h;
            const int kh = h / G;
            oracle_row(q + r * D, k + ((long)b * K * Hkv + kh) * D,
                       v + ((long)b * K * Hkv + kh) * Dv, (long)Hkv * D,
                       (long)Hkv * Dv, D, Dv, qi, Qb, Kb, window, mask, scale, s, orow,
                       &lse_rows[i]);
        }
        free(s);
    }
    return bad ? 3 : 0;
}

/* Gradients of the same attention (padded layout), for a loss whose gradient
 * with respect to O is dO.  The pages print no backward arithmetic (the FlyDSL
 * page, section on FMHA through AOTriton, only names its kernels); it is
 * the derivative of the definition above, written out per row (fp64):
 *   P[q,k]  = exp(s_k - LSE[q]) for k in L(q), 0 otherwise (s, L, LSE as above)
 *   Dq      = sum_j dO[q,j] * O[q,j]
 *   dP[q,k] = sum_j dO[q,j] * V[k,j]
 *   dS[q,k] = P[q,k] * (dP[q,k] - Dq)
 *   dQ[q]   = scale * sum_k dS[q,k] * K[k]
 *   dK[k]   = scale * sum over the rows q and the query heads h of KV head kh of dS[q,k] * Q[q]
 *   dV[k]   = the same sum of P[q,k] * dO[q]
 * O and LSE are recomputed here from the definition (nothing is taken from the
 * device).  Rows without a legal key and padded rows contribute nothing and
 * get dQ = 0; keys no row attends to get dK = dV = 0.
 * dq [B,Q,Hq,D], dk [B,K,Hkv,D], dv [B,K,Hkv,Dv] are written in full. */
int oracle_attn_bwd_padded(const float *q, const float *k, const float *v, const float *dout,
                           double *dq, double *dk, double *dv, int B, int Hq, int Hkv, int Q,
                           int K, int D, int Dv, const int32_t *seqlens_q,
                           const int32_t *seqlens_k, int window, int mask, double scale,
                           int nthreads)
{
    if (check_dims(B, Hq, Hkv, D, Dv) || Q < 0 || K < 0) return 1;
    if (mask < 0 || mask > 2 || (mask == 2 && window > 0)) return 1;
    const int G = Hq / Hkv;
    memset(dq, 0, sizeof(double) * (size_t)B * Q * Hq * D);
    memset(dk, 0, sizeof(double) * (size_t)B * K * Hkv * D);
    memset(dv, 0, sizeof(double) * (size_t)B * K * Hkv * Dv);
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
    /* one (sequence, KV head) per task: it owns its dK / dV rows */
#pragma omp parallel
    {
        const size_t kc = (size_t)(K > 0 ? K : 1);
        double *s = (double *)malloc(sizeof(double) * kc);
        double *orow = (double *)malloc(sizeof(double) * (size_t)Dv);
        if (!s || !orow) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long u = 0; u < (long)B * Hkv; ++u) {
            if (!s || !orow) continue;
            const int b = (int)(u / Hkv), kh = (int)(u % Hkv);
            const int Qb = clamp_len(seqlens_q ? seqlens_q[b] : Q, Q);
            const int Kb = clamp_len(seqlens_k ? seqlens_k[b] : K, K);
            const float *kb = k + ((long)b * K * Hkv + kh) * D;      /* key row stride Hkv*D */
            const float *vb = v + ((long)b * K * Hkv + kh) * Dv;
            double *dkb = dk + ((long)b * K * Hkv + kh) * D;
            double *dvb = dv + ((long)b * K * Hkv + kh) * Dv;
            for (int h = kh * G; h < (kh + 1) * G; ++h)
                for (int qi = 0; qi < Qb; ++qi) {
                    const long r = ((long)b * Q + qi) * Hq + h;
                    const float *qrow = q + r * D;
                    const float *dorow = dout + r * Dv;
                    double lse;
                    oracle_row(qrow, kb, vb, (long)Hkv * D, (long)Hkv * Dv, D, Dv, qi, Qb, Kb,
                               window, mask, scale, s, orow, &lse);
                    if (lse == -INFINITY) continue;
                    long lo, hi;
                    legal_keys(qi, Qb, Kb, window, mask, &lo, &hi);
                    double Dq = 0.0;
                    for (int j = 0; j < Dv; ++j) Dq += (double)dorow[j] * orow[j];
                    double *dqrow = dq + r * D;
                    for (long kk = lo; kk <= hi; ++kk) {
                        const float *krow = kb + kk * (long)Hkv * D;
                        const float *vrow = vb + kk * (long)Hkv * Dv;
                        double acc = 0.0;
                        for (int d = 0; d < D; ++d) acc += (double)qrow[d] * (double)krow[d];
                        const double p = exp(scale * acc - lse);
                        double dp = 0.0;
                        for (int j = 0; j < Dv; ++j) dp += (double)dorow[j] * (double)vrow[j];
                        const double ds = p * (dp - Dq);
                        for (int d = 0; d < D; ++d) {
                            dqrow[d] += scale * ds * (double)krow[d];
                            dkb[kk * (long)Hkv * D + d] += scale * ds * (double)qrow[d];
                        }
                        for (int j = 0; j < Dv; ++j)
                            dvb[kk * (long)Hkv * Dv + j] += p * (double)dorow[j];
                    }
                }
        }
        free(s);
        free(orow);
    }
    return bad ? 3 : 0;
}

/* The same gradients for parts of a large problem (padded layout), each
 * output row computed on its own with the arithmetic of
 * oracle_attn_bwd_padded (O, LSE and Dq of a row are recomputed from the
 * definition wherever the row is needed):
 *   rows [nrows][3] = (b, q, h):  dq_out [nrows][D] (zeros for a padded row
 *                                 or a row without a legal key);
 *   keys [k0, k1) of sequence b, KV head kh:  dk_out [k1-k0][D], dv_out
 *                                 [k1-k0][Dv], summed over every row of every
 *                                 query head of the group that attends to them.
 * Either part may be empty (nrows = 0, or k1 <= k0). */
int oracle_attn_bwd_sampled(const float *q, const float *k, const float *v, const float *dout,
                            int B, int Hq, int Hkv, int Q, int K, int D, int Dv,
                            const int32_t *seqlens_q, const int32_t *seqlens_k, int window,
                            int mask, double scale, const int32_t *rows, long nrows,
                            double *dq_out, int kb, int kkh, int k0, int k1, double *dk_out,
                            double *dv_out, int nthreads)
{
    if (check_dims(B, Hq, Hkv, D, Dv) || Q < 0 || K < 0) return 1;
    if (mask < 0 || mask > 2 || (mask == 2 && window > 0)) return 1;
    const int G = Hq / Hkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
    if (nrows > 0) memset(dq_out, 0, sizeof(double) * (size_t)nrows * D);
    if (k1 > k0) {
        if (kb < 0 || kb >= B || kkh < 0 || kkh >= Hkv || k0 < 0 || k1 > K) return 1;
        memset(dk_out, 0, sizeof(double) * (size_t)(k1 - k0) * D);
        memset(dv_out, 0, sizeof(double) * (size_t)(k1 - k0) * Dv);
    }
    /* dQ rows */
#pragma omp parallel
    {
        const size_t kc = (size_t)(K > 0 ? K : 1);
        double *sc = (double *)malloc(sizeof(double) * kc);
        double *orow = (double *)malloc(sizeof(double) * (size_t)Dv);
        if (!sc || !orow) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 8)
        for (long i = 0; i < nrows; ++i) {
            if (!sc || !orow) continue;
            const int b = rows[3 * i], qi = rows[3 * i + 1], h = rows[3 * i + 2];
            if (b < 0 || b >= B || qi < 0 || qi >= Q || h < 0 || h >= Hq) {
#pragma omp atomic write
                bad = 2;
                continue;
            }
            const int kh = h / G;
            const int Qb = clamp_len(seqlens_q ? seqlens_q[b] : Q, Q);
            const int Kb = clamp_len(seqlens_k ? seqlens_k[b] : K, K);
            if (qi >= Qb) continue;
            const long r = ((long)b * Q + qi) * Hq + h;
            const float *qrow = q + r * D, *dorow = dout + r * Dv;
            const float *kbp = k + ((long)b * K * Hkv + kh) * D;
            const float *vbp = v + ((long)b * K * Hkv + kh) * Dv;
            double lse;
            oracle_row(qrow, kbp, vbp, (long)Hkv * D, (long)Hkv * Dv, D, Dv, qi, Qb, Kb, window,
                       mask, scale, sc, orow, &lse);
            if (lse == -INFINITY) continue;
            long lo, hi;
            legal_keys(qi, Qb, Kb, window, mask, &lo, &hi);
            double Dq = 0.0;
            for (int j = 0; j < Dv; ++j) Dq += (double)dorow[j] * orow[j];
            double *dqrow = dq_out + i * D;
            for (long kk = lo; kk <= hi; ++kk) {
                const float *krow = kbp + kk * (long)Hkv * D;
                const float *vrow = vbp + kk * (long)Hkv * Dv;
                double acc = 0.0, dp = 0.0;
                for (int d = 0; d < D; ++d) acc += (double)qrow[d] * (double)krow[d];
                for (int j = 0; j < Dv; ++j) dp += (double)dorow[j] * (double)vrow[j];
                const double ds = exp(scale * acc - lse) * (dp - Dq);
                for (int d = 0; d < D; ++d) dqrow[d] += scale * ds * (double)krow[d];
            }
        }
        free(sc);
        free(orow);
    }
    if (bad || k1 <= k0) return bad ? 3 : 0;
    /* dK / dV of keys [k0, k1): one task per (head of the group, row) */
    const int Qb = clamp_len(seqlens_q ? seqlens_q[kb] : Q, Q);
    const int Kb = clamp_len(seqlens_k ? seqlens_k[kb] : K, K);
    const long ntask = (long)G * Qb;
    const long nk = k1 - k0;
#pragma omp parallel
    {
        const size_t kc = (size_t)(K > 0 ? K : 1);
        double *sc = (double *)malloc(sizeof(double) * kc);
        double *orow = (double *)malloc(sizeof(double) * (size_t)Dv);
        double *gk = (double *)calloc((size_t)nk * D, sizeof(double));
        double *gv = (double *)calloc((size_t)nk * Dv, sizeof(double));
        if (!sc || !orow || !gk || !gv) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < ntask; ++t) {
            if (!sc || !orow || !gk || !gv) continue;
            const int h = kkh * G + (int)(t / Qb), qi = (int)(t % Qb);
            long lo, hi;
            legal_keys(qi, Qb, Kb, window, mask, &lo, &hi);
            if (hi < lo || hi < k0 || lo >= k1) continue;
            const long r = ((long)kb * Q + qi) * Hq + h;
            const float *qrow = q + r * D, *dorow = dout + r * Dv;
            const float *kbp = k + ((long)kb * K * Hkv + kkh) * D;
            const float *vbp = v + ((long)kb * K * Hkv + kkh) * Dv;
            double lse;
            oracle_row(qrow, kbp, vbp, (long)Hkv * D, (long)Hkv * Dv, D, Dv, qi, Qb, Kb, window,
                       mask, scale, sc, orow, &lse);
            double Dq = 0.0;
            for (int j = 0; j < Dv; ++j) Dq += (double)dorow[j] * orow[j];
            const long a = lo > k0 ? lo : k0, e = hi < k1 - 1 ? hi : k1 - 1;
            for (long kk = a; kk <= e; ++kk) {
                const float *krow = kbp + kk * (long)Hkv * D;
                const float *vrow = vbp + kk * (long)Hkv * Dv;
                double acc = 0.0, dp = 0.0;
                for (int d = 0; d < D; ++d) acc += (double)qrow[d] * (double)krow[d];
                for (int j = 0; j < Dv; ++j) dp += (double)dorow[j] * (double)vrow[j];
                const double p = exp(scale * acc - lse);
                const double ds = p * (dp - Dq);
                for (int d = 0; d < D; ++d) gk[(kk - k0) * D + d] += scale * ds * (double)qrow[d];
                for (int j = 0; j < Dv; ++j) gv[(kk - k0) * Dv + j] += p * (double)dorow[j];
            }
        }
#pragma omp critical
        {
            if (gk && gv) {
                for (long x = 0; x < nk * D; ++x) dk_out[x] += gk[x];
                for (long x = 0; x < nk * Dv; ++x) dv_out[x] += gv[x];
            }
        }
        free(sc);
        free(orow);
        free(gk);
        free(gv);
    }
    return bad ? 3 : 0;
}

/*
 * An arbitrary boolean mask on top of the masks above -- an extension of this
 * library ("Attention execution mapping" (LuisaCompute), section 7, names
 * arbitrary masks as a semantic extension that needs an independent oracle).
 * allow[((b * Hm + hm) * Q + q) * K + k] != 0 lets query row q of sequence b
 * attend to key k, for query head h with hm = h when Hm == Hq and hm = 0 when
 * Hm == 1 (one mask shared by every head).  The legal set is the set of the
 * chosen mask mode intersected with it:
 *     L = { k in [lo, hi] of legal_keys(q) : allow[b, hm, q, k] != 0 }
 * and the definition is otherwise the one at the top of this file: the keys of
 * L are listed explicitly, pass 1 takes their maximum score, pass 2 the
 * normaliser and the weighted sum of V rows; an empty L gives +0 / -inf.
 */
static void oracle_row_allow(const float *qrow, const float *kbase, const float *vbase,
                             long kstride, long vstride, int D, int Dv, int q, int Qb,
                             int Kb, int window, int mask, const uint8_t *allow_row,
                             double scale, long *keys, double *s_scratch, double *orow,
                             double *lse_out)
{
    long lo, hi;                                       /* inclusive bounds */
    legal_keys(q, Qb, Kb, window, mask, &lo, &hi);
    long n = 0;
    for (long k = lo; k <= hi; ++k)
        if (allow_row[k] != 0) keys[n++] = k;
    for (int j = 0; j < Dv; ++j) orow[j] = 0.0;
    if (n == 0) { *lse_out = -INFINITY; return; }
    double m = -INFINITY;
    for (long i = 0; i < n; ++i) {
        const float *krow = kbase + keys[i] * kstride;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += (double)qrow[d] * (double)krow[d];
        s_scratch[i] = scale * acc;
        if (s_scratch[i] > m) m = s_scratch[i];
    }
    double l = 0.0;
    for (long i = 0; i < n; ++i) {
        const double p = exp(s_scratch[i] - m);
        l += p;
        const float *vrow = vbase + keys[i] * vstride;
        for (int j = 0; j < Dv; ++j) orow[j] += p * (double)vrow[j];
    }
    for (int j = 0; j < Dv; ++j) orow[j] /= l;
    *lse_out = m + log(l);
}

/* Padded layout with the boolean mask `allow` [B, Hm, Q, K] (Hm = 1 or Hq);
 * other arguments as oracle_attn_padded. */
int oracle_attn_padded_allow(const float *q, const float *k, const float *v, double *o,
                             double *lse, int B, int Hq, int Hkv, int Q, int K, int D, int Dv,
                             const int32_t *seqlens_q, const int32_t *seqlens_k,
                             const uint8_t *allow, int Hm, int window, int mask, double scale,
                             int nthreads)
{
    if (check_dims(B, Hq, Hkv, D, Dv) || Q < 0 || K < 0 || !allow) return 1;
    if (mask < 0 || mask > 2 || (mask == 2 && window > 0)) return 1;
    if (Hm != 1 && Hm != Hq) return 1;
    const int G = Hq / Hkv;
    const long nrows = (long)B * Q * Hq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int bad = 0;
#pragma omp parallel
    {
        const size_t kn = (size_t)(K > 0 ? K : 1);
        double *s = (double *)malloc(sizeof(double) * kn);
        long *keys = (long *)malloc(sizeof(long) * kn);
        if (!s || !keys) {
#pragma omp atomic write
            bad = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < nrows; ++r) {
            if (!s || !keys) continue;
            const int h = (int)(r % Hq);
            const int qi = (int)((r / Hq) % Q);
            const int b = (int)(r / ((long)Hq * Q));
            const int Qb = clamp_len(seqlens_q ? seqlens_q[b] : Q, Q);
            const int Kb = clamp_len(seqlens_k ? seqlens_k[b] : K, K);
            double *orow = o + r * Dv;
            if (qi >= Qb) {
                for (int j = 0; j < Dv; ++j) orow[j] = 0.0;
                lse[r] = -INFINITY;
                continue;
            }
            const int kh = h / G;
            const int hm = Hm == 1 ? 0 : h;
            const uint8_t *arow = allow + (((long)b * Hm + hm) * Q + qi) * (long)K;
            oracle_row_allow(q + r * D, k + ((long)b * K * Hkv + kh) * D,
                             v + ((long)b * K * Hkv + kh) * Dv, (long)Hkv * D, (long)Hkv * Dv,
                             D, Dv, qi, Qb, Kb, window, mask, arow, scale, keys, s, orow,
                             &lse[r]);
        }
        free(s);
        free(keys);
    }
    return bad ? 3 : 0;
}

/* Number of legal (query, key) pairs of one sequence, per head: the unit the
 * throughput figures count (FLOP = pairs * (2D + 2Dv) per head). */
long long oracle_legal_pairs(int Qb, int Kb, int window, int mask)
{
    long long n = 0;
    for (int q = 0; q < Qb; ++q) {
        long lo, hi;
        legal_keys(q, Qb, Kb, window, mask, &lo, &hi);
        if (hi >= lo) n += hi - lo + 1;
    }
    return n;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
