/*
 * Exact softmax attention in fp64 on the CPU: the ORACLE.
 *
 * This file is test infrastructure. Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load it. The product path (the
 * CUDA library) shares no code with it and never calls it.
 *
 * What it computes (FFPA docs, "CuTe-DSL Backend" page, sections "Hard
 * constraints" and "Varlen (packed THD) API"; "Backends Overview" page,
 * section "Automatic SDPA fallback", for the SDPA-aligned result):
 *
 *   s_ij   = scale * sum_d q[i,d] k[j,d]          over legal keys j only
 *   legal  : j < Lk, and when causal j <= i + (Lk - Lq)   (bottom-right / tail-
 *            aligned mask, applied per sequence for varlen)
 *   LSE_i  = m_i + ln sum_j exp(s_ij - m_i),  m_i = max_j s_ij   (natural log)
 *   P_ij   = exp(s_ij - LSE_i)
 *   O_i    = sum_j P_ij v_j
 *   rows with no legal key: O_i = 0, LSE_i = -inf, and exactly zero gradient.
 *
 * Backward, for the loss L = sum(dO * O):
 *   delta_i = sum_d dO[i,d] O[i,d]
 *   dP_ij   = dO_i . v_j
 *   dS_ij   = P_ij (dP_ij - delta_i)
 *   dQ_i    = scale sum_j dS_ij k_j
 *   dK_j    = scale sum_{query heads h of j's group} sum_i dS_ij q_i
 *   dV_j    = sum_{h in group} sum_i P_ij dO_i
 *
 * GQA/MQA: query head h reads kv head h / (Hq / Hkv) (a zero-stride broadcast
 * of each kv head over a consecutive group of query heads).
 *
 * Plain two-pass per query row, no tiling, no online softmax. OpenMP spreads
 * independent rows (and, for dK/dV, independent key rows) over host cores.
 */
#include <math.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One attention problem for a single (sequence, query head): pointers to its
 * first row and the distance in elements between consecutive rows. */
typedef struct {
    const double *q, *k, *v, *dout;
    double *o, *dq;
    double *lse, *delta; /* stride 1 along rows */
    long q_rs, kv_rs;
    long lq, lk;
} head_view;

static int is_legal(long i, long j, long lq, long lk, int causal)
{
    if (j < 0 || j >= lk) return 0;
    if (!causal) return 1;
    return j <= i + (lk - lq);
}

static double dot(const double* a, const double* b, long n)
{
    double acc = 0.0;
    for (long d = 0; d < n; ++d) acc += a[d] * b[d];
    return acc;
}

/* Forward for row i of one head: writes O_i to oi, LSE_i to *lse_i and, if
 * delta_i is given, delta_i = dO_i . O_i. Scratch s holds lk doubles. */
static void fwd_row(const head_view* hv, long i, long D, int causal, double scale, double* s,
                    double* oi, double* lse_i, double* delta_i)
{
    const double* qi = hv->q + i * hv->q_rs;
    double m = -INFINITY;
    long n_legal = 0;
    for (long j = 0; j < hv->lk; ++j) {
        if (!is_legal(i, j, hv->lq, hv->lk, causal)) continue;
        s[j] = scale * dot(qi, hv->k + j * hv->kv_rs, D);
        if (s[j] > m) m = s[j];
        ++n_legal;
    }
    if (n_legal == 0) {
        for (long d = 0; d < D; ++d) oi[d] = 0.0;
        *lse_i = -INFINITY;
        if (delta_i) *delta_i = 0.0;
        return;
    }
    double l = 0.0;
    for (long j = 0; j < hv->lk; ++j)
        if (is_legal(i, j, hv->lq, hv->lk, causal)) l += exp(s[j] - m);
    const double lse = m + log(l);
    *lse_i = lse;
    for (long d = 0; d < D; ++d) oi[d] = 0.0;
    for (long j = 0; j < hv->lk; ++j) {
        if (!is_legal(i, j, hv->lq, hv->lk, causal)) continue;
        const double p = exp(s[j] - lse);
        const double* vj = hv->v + j * hv->kv_rs;
        for (long d = 0; d < D; ++d) oi[d] += p * vj[d];
    }
    if (delta_i) *delta_i = dot(hv->dout + i * hv->q_rs, oi, D);
}

/* dQ for row i; needs LSE_i and delta_i from fwd_row. */
static void dq_row(const head_view* hv, long i, long D, int causal, double scale)
{
    double* dqi = hv->dq + i * hv->q_rs;
    for (long d = 0; d < D; ++d) dqi[d] = 0.0;
    if (isinf(hv->lse[i])) return; /* empty row: exactly zero */
    const double* qi = hv->q + i * hv->q_rs;
    const double* doi = hv->dout + i * hv->q_rs;
    for (long j = 0; j < hv->lk; ++j) {
        if (!is_legal(i, j, hv->lq, hv->lk, causal)) continue;
        const double* kj = hv->k + j * hv->kv_rs;
        const double p = exp(scale * dot(qi, kj, D) - hv->lse[i]);
        const double dp = dot(doi, hv->v + j * hv->kv_rs, D);
        const double ds = p * (dp - hv->delta[i]);
        for (long d = 0; d < D; ++d) dqi[d] += scale * ds * kj[d];
    }
}

/* Adds the contribution of one query head to dK_j and dV_j (key row j). */
static void dkdv_row_accumulate(const head_view* hv, long j, long D, int causal, double scale,
                                double* dkj, double* dvj)
{
    const double* kj = hv->k + j * hv->kv_rs;
    const double* vj = hv->v + j * hv->kv_rs;
    for (long i = 0; i < hv->lq; ++i) {
        if (!is_legal(i, j, hv->lq, hv->lk, causal)) continue;
        if (isinf(hv->lse[i])) continue;
        const double* qi = hv->q + i * hv->q_rs;
        const double* doi = hv->dout + i * hv->q_rs;
        const double p = exp(scale * dot(qi, kj, D) - hv->lse[i]);
        const double dp = dot(doi, vj, D);
        const double ds = p * (dp - hv->delta[i]);
        for (long d = 0; d < D; ++d) {
            dvj[d] += p * doi[d];
            dkj[d] += scale * ds * qi[d];
        }
    }
}

/* ---- layouts ------------------------------------------------------------
 * dense : q,o,dO,dq [B,Hq,Nq,D]; k,v,dk,dv [B,Hkv,Nkv,D]; lse [B,Hq,Nq]
 * varlen: q,o,dO,dq [Tq,Hq,D];   k,v,dk,dv [Tk,Hkv,D];    lse [Hq,Tq]
 * A "problem" below is a (sequence b, query head h) pair. */
typedef struct {
    int varlen;
    long B, Hq, Hkv, D;
    long Nq, Nkv;          /* dense */
    const int *cu_q, *cu_k; /* varlen, [B+1] */
    long total_q;
} layout;

static head_view make_view(const layout* L, long b, long h,
                           const double* q, const double* k, const double* v, const double* dout,
                           double* o, double* dq, double* lse, double* delta)
{
    head_view hv;
    const long g = L->Hq / L->Hkv;
    const long hk = h / g;
    long q_off, kv_off, lse_off;
    if (!L->varlen) {
        hv.lq = L->Nq;
        hv.lk = L->Nkv;
        hv.q_rs = L->D;
        hv.kv_rs = L->D;
        q_off = ((b * L->Hq + h) * L->Nq) * L->D;
        kv_off = ((b * L->Hkv + hk) * L->Nkv) * L->D;
        lse_off = (b * L->Hq + h) * L->Nq;
    } else {
        const long q0 = L->cu_q[b], k0 = L->cu_k[b];
        hv.lq = L->cu_q[b + 1] - q0;
        hv.lk = L->cu_k[b + 1] - k0;
        hv.q_rs = L->Hq * L->D;
        hv.kv_rs = L->Hkv * L->D;
        q_off = q0 * L->Hq * L->D + h * L->D;
        kv_off = k0 * L->Hkv * L->D + hk * L->D;
        lse_off = h * L->total_q + q0;
    }
    hv.q = q + q_off;
    hv.k = k + kv_off;
    hv.v = v + kv_off;
    hv.dout = dout ? dout + q_off : NULL;
    hv.o = o + q_off;
    hv.dq = dq ? dq + q_off : NULL;
    hv.lse = lse + lse_off;
    hv.delta = delta ? delta + lse_off : NULL;
    return hv;
}

static long seq_lq(const layout* L, long b) { return L->varlen ? L->cu_q[b + 1] - L->cu_q[b] : L->Nq; }
static long seq_lk(const layout* L, long b) { return L->varlen ? L->cu_k[b + 1] - L->cu_k[b] : L->Nkv; }

static void run_fwd(const layout* L, const double* q, const double* k, const double* v,
                    const double* dout, double* o, double* lse, double* delta,
                    int causal, double scale)
{
    long max_lk = 1;
    for (long b = 0; b < L->B; ++b) if (seq_lk(L, b) > max_lk) max_lk = seq_lk(L, b);
    for (long b = 0; b < L->B; ++b) {
        const long lq = seq_lq(L, b);
        const long rows = L->Hq * lq;
#pragma omp parallel
        {
            double* s = (double*)malloc((size_t)max_lk * sizeof(double));
#pragma omp for schedule(dynamic, 8)
            for (long r = 0; r < rows; ++r) {
                const long h = r / lq, i = r % lq;
                head_view hv = make_view(L, b, h, q, k, v, dout, o, NULL, lse, delta);
                fwd_row(&hv, i, L->D, causal, scale, s, hv.o + i * hv.q_rs, hv.lse + i,
                        hv.delta ? hv.delta + i : NULL);
            }
            free(s);
        }
    }
}

static void run_bwd(const layout* L, const double* q, const double* k, const double* v,
                    const double* dout, double* dq, double* dk, double* dv,
                    int causal, double scale)
{
    /* pass 1: O, LSE, delta per row (own forward; O is scratch) */
    size_t q_elems, lse_elems;
    if (!L->varlen) {
        q_elems = (size_t)(L->B * L->Hq * L->Nq * L->D);
        lse_elems = (size_t)(L->B * L->Hq * L->Nq);
    } else {
        q_elems = (size_t)(L->total_q * L->Hq * L->D);
        lse_elems = (size_t)(L->Hq * L->total_q);
    }
    double* o = (double*)calloc(q_elems ? q_elems : 1, sizeof(double));
    double* lse = (double*)calloc(lse_elems ? lse_elems : 1, sizeof(double));
    double* delta = (double*)calloc(lse_elems ? lse_elems : 1, sizeof(double));
    run_fwd(L, q, k, v, dout, o, lse, delta, causal, scale);

    /* pass 2: dQ per query row */
    for (long b = 0; b < L->B; ++b) {
        const long lq = seq_lq(L, b);
        const long rows = L->Hq * lq;
#pragma omp parallel for schedule(dynamic, 8)
        for (long r = 0; r < rows; ++r) {
            const long h = r / lq, i = r % lq;
            head_view hv = make_view(L, b, h, q, k, v, dout, o, dq, lse, delta);
            dq_row(&hv, i, L->D, causal, scale);
        }
    }

    /* pass 3: dK, dV per key row, summed over the query heads of the group */
    const long g = L->Hq / L->Hkv;
    for (long b = 0; b < L->B; ++b) {
        const long lk = seq_lk(L, b);
        const long rows = L->Hkv * lk;
#pragma omp parallel for schedule(dynamic, 8)
        for (long r = 0; r < rows; ++r) {
            const long hk = r / lk, j = r % lk;
            head_view first = make_view(L, b, hk * g, q, k, v, dout, o, dq, lse, delta);
            /* dk/dv share k's layout: offset of row j of this kv head */
            const long off = (first.k - k) + j * first.kv_rs;
            double* dkj = dk + off;
            double* dvj = dv + off;
            for (long d = 0; d < L->D; ++d) { dkj[d] = 0.0; dvj[d] = 0.0; }
            for (long h = hk * g; h < (hk + 1) * g; ++h) {
                head_view hv = make_view(L, b, h, q, k, v, dout, o, dq, lse, delta);
                dkdv_row_accumulate(&hv, j, L->D, causal, scale, dkj, dvj);
            }
        }
    }
    free(o);
    free(lse);
    free(delta);
}

/* ---- exported entry points (fp64, host memory, contiguous) --------------- */

int ffpa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void ffpa_oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

void ffpa_oracle_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                     long B, long Hq, long Hkv, long Nq, long Nkv, long D, int causal, double scale)
{
    layout L = {0, B, Hq, Hkv, D, Nq, Nkv, NULL, NULL, 0};
    run_fwd(&L, q, k, v, NULL, o, lse, NULL, causal, scale);
}

void ffpa_oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
                     double* dq, double* dk, double* dv,
                     long B, long Hq, long Hkv, long Nq, long Nkv, long D, int causal, double scale)
{
    layout L = {0, B, Hq, Hkv, D, Nq, Nkv, NULL, NULL, 0};
    run_bwd(&L, q, k, v, dout, dq, dk, dv, causal, scale);
}

void ffpa_oracle_varlen_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                            const int* cu_q, const int* cu_k, long batch, long total_q,
                            long Hq, long Hkv, long D, int causal, double scale)
{
    layout L = {1, batch, Hq, Hkv, D, 0, 0, cu_q, cu_k, total_q};
    run_fwd(&L, q, k, v, NULL, o, lse, NULL, causal, scale);
}

void ffpa_oracle_varlen_bwd(const double* q, const double* k, const double* v, const double* dout,
                            double* dq, double* dk, double* dv,
                            const int* cu_q, const int* cu_k, long batch, long total_q,
                            long Hq, long Hkv, long D, int causal, double scale)
{
    layout L = {1, batch, Hq, Hkv, D, 0, 0, cu_q, cu_k, total_q};
    run_bwd(&L, q, k, v, dout, dq, dk, dv, causal, scale);
}

/* Forward for a subset of query rows of one dense head (rows[0..n_rows)),
 * used to time or check a bounded sample of a large problem. o is [n_rows, D],
 * lse is [n_rows]. q is [Nq, D] of that head, k and v are [Nkv, D]. */
void ffpa_oracle_fwd_rows(const double* q, const double* k, const double* v,
                          const long* rows, long n_rows, double* o, double* lse,
                          long Nq, long Nkv, long D, int causal, double scale)
{
#pragma omp parallel
    {
        double* s = (double*)malloc((size_t)(Nkv > 0 ? Nkv : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < n_rows; ++r) {
            head_view hv;
            hv.q = q; hv.k = k; hv.v = v; hv.dout = NULL;
            hv.q_rs = D; hv.kv_rs = D; hv.lq = Nq; hv.lk = Nkv;
            hv.o = NULL; hv.dq = NULL; hv.lse = NULL; hv.delta = NULL;
            fwd_row(&hv, rows[r], D, causal, scale, s, o + r * D, lse + r, NULL);
        }
        free(s);
    }
}
