/*
 * attn_oracle.c -- fp64 CPU oracle for scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously-correct
 * definition that the CUDA path is checked against.  Only the test suite,
 * the package's smoke check and the benchmark's CPU-baseline leg may load
 * it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the definition, not the tiled method):
 *   The tiled method of "noflash-attention" (ai-navigate-news forum post,
 *   section "The DIY approach") loops over query chunks and key chunks with
 *   an online softmax and says it is the same math as forming the full score
 *   matrix.  So the oracle is that plain math, one query row at a time:
 *
 *     for every (b, h, i):  g = h / G            (G = Hq / Hkv, contiguous groups)
 *       s_j   = scale * sum_d q[b,h,i,d] * k[b,g,j,d]   for each allowed key j
 *       m     = max_j s_j
 *       l     = sum_j exp(s_j - m)
 *       o[d]  = sum_j exp(s_j - m) * v[b,g,j,d] / l
 *       lse   = m + log(l)                        (natural log of sum_j exp(s_j))
 *
 *   "Allowed" is every key, or with the causal mask the keys j <= i
 *   (top-left alignment, the is_causal convention of the SDPA call the forum
 *   post patches).  The forward also takes causal = 2, bottom-right
 *   alignment: the Nq queries are the LAST Nq positions of a sequence whose
 *   first Nk positions are the keys, so query i sees keys j <= i + (Nk - Nq)
 *   (the KV-cache decode of the post's LLM-inference table; Nq <= Nk).
 *
 *   Optional attention bias (the attn_mask argument of the SDPA call the
 *   post patches): b[b,h,i,j] is added to s_j before the softmax (natural-log
 *   units; -inf removes key j; a boolean mask is b = 0 / -inf).  A row whose
 *   every key is removed has no softmax: the reading used here is O = 0 and
 *   lse = -inf (the same as a row with no allowed key).  The default scale 1/sqrt(D) is the one the ai-manual.ru
 *   page's chunked snippet divides by (section "3 Samopisnyi memory-efficient
 *   attention"); the caller passes it explicitly.  No flush-to-zero and no
 *   epsilon: this is the exact result the tiled method approximates.
 *
 *   Backward (the autograd tier of the forum post, section "Other areas where
 *   this could be useful"), from the same definition, per row i:
 *       P_ij  = exp(s_ij - lse_i)
 *       dP_ij = sum_d dout[i,d] * v[j,d]
 *       Delta_i = sum_j P_ij * dP_ij
 *       dS_ij = P_ij * (dP_ij - Delta_i)
 *       dq[i,:] = scale * sum_j dS_ij * k[j,:]
 *       dk[j,:] += scale * dS_ij * q[i,:]      (summed over the G heads of a group)
 *       dv[j,:] += P_ij * dout[i,:]             (summed over the G heads of a group)
 *
 * Layout: q, out, dout, dq: [B, Hq, Nq, D]; k, v, dk, dv: [B, Hkv, Nk, D];
 * lse: [B, Hq, Nq]; all row-major, fp64.
 *
 * Return value of every entry point: 0 on success, -1 on a bad argument,
 * -2 when memory for the per-thread score row could not be obtained.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Number of keys that query position i may attend to. */
static int64_t allowed_keys(int64_t i, int64_t Nk, int causal)
{
    if (!causal) return Nk;
    return (i + 1 < Nk) ? (i + 1) : Nk;
}

/* One query row of the forward definition.  s: scratch of Nk doubles.
 * bias_row: the row's additive bias over the keys, or NULL. */
static void fwd_one_row(const double *q_row, const double *k_head, const double *v_head,
                        const double *bias_row, int64_t nkeys, int64_t D, double scale,
                        double *s, double *o_row, double *lse_out)
{
    double m = -INFINITY;
    for (int64_t j = 0; j < nkeys; ++j) {
        const double *k_row = k_head + j * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += q_row[d] * k_row[d];
        s[j] = scale * dot;
        if (bias_row) s[j] += bias_row[j];
        if (s[j] > m) m = s[j];
    }
    if (m == -INFINITY) {   /* every key removed: O = 0, lse = -inf */
        for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
        *lse_out = -INFINITY;
        return;
    }
    double l = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
    for (int64_t j = 0; j < nkeys; ++j) {
        const double *v_row = v_head + j * D;
        const double w = s[j] / l;
        for (int64_t d = 0; d < D; ++d) o_row[d] += w * v_row[d];
    }
    *lse_out = m + log(l);
}

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int64_t Hq, Hkv, Nq, Nk, D;
    double scale;
    int causal;
    const double *bias;    /* additive bias, or NULL */
    int64_t bsb, bsh, bsq; /* its element strides over batch, query head, query (0: broadcast) */
    const int64_t *rows;   /* flattened row ids (b*Hq + h)*Nq + i, or NULL for all */
    int64_t row_begin, row_end; /* this thread's slice of the row list */
    int status;
} fwd_job_t;

static void *fwd_worker(void *arg)
{
    fwd_job_t *jb = (fwd_job_t *)arg;
    double *s = (double *)malloc((size_t)(jb->Nk > 0 ? jb->Nk : 1) * sizeof(double));
    if (!s) { jb->status = -2; return NULL; }
    const int64_t G = jb->Hq / jb->Hkv;
    for (int64_t t = jb->row_begin; t < jb->row_end; ++t) {
        const int64_t r = jb->rows ? jb->rows[t] : t;
        const int64_t i = r % jb->Nq;
        const int64_t bh = r / jb->Nq;          /* b*Hq + h */
        const int64_t b = bh / jb->Hq, h = bh % jb->Hq;
        const int64_t g = h / G;
        const double *q_row = jb->q + r * jb->D;
        const double *k_head = jb->k + (b * jb->Hkv + g) * jb->Nk * jb->D;
        const double *v_head = jb->v + (b * jb->Hkv + g) * jb->Nk * jb->D;
        /* bottom-right: query i sits at sequence position i + (Nk - Nq) */
        const int64_t seq_pos = (jb->causal == 2) ? i + (jb->Nk - jb->Nq) : i;
        const double *bias_row = jb->bias ? jb->bias + b * jb->bsb + h * jb->bsh + i * jb->bsq : NULL;
        fwd_one_row(q_row, k_head, v_head, bias_row, allowed_keys(seq_pos, jb->Nk, jb->causal),
                    jb->D, jb->scale, s, jb->o + t * jb->D, jb->lse + t);
    }
    free(s);
    jb->status = 0;
    return NULL;
}

static int check_shape(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    return 0;
}

/*
 * Forward over a list of rows.  rows[t] = (b*Hq + h)*Nq + i.  Results are
 * written compactly: o[t*D + d], lse[t].  rows == NULL means every row in
 * order, so o and lse then have the full [B,Hq,Nq,(D)] layout.
 */
int oracle_attn_fwd_rows_bias(const double *q, const double *k, const double *v,
                              int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                              double scale, int causal,
                              const double *bias, int64_t bsb, int64_t bsh, int64_t bsq,
                              const int64_t *rows, int64_t n_rows,
                              double *o, double *lse, int nthreads)
{
    if (bias && (bsb < 0 || bsh < 0 || bsq < 0)) return -1;
    if (check_shape(B, Hq, Hkv, Nq, Nk, D)) return -1;
    if (!q || !k || !v || !o || !lse) return -1;
    if (causal < 0 || causal > 2 || (causal == 2 && Nq > Nk)) return -1;
    const int64_t total = rows ? n_rows : B * Hq * Nq;
    if (rows) {
        for (int64_t t = 0; t < n_rows; ++t)
            if (rows[t] < 0 || rows[t] >= B * Hq * Nq) return -1;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)(total > 0 ? total : 1);

    fwd_job_t *jobs = (fwd_job_t *)calloc((size_t)nthreads, sizeof(fwd_job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -2; }
    for (int t = 0; t < nthreads; ++t) {
        fwd_job_t *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->o = o; jb->lse = lse;
        jb->Hq = Hq; jb->Hkv = Hkv; jb->Nq = Nq; jb->Nk = Nk; jb->D = D;
        jb->scale = scale; jb->causal = causal; jb->rows = rows;
        jb->bias = bias; jb->bsb = bsb; jb->bsh = bsh; jb->bsq = bsq;
        jb->row_begin = total * t / nthreads;
        jb->row_end = total * (t + 1) / nthreads;
        jb->status = -2;
    }
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&tids[t], NULL, fwd_worker, &jobs[t]) != 0) jobs[t].status = 1;
    fwd_worker(&jobs[0]);
    int rc = jobs[0].status;
    for (int t = 1; t < nthreads; ++t) {
        if (jobs[t].status == 1) { fwd_worker(&jobs[t]); }  /* thread not started: run inline */
        else pthread_join(tids[t], NULL);
        if (jobs[t].status != 0) rc = jobs[t].status;
    }
    free(jobs); free(tids);
    return rc;
}

/* Forward over a list of rows without a bias. */
int oracle_attn_fwd_rows(const double *q, const double *k, const double *v,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                         double scale, int causal,
                         const int64_t *rows, int64_t n_rows,
                         double *o, double *lse, int nthreads)
{
    return oracle_attn_fwd_rows_bias(q, k, v, B, Hq, Hkv, Nq, Nk, D, scale, causal, NULL, 0, 0, 0,
                                     rows, n_rows, o, lse, nthreads);
}

/* Full forward: every row, outputs in the [B,Hq,Nq,D] / [B,Hq,Nq] layout. */
int oracle_attn_fwd(const double *q, const double *k, const double *v,
                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                    double scale, int causal, double *o, double *lse, int nthreads)
{
    return oracle_attn_fwd_rows(q, k, v, B, Hq, Hkv, Nq, Nk, D, scale, causal,
                                NULL, 0, o, lse, nthreads);
}

typedef struct {
    const double *q, *k, *v, *dout;
    double *dq;
    double *dk_part, *dv_part;     /* this thread's private [Nk, D] sums */
    int64_t b, g;                  /* the KV-head unit */
    int64_t Hq, Hkv, Nq, Nk, D;
    double scale;
    int causal;
    const double *bias;            /* additive bias as in the forward, or NULL */
    int64_t bsb, bsh, bsq;
    int64_t row_begin, row_end;    /* slice of the unit's G*Nq rows (head-major) */
    int status;
} bwd_job_t;

static void *bwd_worker(void *arg)
{
    bwd_job_t *jb = (bwd_job_t *)arg;
    const int64_t D = jb->D, Nk = jb->Nk, Nq = jb->Nq;
    const int64_t G = jb->Hq / jb->Hkv;
    const int64_t b = jb->b, g = jb->g;
    double *p = (double *)malloc((size_t)Nk * sizeof(double));
    double *dp = (double *)malloc((size_t)Nk * sizeof(double));
    if (!p || !dp) { free(p); free(dp); jb->status = -2; return NULL; }
    const int64_t u = b * jb->Hkv + g;
    const double *k_head = jb->k + u * Nk * D;
    const double *v_head = jb->v + u * Nk * D;
    double *dk_head = jb->dk_part;
    double *dv_head = jb->dv_part;
    memset(dk_head, 0, (size_t)(Nk * D) * sizeof(double));
    memset(dv_head, 0, (size_t)(Nk * D) * sizeof(double));
    for (int64_t fr = jb->row_begin; fr < jb->row_end; ++fr) {
        const int64_t hl = fr / Nq, i = fr % Nq;
        const int64_t h = g * G + hl;
        const int64_t r = (b * jb->Hq + h) * Nq + i;
        const double *q_row = jb->q + r * D;
        const double *do_row = jb->dout + r * D;
        double *dq_row = jb->dq + r * D;
        const int64_t nkeys = allowed_keys(i, Nk, jb->causal);
        const double *bias_row = jb->bias ? jb->bias + b * jb->bsb + h * jb->bsh + i * jb->bsq : NULL;
        /* scores and their log-sum-exp, as in the forward definition */
        double m = -INFINITY;
        for (int64_t j = 0; j < nkeys; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += q_row[d] * k_head[j * D + d];
            p[j] = jb->scale * dot;
            if (bias_row) p[j] += bias_row[j];
            if (p[j] > m) m = p[j];
        }
        if (m == -INFINITY) {   /* every key removed: O = 0 does not depend on q, k, v */
            for (int64_t d = 0; d < D; ++d) dq_row[d] = 0.0;
            continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) l += exp(p[j] - m);
        const double lse = m + log(l);
        /* P, dP and Delta */
        double delta = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            p[j] = exp(p[j] - lse);
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += do_row[d] * v_head[j * D + d];
            dp[j] = dot;
            delta += p[j] * dp[j];
        }
        for (int64_t d = 0; d < D; ++d) dq_row[d] = 0.0;
        for (int64_t j = 0; j < nkeys; ++j) {
            const double ds = p[j] * (dp[j] - delta);
            for (int64_t d = 0; d < D; ++d) {
                dq_row[d] += jb->scale * ds * k_head[j * D + d];
                dk_head[j * D + d] += jb->scale * ds * q_row[d];
                dv_head[j * D + d] += p[j] * do_row[d];
            }
        }
    }
    free(p); free(dp);
    jb->status = 0;
    return NULL;
}

/*
 * Full backward from the definition.  For each KV-head unit (b, g) the
 * unit's G*Nq query rows are split among the threads; every thread sums its
 * rows' contributions to dk/dv in a private buffer, and the buffers are added
 * up after the join, so no two threads ever write the same element.
 */
int oracle_attn_bwd_bias(const double *q, const double *k, const double *v, const double *dout,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                         double scale, int causal,
                         const double *bias, int64_t bsb, int64_t bsh, int64_t bsq,
                         double *dq, double *dk, double *dv, int nthreads)
{
    if (check_shape(B, Hq, Hkv, Nq, Nk, D)) return -1;
    if (bias && (bsb < 0 || bsh < 0 || bsq < 0)) return -1;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
    if (causal < 0 || causal > 1) return -1;   /* the backward covers none / top-left */
    const int64_t G = Hq / Hkv;
    const int64_t unit_rows = G * Nq;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > unit_rows) nthreads = (int)unit_rows;
    bwd_job_t *jobs = (bwd_job_t *)calloc((size_t)nthreads, sizeof(bwd_job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    double *parts = (double *)malloc((size_t)nthreads * 2 * (size_t)(Nk * D) * sizeof(double));
    if (!jobs || !tids || !parts) { free(jobs); free(tids); free(parts); return -2; }
    int rc = 0;
    for (int64_t b = 0; b < B && rc == 0; ++b) {
        for (int64_t g = 0; g < Hkv && rc == 0; ++g) {
            for (int t = 0; t < nthreads; ++t) {
                bwd_job_t *jb = &jobs[t];
                jb->q = q; jb->k = k; jb->v = v; jb->dout = dout; jb->dq = dq;
                jb->dk_part = parts + (size_t)(2 * t) * (size_t)(Nk * D);
                jb->dv_part = parts + (size_t)(2 * t + 1) * (size_t)(Nk * D);
                jb->b = b; jb->g = g;
                jb->Hq = Hq; jb->Hkv = Hkv; jb->Nq = Nq; jb->Nk = Nk; jb->D = D;
                jb->scale = scale; jb->causal = causal;
                jb->bias = bias; jb->bsb = bsb; jb->bsh = bsh; jb->bsq = bsq;
                jb->row_begin = unit_rows * t / nthreads;
                jb->row_end = unit_rows * (t + 1) / nthreads;
                jb->status = -2;
            }
            for (int t = 1; t < nthreads; ++t)
                if (pthread_create(&tids[t], NULL, bwd_worker, &jobs[t]) != 0) jobs[t].status = 1;
            bwd_worker(&jobs[0]);
            if (jobs[0].status != 0) rc = jobs[0].status;
            for (int t = 1; t < nthreads; ++t) {
                if (jobs[t].status == 1) { bwd_worker(&jobs[t]); }
                else pthread_join(tids[t], NULL);
                if (jobs[t].status != 0) rc = jobs[t].status;
            }
            const int64_t u = b * Hkv + g;
            for (int64_t e = 0; e < Nk * D; ++e) {
                double sk = 0.0, sv = 0.0;
                for (int t = 0; t < nthreads; ++t) {
                    sk += jobs[t].dk_part[e];
                    sv += jobs[t].dv_part[e];
                }
                dk[u * Nk * D + e] = sk;
                dv[u * Nk * D + e] = sv;
            }
        }
    }
    free(jobs); free(tids); free(parts);
    return rc;
}

/* Backward without a bias. */
int oracle_attn_bwd(const double *q, const double *k, const double *v, const double *dout,
                    int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t D,
                    double scale, int causal,
                    double *dq, double *dk, double *dv, int nthreads)
{
    return oracle_attn_bwd_bias(q, k, v, dout, B, Hq, Hkv, Nq, Nk, D, scale, causal, NULL, 0, 0, 0,
                                dq, dk, dv, nthreads);
}
