/*
 * ORACLE -- test infrastructure, not product code.
 *
 * A plain, slow fp64 CPU implementation of exact scaled-dot-product
 * attention and of the log-sum-exp merge of per-chunk partial results.
 * Only the test-suite, the smoke check and the benchmark's CPU-baseline leg
 * load this library; the CUDA path never links, includes or calls it, and
 * the two share no source.
 *
 * Where each definition comes from:
 *
 *  attention   page "Ulysses与Ring-Attention序列并行技术详解" (Ulysses and
 *              Ring-Attention sequence parallelism explained), Ulysses part,
 *              ulysses_attention_forward listing: scores are Q times K
 *              transposed divided by the square root of the head dimension,
 *              a softmax over the keys, then the weighted sum of V rows.
 *              The softmax is evaluated with the row maximum subtracted
 *              before exponentiation, the local maximum m_i and local
 *              exponent sum z_i of page "ms-swift支持Ulysses与Ring-Attention
 *              降低长文本显存占用", section "Ring-Attention：面向大规模部署的
 *              工程利器". lse is m + ln(z), natural log as the pages' torch.log.
 *
 *  masking     causal masking and the global offsets q_off / kv_off are not
 *              on the pages. Reading taken: query row r of a block starting at
 *              global position q_off sees key j of a chunk starting at kv_off
 *              iff kv_off + j <= q_off + r. A row that sees no key has
 *              O = 0 and lse = -inf (the empty softmax).
 *
 *  GQA         not on the pages. Reading taken: query head hq reads KV head
 *              hq / (Hq / Hkv) (contiguous groups).
 *
 *  merge       page "Ulysses与Ring-Attention序列并行技术详解", Ring-Attention
 *              part, the log-space accumulation listing (output_acc,
 *              logsumexp_acc). As printed, that listing starts the
 *              accumulator at lse = 0 and takes its maximum over the query
 *              axis; the reading taken is the intended per-row merge of
 *              partials (O_i, lse_i):
 *                M = max_i lse_i,  w_i = exp(lse_i - M),
 *                lse = M + ln(sum_i w_i),  O = sum_i w_i O_i / sum_i w_i,
 *              with an empty accumulator (all lse_i = -inf) giving O = 0,
 *              lse = -inf.
 *
 * Inputs are the raw bf16 bit patterns; every value is widened exactly to
 * double. All arithmetic is IEEE double with the host libm's exp and log,
 * compiled without fast-math, in the order of the definitions above.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    int B, Hq, Hkv, Sq, Skv, D;
    long long q_off, kv_off;
    long long q_head_stride, kv_head_stride; /* elements between heads' row 0 */
    int causal;
    double scale;
    const long long *rows; /* NULL: all rows; else [B*Hq][nrows] row indices */
    int nrows;
    double *o, *lse;
    int nthreads;
    int tid;
} attn_job;

/* One query row of one (batch, query head): the definition, written out. */
static void attention_row(const attn_job *j, int b, int hq, long long r, double *o_row,
                          double *lse_out, double *s)
{
    const int D = j->D;
    const int group = j->Hq / j->Hkv;
    const int hkv = hq / group;
    const uint16_t *qr = j->q + (long long)(b * j->Hq + hq) * j->q_head_stride + r * D;
    const uint16_t *kh = j->k + (long long)(b * j->Hkv + hkv) * j->kv_head_stride;
    const uint16_t *vh = j->v + (long long)(b * j->Hkv + hkv) * j->kv_head_stride;

    /* Visible keys: all of them, or under causal masking those whose global
     * position does not exceed the query's. */
    long long nvis = j->Skv;
    if (j->causal) {
        long long last = j->q_off + r - j->kv_off; /* largest visible key index */
        nvis = last + 1;
        if (nvis < 0) nvis = 0;
        if (nvis > j->Skv) nvis = j->Skv;
    }
    for (int d = 0; d < D; d++) o_row[d] = 0.0;
    if (nvis == 0) {
        *lse_out = -INFINITY;
        return;
    }

    /* s_j = scale * <q, k_j> */
    for (long long t = 0; t < nvis; t++) {
        const uint16_t *kr = kh + t * D;
        double dot = 0.0;
        for (int d = 0; d < D; d++) dot += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);
        s[t] = j->scale * dot;
    }
    /* m = max_j s_j */
    double m = s[0];
    for (long long t = 1; t < nvis; t++)
        if (s[t] > m) m = s[t];
    /* l = sum_j exp(s_j - m);  O = sum_j exp(s_j - m) v_j / l */
    double l = 0.0;
    for (long long t = 0; t < nvis; t++) {
        double p = exp(s[t] - m);
        l += p;
        const uint16_t *vr = vh + t * D;
        for (int d = 0; d < D; d++) o_row[d] += p * bf16_to_double(vr[d]);
    }
    for (int d = 0; d < D; d++) o_row[d] /= l;
    *lse_out = m + log(l);
}

static void *attention_worker(void *arg)
{
    const attn_job *j = (const attn_job *)arg;
    const long long per_head = j->rows ? j->nrows : j->Sq;
    const long long total = (long long)j->B * j->Hq * per_head;
    double *s = (double *)malloc(sizeof(double) * (size_t)(j->Skv > 0 ? j->Skv : 1));
    if (!s) return (void *)1;
    /* Rows are dealt round-robin so causal rows of every length are spread
     * over all threads. */
    for (long long item = j->tid; item < total; item += j->nthreads) {
        long long bh = item / per_head;
        long long i = item % per_head;
        int b = (int)(bh / j->Hq), hq = (int)(bh % j->Hq);
        long long r = j->rows ? j->rows[bh * j->nrows + i] : i;
        attention_row(j, b, hq, r, j->o + item * j->D, j->lse + item, s);
    }
    free(s);
    return NULL;
}

/*
 * Exact attention for every (batch, query head, query row), or for the rows
 * listed in `rows` ([B*Hq][nrows], each in [0, Sq)).
 *
 *   q  bf16 bits, row r of head (b, hq) at q + (b*Hq + hq)*q_head_stride + r*D
 *   k, v  bf16 bits, key t of KV head (b, hkv) at k + (b*Hkv + hkv)*kv_head_stride + t*D
 *   o  [B*Hq][rows per head][D] doubles;  lse  [B*Hq][rows per head] doubles
 *
 * Returns 0, or -1 on invalid arguments or allocation failure.
 */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                     int Hkv, int Sq, int Skv, int D, long long q_off, long long kv_off,
                     long long q_head_stride, long long kv_head_stride, int causal,
                     double scale, const long long *rows, int nrows, double *o, double *lse,
                     int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Sq < 0 || Skv < 0 || D <= 0)
        return -1;
    if (rows) {
        for (long long i = 0; i < (long long)B * Hq * nrows; i++)
            if (rows[i] < 0 || rows[i] >= Sq) return -1;
    }
    if (nthreads < 1) nthreads = 1;
    attn_job *jobs = (attn_job *)calloc((size_t)nthreads, sizeof(attn_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    int rc = 0;
    for (int t = 0; t < nthreads; t++) {
        attn_job j = {q, k, v, B, Hq, Hkv, Sq, Skv, D, q_off, kv_off, q_head_stride,
                      kv_head_stride, causal, scale, rows, nrows, o, lse, nthreads, t};
        jobs[t] = j;
    }
    int started = 0;
    for (; started < nthreads; started++)
        if (pthread_create(&th[started], NULL, attention_worker, &jobs[started]) != 0) break;
    if (started == 0) {
        /* no threads available: run everything on this one */
        jobs[0].nthreads = 1;
        if (attention_worker(&jobs[0])) rc = -1;
    } else {
        if (started < nthreads) {
            /* the jobs that did not start are run here, in turn */
            for (int t = started; t < nthreads; t++)
                if (attention_worker(&jobs[t])) rc = -1;
        }
        for (int t = 0; t < started; t++) {
            void *ret = NULL;
            pthread_join(th[t], &ret);
            if (ret) rc = -1;
        }
    }
    free(jobs);
    free(th);
    return rc;
}

/*
 * Merge of P partial results per row.
 *   o_parts [P][nrows][D], lse_parts [P][nrows]  ->  o [nrows][D], lse [nrows]
 */
void oracle_lse_merge(const double *o_parts, const double *lse_parts, int P, long long nrows,
                      int D, double *o, double *lse)
{
    for (long long r = 0; r < nrows; r++) {
        double M = -INFINITY;
        for (int i = 0; i < P; i++)
            if (lse_parts[(long long)i * nrows + r] > M) M = lse_parts[(long long)i * nrows + r];
        double *orow = o + r * D;
        for (int d = 0; d < D; d++) orow[d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double wsum = 0.0;
        for (int i = 0; i < P; i++) {
            double li = lse_parts[(long long)i * nrows + r];
            if (li == -INFINITY) continue; /* an empty partial has zero weight */
            double w = exp(li - M);
            wsum += w;
            const double *oi = o_parts + ((long long)i * nrows + r) * D;
            for (int d = 0; d < D; d++) orow[d] += w * oi[d];
        }
        for (int d = 0; d < D; d++) orow[d] /= wsum;
        lse[r] = M + log(wsum);
    }
}

/*
 * Backward of attention: the gradients of Q, K and V for a loss whose
 * gradient with respect to O is dO. The pages mention the backward pass that
 * FlashAttention recomputes block by block (page "ms-swift集成FlashAttention
 * 2/3，长文本训练更高效", section "FlashAttention 如何破局？不只是融合内核")
 * without writing it out; this is the chain rule through the definition above
 * (visibility and GQA mapping as there, q_off = kv_off = 0, Sq = Skv = S):
 *   P_ij  = exp(s_ij - m_i) / l_i                 (the softmax of row i)
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = <dO_i, v_j>
 *   dS_ij = P_ij (dP_ij - sum_t P_it dP_it)        (the softmax Jacobian)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 * dK and dV of a KV head sum over the query heads of its group.
 */
typedef struct {
    const uint16_t *q, *k, *v, *dout;
    int B, Hq, Hkv, S, D, causal;
    double scale;
    double *dq, *dk, *dv;
    int nthreads, tid;
} bwd_job;

static void *backward_worker(void *arg)
{
    const bwd_job *j = (const bwd_job *)arg;
    const int S = j->S, D = j->D, group = j->Hq / j->Hkv;
    double *p = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    if (!p || !dp) {
        free(p);
        free(dp);
        return (void *)1;
    }
    /* one (batch, KV head) per item: its dK, dV and its query heads' dQ */
    for (int item = j->tid; item < j->B * j->Hkv; item += j->nthreads) {
        const int b = item / j->Hkv, hkv = item % j->Hkv;
        const uint16_t *kh = j->k + ((long long)b * j->Hkv + hkv) * S * D;
        const uint16_t *vh = j->v + ((long long)b * j->Hkv + hkv) * S * D;
        double *dkh = j->dk + ((long long)b * j->Hkv + hkv) * S * D;
        double *dvh = j->dv + ((long long)b * j->Hkv + hkv) * S * D;
        for (long long t = 0; t < (long long)S * D; t++) dkh[t] = dvh[t] = 0.0;
        for (int hq = hkv * group; hq < (hkv + 1) * group; hq++) {
            const uint16_t *qh = j->q + ((long long)b * j->Hq + hq) * S * D;
            const uint16_t *doh = j->dout + ((long long)b * j->Hq + hq) * S * D;
            double *dqh = j->dq + ((long long)b * j->Hq + hq) * S * D;
            for (long long i = 0; i < S; i++) {
                const long long nvis = j->causal ? i + 1 : S;
                const uint16_t *qi = qh + i * D, *doi = doh + i * D;
                double *dqi = dqh + i * D;
                for (int d = 0; d < D; d++) dqi[d] = 0.0;
                /* the row's softmax */
                double m = -INFINITY;
                for (long long t = 0; t < nvis; t++) {
                    double dot = 0.0;
                    for (int d = 0; d < D; d++) dot += bf16_to_double(qi[d]) * bf16_to_double(kh[t * D + d]);
                    p[t] = j->scale * dot;
                    if (p[t] > m) m = p[t];
                }
                double l = 0.0;
                for (long long t = 0; t < nvis; t++) {
                    p[t] = exp(p[t] - m);
                    l += p[t];
                }
                for (long long t = 0; t < nvis; t++) p[t] /= l;
                /* dP and its P-weighted row sum */
                double psum = 0.0;
                for (long long t = 0; t < nvis; t++) {
                    double dot = 0.0;
                    for (int d = 0; d < D; d++) dot += bf16_to_double(doi[d]) * bf16_to_double(vh[t * D + d]);
                    dp[t] = dot;
                    psum += p[t] * dot;
                }
                for (long long t = 0; t < nvis; t++) {
                    const double ds = p[t] * (dp[t] - psum);
                    for (int d = 0; d < D; d++) {
                        dqi[d] += j->scale * ds * bf16_to_double(kh[t * D + d]);
                        dkh[t * D + d] += j->scale * ds * bf16_to_double(qi[d]);
                        dvh[t * D + d] += p[t] * bf16_to_double(doi[d]);
                    }
                }
            }
        }
    }
    free(p);
    free(dp);
    return NULL;
}

/*
 * q, k, v, dout: bf16 bits, contiguous [B][H][S][D]; dq [B][Hq][S][D], dk and
 * dv [B][Hkv][S][D] doubles (outputs). Returns 0, or -1 on invalid arguments.
 */
int oracle_attention_backward(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const uint16_t *dout, int B, int Hq, int Hkv, int S, int D,
                              int causal, double scale, double *dq, double *dk, double *dv,
                              int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || S < 0 || D <= 0) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    bwd_job jobs[256];
    int rc = 0;
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (bwd_job){q, k, v, dout, B, Hq, Hkv, S, D, causal, scale, dq, dk, dv, nthreads, t};
        if (pthread_create(&th[t], NULL, backward_worker, &jobs[t]) != 0) {
            nthreads = t;
            rc = -1;
            break;
        }
    }
    for (int t = 0; t < nthreads; t++) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret) rc = -1;
    }
    return rc;
}

/*
 * dQ of selected query rows only: the same chain rule for one row at a time
 * (dQ_i needs only row i's softmax and dP), for checking outputs of problems
 * too large to differentiate whole. rows: int64 [B*Hq][n] row indices (each
 * in [0, S)); dq_rows: doubles [B*Hq][n][D] (output). Returns 0, or -1 on
 * invalid arguments.
 */
typedef struct {
    const uint16_t *q, *k, *v, *dout;
    int B, Hq, Hkv, S, D, causal;
    double scale;
    const long long *rows;
    int n;
    double *dq_rows;
    int nthreads, tid;
} dq_rows_job;

static void *dq_rows_worker(void *arg)
{
    const dq_rows_job *j = (const dq_rows_job *)arg;
    const int S = j->S, D = j->D, group = j->Hq / j->Hkv;
    double *p = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    if (!p || !dp) {
        free(p);
        free(dp);
        return (void *)1;
    }
    for (long long item = j->tid; item < (long long)j->B * j->Hq * j->n; item += j->nthreads) {
        const long long bh = item / j->n;
        const int b = (int)(bh / j->Hq), hq = (int)(bh % j->Hq), hkv = hq / group;
        const long long i = j->rows[item];
        const uint16_t *kh = j->k + ((long long)b * j->Hkv + hkv) * S * D;
        const uint16_t *vh = j->v + ((long long)b * j->Hkv + hkv) * S * D;
        const uint16_t *qi = j->q + (bh * S + i) * D, *doi = j->dout + (bh * S + i) * D;
        double *dqi = j->dq_rows + item * D;
        const long long nvis = j->causal ? i + 1 : S;
        for (int d = 0; d < D; d++) dqi[d] = 0.0;
        double m = -INFINITY;
        for (long long t = 0; t < nvis; t++) {
            double dot = 0.0;
            for (int d = 0; d < D; d++) dot += bf16_to_double(qi[d]) * bf16_to_double(kh[t * D + d]);
            p[t] = j->scale * dot;
            if (p[t] > m) m = p[t];
        }
        double l = 0.0;
        for (long long t = 0; t < nvis; t++) {
            p[t] = exp(p[t] - m);
            l += p[t];
        }
        for (long long t = 0; t < nvis; t++) p[t] /= l;
        double psum = 0.0;
        for (long long t = 0; t < nvis; t++) {
            double dot = 0.0;
            for (int d = 0; d < D; d++) dot += bf16_to_double(doi[d]) * bf16_to_double(vh[t * D + d]);
            dp[t] = dot;
            psum += p[t] * dot;
        }
        for (long long t = 0; t < nvis; t++) {
            const double ds = p[t] * (dp[t] - psum);
            for (int d = 0; d < D; d++) dqi[d] += j->scale * ds * bf16_to_double(kh[t * D + d]);
        }
    }
    free(p);
    free(dp);
    return NULL;
}

int oracle_attention_backward_dq_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                      const uint16_t *dout, int B, int Hq, int Hkv, int S, int D,
                                      int causal, double scale, const long long *rows, int n,
                                      double *dq_rows, int nthreads)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || S < 0 || D <= 0 || n < 0) return -1;
    for (long long t = 0; t < (long long)B * Hq * n; t++)
        if (rows[t] < 0 || rows[t] >= S) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    dq_rows_job jobs[256];
    int rc = 0;
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (dq_rows_job){q, k, v, dout, B, Hq, Hkv, S, D, causal, scale, rows, n, dq_rows, nthreads, t};
        if (pthread_create(&th[t], NULL, dq_rows_worker, &jobs[t]) != 0) {
            nthreads = t;
            rc = -1;
            break;
        }
    }
    for (int t = 0; t < nthreads; t++) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret) rc = -1;
    }
    return rc;
}
