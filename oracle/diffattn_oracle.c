/*
 * Differential attention (causal) -- fp64 CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call this code:
 * only tests/, the smoke check in __graft_entry__ and the cpu_baseline /
 * --impl reference legs of bench.py load it.  It shares no code, header or
 * constant with the CUDA library.
 *
 * Every function is the plain definition written out in double precision:
 * materialise the causal scores of one query row, take a max-subtracted
 * softmax, form the weighted sum of value rows, then apply the
 * differential combine.  No online softmax, no tiling, no fusion.
 * Rows are independent by definition; threads only split the list of rows.
 *
 * Sources (page titles as printed on the pages):
 *   "Differential Transformer V2", pseudo-code DiffAttnV1 / DiffAttnV2:
 *       attn_b = flash_attn_func(q_b, k_b, v); lam_init = 0.8 - 0.6 exp(-0.3 layer_index);
 *       lam = exp(sum(lam_q1*lam_k1)) - exp(sum(lam_q2*lam_k2)) + lam_init;
 *       attn = rmsnorm(attn1 - lam*attn2) * (1 - lam_init)            (V1)
 *       attn = attn[:,0::2] - sigmoid(lam) * attn[:,1::2]            (V2)
 *   "How best to implement a differential transformer?" (nanoGPT issue 567),
 *       first CausalSelfAttention: subln = RMSNorm(2*head_dim, eps=1e-5,
 *       no affine); second: scores scaled by 1/sqrt(k.size(-1)) and masked
 *       with a lower-triangular causal mask.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - softmax scale is 1/sqrt(d), d = query/key head dim;
 *   - RMSNorm is x / sqrt(mean(x^2) + 1e-5) over the 2d channels of one
 *     (token, diff head) row, no weight;
 *   - V2 pair i uses heads 2i (kept) and 2i+1 (subtracted); query head h
 *     reads kv head h / (Hq/Hkv) (GQA groups contiguous);
 *   - decode: one query attends every one of the L cache rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- one causal softmax-attention row -------------------------------- */
/* q: [dqk]; keys row j at k + j*k_stride; values row j at v + j*v_stride.
 * Attends keys 0..n-1.  Writes a[dv] = sum_j softmax(q.k_j * scale)_j v_j.
 * scores: caller-provided scratch of n doubles. */
static void attend_row(const double *q, const double *k, int64_t k_stride,
                       const double *v, int64_t v_stride, int64_t n, int dqk,
                       int dv, double scale, double *scores, double *a)
{
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        const double *kj = k + j * k_stride;
        double s = 0.0;
        for (int c = 0; c < dqk; ++c)
            s += q[c] * kj[c];
        s *= scale;
        scores[j] = s;
        if (s > mx)
            mx = s;
    }
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        scores[j] = exp(scores[j] - mx);
        sum += scores[j];
    }
    for (int c = 0; c < dv; ++c)
        a[c] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        const double p = scores[j] / sum;
        const double *vj = v + j * v_stride;
        for (int c = 0; c < dv; ++c)
            a[c] += p * vj[c];
    }
}

/* lam_init = 0.8 - 0.6 exp(-0.3 layer_index)  (DiffAttnV1 pseudo-code) */
double oracle_lambda_init(int layer_index)
{
    return 0.8 - 0.6 * exp(-0.3 * (double)layer_index);
}

/* lam = exp(sum(lq1*lk1)) - exp(sum(lq2*lk2)) + lam_init  (DiffAttnV1) */
double oracle_lambda_full(const double *lq1, const double *lk1,
                          const double *lq2, const double *lk2, int d,
                          double lam_init)
{
    double s1 = 0.0, s2 = 0.0;
    for (int c = 0; c < d; ++c) {
        s1 += lq1[c] * lk1[c];
        s2 += lq2[c] * lk2[c];
    }
    return exp(s1) - exp(s2) + lam_init;
}

/* RMSNorm without affine weight: y = x / sqrt(mean(x^2) + eps) */
void oracle_rmsnorm(const double *x, int n, double eps, double *y)
{
    double ms = 0.0;
    for (int c = 0; c < n; ++c)
        ms += x[c] * x[c];
    ms /= (double)n;
    const double r = 1.0 / sqrt(ms + eps);
    for (int c = 0; c < n; ++c)
        y[c] = x[c] * r;
}

/* ---- work splitting over rows ----------------------------------------- */
typedef struct {
    int kind;                 /* 1 = V1, 2 = V2 prefill, 3 = V2 decode */
    const double *q1, *q2, *k1, *k2, *v, *lam;
    double lam_full, lam_init;
    int B, T, H, dqk, dv, Hkv, G;
    int64_t L;
    const int64_t *lens;      /* decode: cached rows per sequence, or NULL for L */
    const int64_t *rows;      /* nrows row ids, or NULL for all */
    int64_t nrows;
    double *out;
    int tid, nthreads;
} job_t;

/* V1 row id r = (b*T + t)*H + h.  Layouts (contiguous):
 *   q1,q2,k1,k2 (B,T,H,d); v (B,T,H,2d); out row = 2d doubles. */
/* DiffAttnV1 after the two attentions: x = a1 - lam*a2, RMSNorm over the
 * 2d channels (no affine weight), times (1 - lam_init). */
static void v1_combine(const job_t *J, const double *a1, const double *a2,
                       double *x, double *y)
{
    const int dv = J->dv;
    for (int c = 0; c < dv; ++c)
        x[c] = a1[c] - J->lam_full * a2[c];
    oracle_rmsnorm(x, dv, 1e-5, y);
    for (int c = 0; c < dv; ++c)
        y[c] *= (1.0 - J->lam_init);
}

static void v1_row(const job_t *J, int64_t r, double *scores, double *a1,
                   double *a2, double *x, double *y)
{
    const int H = J->H, T = J->T, d = J->dqk, dv = J->dv;
    const int h = (int)(r % H);
    const int t = (int)((r / H) % T);
    const int b = (int)(r / ((int64_t)H * T));
    const int64_t qk_row = (int64_t)H * d;   /* stride between tokens */
    const int64_t v_row = (int64_t)H * dv;
    const double *q1 = J->q1 + (((int64_t)b * T + t) * H + h) * d;
    const double *q2 = J->q2 + (((int64_t)b * T + t) * H + h) * d;
    const double *k1 = J->k1 + ((int64_t)b * T * H + h) * d;
    const double *k2 = J->k2 + ((int64_t)b * T * H + h) * d;
    const double *v = J->v + ((int64_t)b * T * H + h) * dv;
    const double scale = 1.0 / sqrt((double)d);
    /* causal: keys 0..t */
    attend_row(q1, k1, qk_row, v, v_row, (int64_t)t + 1, d, dv, scale, scores, a1);
    attend_row(q2, k2, qk_row, v, v_row, (int64_t)t + 1, d, dv, scale, scores, a2);
    v1_combine(J, a1, a2, x, y);
}

/* V2 prefill row id r = (b*T + t)*P + i, P = H (pairs).  Layouts:
 *   q (B,T,2P,D); k,v (B,T,Hkv,D); lam (B,T,P); out row = D doubles. */
static void v2_row(const job_t *J, int64_t r, double *scores, double *a1,
                   double *a2, double *y)
{
    const int P = J->H, T = J->T, D = J->dqk, Hkv = J->Hkv, G = J->G;
    const int Hq = 2 * P;
    const int i = (int)(r % P);
    const int t = (int)((r / P) % T);
    const int b = (int)(r / ((int64_t)P * T));
    const int he = 2 * i, ho = 2 * i + 1;
    const int g = he / G;        /* == ho / G because G is even */
    const double *qe = J->q1 + (((int64_t)b * T + t) * Hq + he) * D;
    const double *qo = J->q1 + (((int64_t)b * T + t) * Hq + ho) * D;
    const double *k = J->k1 + ((int64_t)b * T * Hkv + g) * D;
    const double *v = J->v + ((int64_t)b * T * Hkv + g) * D;
    const int64_t kv_row = (int64_t)Hkv * D;
    const double scale = 1.0 / sqrt((double)D);
    attend_row(qe, k, kv_row, v, kv_row, (int64_t)t + 1, D, D, scale, scores, a1);
    attend_row(qo, k, kv_row, v, kv_row, (int64_t)t + 1, D, D, scale, scores, a2);
    const double lg = J->lam[((int64_t)b * T + t) * P + i];
    const double sg = 1.0 / (1.0 + exp(-lg));
    for (int c = 0; c < D; ++c)
        y[c] = a1[c] - sg * a2[c];
}

/* V2 decode row id r = b*P + i.  Layouts:
 *   q (B,2P,D); k,v cache (B,L,Hkv,D); lam (B,P); out row = D doubles.
 * The single new query attends all L cache rows (its own K/V included). */
static void dec_row(const job_t *J, int64_t r, double *scores, double *a1,
                    double *a2, double *y)
{
    const int P = J->H, D = J->dqk, Hkv = J->Hkv, G = J->G;
    const int Hq = 2 * P;
    const int64_t Lc = J->L;   /* rows allocated per sequence */
    const int i = (int)(r % P);
    const int b = (int)(r / P);
    const int64_t L = J->lens ? J->lens[b] : Lc;   /* rows this sequence attends */
    const int he = 2 * i, ho = 2 * i + 1;
    const int g = he / G;
    const double *qe = J->q1 + ((int64_t)b * Hq + he) * D;
    const double *qo = J->q1 + ((int64_t)b * Hq + ho) * D;
    const double *k = J->k1 + ((int64_t)b * Lc * Hkv + g) * D;
    const double *v = J->v + ((int64_t)b * Lc * Hkv + g) * D;
    const int64_t kv_row = (int64_t)Hkv * D;
    const double scale = 1.0 / sqrt((double)D);
    attend_row(qe, k, kv_row, v, kv_row, L, D, D, scale, scores, a1);
    attend_row(qo, k, kv_row, v, kv_row, L, D, D, scale, scores, a2);
    const double lg = J->lam[(int64_t)b * P + i];
    const double sg = 1.0 / (1.0 + exp(-lg));
    for (int c = 0; c < D; ++c)
        y[c] = a1[c] - sg * a2[c];
}

/* V1 decode row id r = b*H + h.  Layouts:
 *   q1, q2 (B,H,d); k1, k2 caches (B,L,H,d); v cache (B,L,H,2d); out row 2d.
 * The new token attends cached rows 0 .. len_b - 1 of both branches. */
static void v1dec_row(const job_t *J, int64_t r, double *scores, double *a1,
                      double *a2, double *x, double *y)
{
    const int H = J->H, d = J->dqk, dv = J->dv;
    const int64_t Lc = J->L;
    const int h = (int)(r % H);
    const int b = (int)(r / H);
    const int64_t L = J->lens ? J->lens[b] : Lc;
    const double *q1 = J->q1 + ((int64_t)b * H + h) * d;
    const double *q2 = J->q2 + ((int64_t)b * H + h) * d;
    const double *k1 = J->k1 + ((int64_t)b * Lc * H + h) * d;
    const double *k2 = J->k2 + ((int64_t)b * Lc * H + h) * d;
    const double *v = J->v + ((int64_t)b * Lc * H + h) * dv;
    const double scale = 1.0 / sqrt((double)d);
    attend_row(q1, k1, (int64_t)H * d, v, (int64_t)H * dv, L, d, dv, scale, scores, a1);
    attend_row(q2, k2, (int64_t)H * d, v, (int64_t)H * dv, L, d, dv, scale, scores, a2);
    v1_combine(J, a1, a2, x, y);
}

static void *worker(void *arg)
{
    const job_t *J = (const job_t *)arg;
    const int64_t nkeys = (J->kind >= 3) ? J->L : (int64_t)J->T;
    const int dv = J->dv;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(nkeys > 0 ? nkeys : 1));
    double *buf = (double *)malloc(sizeof(double) * (size_t)dv * 4);
    if (!scores || !buf) {
        free(scores);
        free(buf);
        return (void *)1;
    }
    double *a1 = buf, *a2 = buf + dv, *x = buf + 2 * dv;
    for (int64_t n = J->tid; n < J->nrows; n += J->nthreads) {
        const int64_t r = J->rows ? J->rows[n] : n;
        double *y = J->out + n * dv;
        if (J->kind == 1)
            v1_row(J, r, scores, a1, a2, x, y);
        else if (J->kind == 2)
            v2_row(J, r, scores, a1, a2, y);
        else if (J->kind == 3)
            dec_row(J, r, scores, a1, a2, y);
        else
            v1dec_row(J, r, scores, a1, a2, x, y);
    }
    free(scores);
    free(buf);
    return NULL;
}

static int run_jobs(const job_t *proto, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    job_t jobs[256];
    pthread_t th[256];
    int started[256];
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = *proto;
        jobs[i].tid = i;
        jobs[i].nthreads = nthreads;
        started[i] = pthread_create(&th[i], NULL, worker, &jobs[i]) == 0;
        if (!started[i])
            rc = 2;
    }
    for (int i = 0; i < nthreads; ++i) {
        if (started[i]) {
            void *ret = NULL;
            pthread_join(th[i], &ret);
            if (ret)
                rc = 1;
        }
    }
    return rc;
}

/* DIFF V1 forward.  rows: ids (b*T+t)*H+h, or NULL for all B*T*H rows in
 * that order.  out: nrows x 2d.  Returns 0 on success. */
int oracle_v1_fwd(const double *q1, const double *q2, const double *k1,
                  const double *k2, const double *v, const double *lq1,
                  const double *lk1, const double *lq2, const double *lk2,
                  int B, int T, int H, int d, int layer_index,
                  const int64_t *rows, int64_t nrows, double *out,
                  int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof(J));
    J.kind = 1;
    J.q1 = q1; J.q2 = q2; J.k1 = k1; J.k2 = k2; J.v = v;
    J.B = B; J.T = T; J.H = H; J.dqk = d; J.dv = 2 * d;
    J.lam_init = oracle_lambda_init(layer_index);
    J.lam_full = oracle_lambda_full(lq1, lk1, lq2, lk2, d, J.lam_init);
    J.rows = rows;
    J.nrows = rows ? nrows : (int64_t)B * T * H;
    J.out = out;
    return run_jobs(&J, nthreads);
}

/* DIFF V2 prefill.  Hq query heads (even), Hkv kv heads, G = Hq/Hkv even.
 * rows: ids (b*T+t)*(Hq/2)+i, or NULL for all.  out: nrows x D. */
int oracle_v2_fwd(const double *q, const double *k, const double *v,
                  const double *lam, int B, int T, int Hq, int Hkv, int D,
                  const int64_t *rows, int64_t nrows, double *out,
                  int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof(J));
    J.kind = 2;
    J.q1 = q; J.k1 = k; J.v = v; J.lam = lam;
    J.B = B; J.T = T; J.H = Hq / 2; J.dqk = D; J.dv = D;
    J.Hkv = Hkv; J.G = Hq / Hkv;
    J.rows = rows;
    J.nrows = rows ? nrows : (int64_t)B * T * (Hq / 2);
    J.out = out;
    return run_jobs(&J, nthreads);
}

/* DIFF V2 decode: one query token per sequence against an L-row cache.
 * lens: rows attended per sequence (each in 1..L), or NULL for all L.
 * rows: ids b*(Hq/2)+i, or NULL for all.  out: nrows x D. */
int oracle_v2_decode(const double *q, const double *k, const double *v,
                     const double *lam, int B, int64_t L, int Hq, int Hkv,
                     int D, const int64_t *lens, const int64_t *rows,
                     int64_t nrows, double *out, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof(J));
    J.kind = 3;
    J.lens = lens;
    J.q1 = q; J.k1 = k; J.v = v; J.lam = lam;
    J.B = B; J.L = L; J.H = Hq / 2; J.dqk = D; J.dv = D;
    J.Hkv = Hkv; J.G = Hq / Hkv;
    J.rows = rows;
    J.nrows = rows ? nrows : (int64_t)B * (Hq / 2);
    J.out = out;
    return run_jobs(&J, nthreads);
}

/* DIFF V1 decode: the V1 operation for one new query token per sequence
 * against L cached rows (its own K/V included).  q1, q2 (B,H,d); k1, k2
 * (B,L,H,d); v (B,L,H,2d); lens rows attended per sequence or NULL for L.
 * rows: ids b*H+h, or NULL for all.  out: nrows x 2d. */
int oracle_v1_decode(const double *q1, const double *q2, const double *k1,
                     const double *k2, const double *v, const double *lq1,
                     const double *lk1, const double *lq2, const double *lk2,
                     int B, int64_t L, int H, int d, int layer_index,
                     const int64_t *lens, const int64_t *rows, int64_t nrows,
                     double *out, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof(J));
    J.kind = 4;
    J.lens = lens;
    J.q1 = q1; J.q2 = q2; J.k1 = k1; J.k2 = k2; J.v = v;
    J.B = B; J.L = L; J.H = H; J.dqk = d; J.dv = 2 * d;
    J.lam_init = oracle_lambda_init(layer_index);
    J.lam_full = oracle_lambda_full(lq1, lk1, lq2, lk2, d, J.lam_init);
    J.rows = rows;
    J.nrows = rows ? nrows : (int64_t)B * H;
    J.out = out;
    return run_jobs(&J, nthreads);
}
