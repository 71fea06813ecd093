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
 * The gradients (end of file) follow the chain rule of the same definitions
 * row by row; threads split the list of heads (V1) or kv groups (V2), whose
 * gradients do not overlap.
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
 *   modded-nanogpt pull request "New Record: Paired Head Attention (-3.5s,
 *       -65 steps)", section "Updates in PR": the k, q and v of two heads are
 *       interleaved into one sequence twice as long, attended causally with
 *       one softmax (paired_row below).
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

/* ---- row log-sum-exp of the causal scores ---------------------------- */
/* For every batch entry b, query head h and row t: the log-sum-exp (natural
 * log) of the scaled scores that row's softmax normalises,
 *   lse = log sum_{j <= t} exp(q_t . k_j / sqrt(d)),
 * taken as max + log(sum exp(s - max)).  q (B, T, Hq, d), k (B, T, Hk, d)
 * contiguous, query head h reads key head h / (Hq / Hk); out (B, Hq, T). */
void oracle_lse(const double *q, const double *k, int B, int T, int Hq, int Hk,
                int d, double *out)
{
    const double scale = 1.0 / sqrt((double)d);
    const int G = Hq / Hk;
    double *s = (double *)malloc(sizeof(double) * (size_t)T);
    if (!s) return;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h)
            for (int t = 0; t < T; ++t) {
                const double *qt = q + (((int64_t)b * T + t) * Hq + h) * d;
                const int n = t + 1;   /* causal: keys 0 .. t */
                double mx = -INFINITY;
                for (int j = 0; j < n; ++j) {
                    const double *kj = k + (((int64_t)b * T + j) * Hk + h / G) * d;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c)
                        acc += qt[c] * kj[c];
                    s[j] = acc * scale;
                    if (s[j] > mx) mx = s[j];
                }
                double sum = 0.0;
                for (int j = 0; j < n; ++j)
                    sum += exp(s[j] - mx);
                out[((int64_t)b * Hq + h) * T + t] = mx + log(sum);
            }
    free(s);
}

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
    int kind;                 /* 1 = V1, 2 = V2 prefill, 3 = V2 decode, 4 = V1 decode, 5 = paired heads */
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

/* Paired Head Attention row id r = (b*T + t)*H + h (modded-nanogpt pull
 * request "New Record: Paired Head Attention (-3.5s, -65 steps)", section
 * "Updates in PR").  The k, q and v of heads 2i and 2i+1 are
 * interleaved into one sequence of length 2T, position 2t + e holding token t
 * of head 2i + e; plain causal softmax attention runs over that sequence and
 * its outputs are de-interleaved back to (token, head).  So the query of
 * token t, head 2i + e attends the interleaved positions 0 .. 2t + e: both
 * heads' keys of tokens before t, head 2i's key of token t, and for e = 1
 * also its own.  Layouts (contiguous): q, k, v (B,T,H,D); out row = D. */
static void paired_row(const job_t *J, int64_t r, double *scores, double *a)
{
    const int H = J->H, T = J->T, D = J->dqk;
    const int h = (int)(r % H);
    const int t = (int)((r / H) % T);
    const int b = (int)(r / ((int64_t)H * T));
    const int i = h / 2, e = h % 2;
    const double *q = J->q1 + (((int64_t)b * T + t) * H + h) * D;
    const double scale = 1.0 / sqrt((double)D);
    const int64_t n = 2 * (int64_t)t + e + 1;      /* interleaved positions 0 .. 2t+e */
    double mx = -INFINITY;
    for (int64_t s = 0; s < n; ++s) {
        const int64_t ts = s / 2, hs = 2 * i + (int)(s % 2);
        const double *ks = J->k1 + (((int64_t)b * T + ts) * H + hs) * D;
        double x = 0.0;
        for (int c = 0; c < D; ++c)
            x += q[c] * ks[c];
        x *= scale;
        scores[s] = x;
        if (x > mx)
            mx = x;
    }
    double sum = 0.0;
    for (int64_t s = 0; s < n; ++s) {
        scores[s] = exp(scores[s] - mx);
        sum += scores[s];
    }
    for (int c = 0; c < D; ++c)
        a[c] = 0.0;
    for (int64_t s = 0; s < n; ++s) {
        const int64_t ts = s / 2, hs = 2 * i + (int)(s % 2);
        const double *vs = J->v + (((int64_t)b * T + ts) * H + hs) * D;
        const double w = scores[s] / sum;
        for (int c = 0; c < D; ++c)
            a[c] += w * vs[c];
    }
}

static void *worker(void *arg)
{
    const job_t *J = (const job_t *)arg;
    const int64_t nkeys = (J->kind == 5) ? 2 * (int64_t)J->T : (J->kind >= 3) ? J->L : (int64_t)J->T;
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
        else if (J->kind == 5)
            paired_row(J, r, scores, y);
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

/* Paired Head Attention forward: H heads (even), pairs (2i, 2i+1).
 * rows: ids (b*T+t)*H+h, or NULL for all.  out: nrows x D. */
int oracle_paired_fwd(const double *q, const double *k, const double *v,
                      int B, int T, int H, int D, const int64_t *rows,
                      int64_t nrows, double *out, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof(J));
    J.kind = 5;
    J.q1 = q; J.k1 = k; J.v = v;
    J.B = B; J.T = T; J.H = H; J.dqk = D; J.dv = D;
    J.rows = rows;
    J.nrows = rows ? nrows : (int64_t)B * T * H;
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

/* ======================================================================
 * Gradients (the backward of the same definitions).
 *
 * Written from the chain rule of the forward definitions above, with the
 * softmax Jacobian taken as is (no flash-style shortcut):
 *   one attention row a = sum_j p_j v_j, p = softmax(scale q.k_j), with
 *   upstream gradient g = dL/da:
 *     dL/dv_j += p_j g
 *     dp_j     = g . v_j
 *     ds_j     = p_j (dp_j - sum_l p_l dp_l)
 *     dL/dq   += scale sum_j ds_j k_j
 *     dL/dk_j += scale ds_j q
 *   RMSNorm y_c = x_c r, r = (mean(x^2) + eps)^(-1/2):
 *     dL/dx_c = r dy_c - r^3 x_c (sum_e dy_e x_e) / n
 *   DiffAttnV1: out = (1 - lam_init) y, x = a1 - lam a2:
 *     g1 = dL/dx, g2 = -lam dL/dx, dL/dlam = -sum (dL/dx . a2) over all rows;
 *     lam = exp(lq1.lk1) - exp(lq2.lk2) + lam_init:
 *     dlq1 = dlam exp(lq1.lk1) lk1, dlk1 = dlam exp(lq1.lk1) lq1,
 *     dlq2 = -dlam exp(lq2.lk2) lk2, dlk2 = -dlam exp(lq2.lk2) lq2.
 *   DiffAttnV2: out = a_e - sigmoid(l) a_o:
 *     g_e = dout, g_o = -sigmoid(l) dout,
 *     dL/dl = -sigmoid(l) (1 - sigmoid(l)) (dout . a_o).
 * ==================================================================== */

/* Backward of one attention row over keys 0..n-1.  g: upstream gradient
 * [dv]; accumulates into dq [dqk], dk rows (stride k_stride) and dv rows
 * (stride v_stride).  p, dp: scratch of n doubles each. */
static void attend_row_bwd(const double *q, const double *k, int64_t k_stride,
                           const double *v, int64_t v_stride, int64_t n,
                           int dqk, int dvd, double scale, const double *g,
                           double *p, double *dp, double *dq, double *dk,
                           double *dv)
{
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        const double *kj = k + j * k_stride;
        double s = 0.0;
        for (int c = 0; c < dqk; ++c)
            s += q[c] * kj[c];
        p[j] = s * scale;
        if (p[j] > mx)
            mx = p[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        p[j] = exp(p[j] - mx);
        sum += p[j];
    }
    double pdp = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        p[j] /= sum;
        const double *vj = v + j * v_stride;
        double t = 0.0;
        for (int c = 0; c < dvd; ++c)
            t += g[c] * vj[c];
        dp[j] = t;
        pdp += p[j] * t;
    }
    for (int64_t j = 0; j < n; ++j) {
        const double ds = p[j] * (dp[j] - pdp);
        const double *kj = k + j * k_stride;
        double *dkj = dk + j * k_stride;
        double *dvj = dv + j * v_stride;
        for (int c = 0; c < dqk; ++c) {
            dq[c] += scale * ds * kj[c];
            dkj[c] += scale * ds * q[c];
        }
        for (int c = 0; c < dvd; ++c)
            dvj[c] += p[j] * g[c];
    }
}

typedef struct {
    int kind;                 /* 1 = V1, 2 = V2 */
    const double *q1, *q2, *k1, *k2, *v, *lam, *dout;
    double lam_full, lam_init;
    int B, T, H, dqk, dv, Hkv, G;
    const int64_t *units;     /* V1: head ids b*H+h; V2: group ids b*Hkv+g */
    int64_t nunits;
    double *dq1, *dq2, *dk1, *dk2, *dvv, *dlam;   /* dlam: V1 one partial per unit, V2 (B,T,Hq/2) */
    double *dlam_abs;         /* V1: per unit, sum over rows and channels of |dx_c a2_c| */
    int tid, nthreads;
} bjob_t;

/* V1 head (b, h): every row t, both branches. */
static void v1_head_bwd(const bjob_t *J, int64_t u, int64_t slot, double *p,
                        double *dp, double *buf)
{
    const int H = J->H, T = J->T, d = J->dqk, dvd = J->dv;
    const int h = (int)(u % H);
    const int b = (int)(u / H);
    const int64_t qk_row = (int64_t)H * d, v_row = (int64_t)H * dvd;
    const double scale = 1.0 / sqrt((double)d);
    double *a1 = buf, *a2 = buf + dvd, *x = buf + 2 * dvd, *dx = buf + 3 * dvd;
    double *g2 = buf + 4 * dvd;
    const int64_t kbase = (int64_t)b * T * H + h;
    double dlam = 0.0, dlam_abs = 0.0;
    for (int t = 0; t < T; ++t) {
        const int64_t row = ((int64_t)b * T + t) * H + h;
        const double *q1 = J->q1 + row * d, *q2 = J->q2 + row * d;
        attend_row(q1, J->k1 + kbase * d, qk_row, J->v + kbase * dvd, v_row, (int64_t)t + 1, d, dvd, scale, p, a1);
        attend_row(q2, J->k2 + kbase * d, qk_row, J->v + kbase * dvd, v_row, (int64_t)t + 1, d, dvd, scale, p, a2);
        double ms = 0.0, xdy = 0.0;
        const double *dout = J->dout + row * dvd;
        for (int c = 0; c < dvd; ++c) {
            x[c] = a1[c] - J->lam_full * a2[c];
            ms += x[c] * x[c];
            xdy += x[c] * (1.0 - J->lam_init) * dout[c];
        }
        ms /= (double)dvd;
        const double r = 1.0 / sqrt(ms + 1e-5);
        double xa2 = 0.0;
        for (int c = 0; c < dvd; ++c) {
            const double dy = (1.0 - J->lam_init) * dout[c];
            dx[c] = r * dy - r * r * r * x[c] * xdy / (double)dvd;
            g2[c] = -J->lam_full * dx[c];
            xa2 += dx[c] * a2[c];
            dlam_abs += fabs(dx[c] * a2[c]);
        }
        dlam -= xa2;
        attend_row_bwd(q1, J->k1 + kbase * d, qk_row, J->v + kbase * dvd, v_row, (int64_t)t + 1, d, dvd, scale,
                       dx, p, dp, J->dq1 + row * d, J->dk1 + kbase * d, J->dvv + kbase * dvd);
        attend_row_bwd(q2, J->k2 + kbase * d, qk_row, J->v + kbase * dvd, v_row, (int64_t)t + 1, d, dvd, scale,
                       g2, p, dp, J->dq2 + row * d, J->dk2 + kbase * d, J->dvv + kbase * dvd);
    }
    J->dlam[slot] = dlam;
    J->dlam_abs[slot] = dlam_abs;
}

/* V2 kv group (b, g): the pairs whose heads read kv head g, every row t. */
static void v2_group_bwd(const bjob_t *J, int64_t u, double *p, double *dp,
                         double *buf)
{
    const int Hkv = J->Hkv, T = J->T, D = J->dqk, G = J->G;
    const int P = J->H, Hq = 2 * P;
    const int g = (int)(u % Hkv);
    const int b = (int)(u / Hkv);
    const int64_t q_row = (int64_t)Hq * D, kv_row = (int64_t)Hkv * D;
    const double scale = 1.0 / sqrt((double)D);
    double *ae = buf, *ao = buf + D, *go = buf + 2 * D;
    const double *k = J->k1 + ((int64_t)b * T * Hkv + g) * D;
    const double *v = J->v + ((int64_t)b * T * Hkv + g) * D;
    double *dk = J->dk1 + ((int64_t)b * T * Hkv + g) * D;
    double *dv = J->dvv + ((int64_t)b * T * Hkv + g) * D;
    for (int i = g * G / 2; i < (g + 1) * G / 2; ++i) {
        const int he = 2 * i, ho = 2 * i + 1;
        for (int t = 0; t < T; ++t) {
            const int64_t tok = (int64_t)b * T + t;
            const double *qe = J->q1 + (tok * Hq + he) * D;
            const double *qo = J->q1 + (tok * Hq + ho) * D;
            const double *dout = J->dout + (tok * P + i) * D;
            attend_row(qe, k, kv_row, v, kv_row, (int64_t)t + 1, D, D, scale, p, ae);
            attend_row(qo, k, kv_row, v, kv_row, (int64_t)t + 1, D, D, scale, p, ao);
            const double sg = 1.0 / (1.0 + exp(-J->lam[tok * P + i]));
            double da = 0.0;
            for (int c = 0; c < D; ++c) {
                go[c] = -sg * dout[c];
                da += dout[c] * ao[c];
            }
            J->dlam[tok * P + i] = -sg * (1.0 - sg) * da;
            attend_row_bwd(qe, k, kv_row, v, kv_row, (int64_t)t + 1, D, D, scale, dout, p, dp,
                           J->dq1 + (tok * Hq + he) * D, dk, dv);
            attend_row_bwd(qo, k, kv_row, v, kv_row, (int64_t)t + 1, D, D, scale, go, p, dp,
                           J->dq1 + (tok * Hq + ho) * D, dk, dv);
        }
    }
    (void)q_row;
}

static void *bwd_worker(void *arg)
{
    const bjob_t *J = (const bjob_t *)arg;
    double *p = (double *)malloc(sizeof(double) * (size_t)J->T * 2);
    double *buf = (double *)malloc(sizeof(double) * (size_t)J->dv * 6);
    if (!p || !buf) {
        free(p);
        free(buf);
        return (void *)1;
    }
    for (int64_t n = J->tid; n < J->nunits; n += J->nthreads) {
        if (J->kind == 1)
            v1_head_bwd(J, J->units[n], n, p, p + J->T, buf);
        else
            v2_group_bwd(J, J->units[n], p, p + J->T, buf);
    }
    free(p);
    free(buf);
    return NULL;
}

static int run_bwd_jobs(const bjob_t *proto, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    bjob_t jobs[256];
    pthread_t th[256];
    int started[256];
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        jobs[i] = *proto;
        jobs[i].tid = i;
        jobs[i].nthreads = nthreads;
        started[i] = pthread_create(&th[i], NULL, bwd_worker, &jobs[i]) == 0;
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

/* DIFF V1 backward.  Inputs as oracle_v1_fwd (contiguous), dout (B,T,H,2d).
 * heads: ids b*H+h to differentiate (NULL = all); gradients are written for
 * those heads only (dq1, dq2, dk1, dk2 (B,T,H,d), dv (B,T,H,2d), zeroed by
 * the caller).  dlam_vec: 4*d doubles (dlq1, dlk1, dlq2, dlk2) from the
 * listed heads' contribution to dL/dlam.  dlam_abs_out: the sum of
 * |dx_c a2_c| behind dL/dlam = -sum dx_c a2_c (the size of the terms that
 * cancel in it, a scale for comparing a rounded result).  Returns 0 on
 * success. */
int oracle_v1_bwd(const double *q1, const double *q2, const double *k1,
                  const double *k2, const double *v, const double *lq1,
                  const double *lk1, const double *lq2, const double *lk2,
                  const double *dout, int B, int T, int H, int d,
                  int layer_index, const int64_t *heads, int64_t nheads,
                  double *dq1, double *dq2, double *dk1, double *dk2,
                  double *dv, double *dlam_vec, double *dlam_abs_out,
                  int nthreads)
{
    bjob_t J;
    memset(&J, 0, sizeof(J));
    J.kind = 1;
    J.q1 = q1; J.q2 = q2; J.k1 = k1; J.k2 = k2; J.v = v; J.dout = dout;
    J.B = B; J.T = T; J.H = H; J.dqk = d; J.dv = 2 * d;
    J.lam_init = oracle_lambda_init(layer_index);
    J.lam_full = oracle_lambda_full(lq1, lk1, lq2, lk2, d, J.lam_init);
    J.dq1 = dq1; J.dq2 = dq2; J.dk1 = dk1; J.dk2 = dk2; J.dvv = dv;
    const int64_t n = heads ? nheads : (int64_t)B * H;
    int64_t *ids = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    double *part = (double *)calloc((size_t)(n > 0 ? n : 1) * 2, sizeof(double));
    if (!ids || !part) {
        free(ids);
        free(part);
        return 3;
    }
    for (int64_t i = 0; i < n; ++i)
        ids[i] = heads ? heads[i] : i;
    J.units = ids; J.nunits = n; J.dlam = part; J.dlam_abs = part + n;
    const int rc = run_bwd_jobs(&J, nthreads);
    double dlam = 0.0, dlam_abs = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        dlam += part[i];
        dlam_abs += part[n + i];
    }
    *dlam_abs_out = dlam_abs;
    double s1 = 0.0, s2 = 0.0;
    for (int c = 0; c < d; ++c) {
        s1 += lq1[c] * lk1[c];
        s2 += lq2[c] * lk2[c];
    }
    for (int c = 0; c < d; ++c) {
        dlam_vec[c] = dlam * exp(s1) * lk1[c];
        dlam_vec[d + c] = dlam * exp(s1) * lq1[c];
        dlam_vec[2 * d + c] = -dlam * exp(s2) * lk2[c];
        dlam_vec[3 * d + c] = -dlam * exp(s2) * lq2[c];
    }
    free(ids);
    free(part);
    return rc;
}

/* DIFF V2 backward.  Inputs as oracle_v2_fwd (contiguous), dout (B,T,Hq/2,D).
 * groups: ids b*Hkv+g (NULL = all); gradients for those kv groups only: dq
 * (B,T,Hq,D) rows of the group's heads, dk, dv (B,T,Hkv,D), dlam (B,T,Hq/2)
 * entries of the group's pairs; all zeroed by the caller. */
int oracle_v2_bwd(const double *q, const double *k, const double *v,
                  const double *lam, const double *dout, int B, int T, int Hq,
                  int Hkv, int D, const int64_t *groups, int64_t ngroups,
                  double *dq, double *dk, double *dv, double *dlam,
                  int nthreads)
{
    if (Hq % Hkv != 0 || ((Hq / Hkv) & 1))
        return 4;
    bjob_t J;
    memset(&J, 0, sizeof(J));
    J.kind = 2;
    J.q1 = q; J.k1 = k; J.v = v; J.lam = lam; J.dout = dout;
    J.B = B; J.T = T; J.H = Hq / 2; J.dqk = D; J.dv = D; J.Hkv = Hkv; J.G = Hq / Hkv;
    J.dq1 = dq; J.dk1 = dk; J.dvv = dv; J.dlam = dlam;
    const int64_t n = groups ? ngroups : (int64_t)B * Hkv;
    int64_t *ids = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!ids)
        return 3;
    for (int64_t i = 0; i < n; ++i)
        ids[i] = groups ? groups[i] : i;
    J.units = ids; J.nunits = n;
    const int rc = run_bwd_jobs(&J, nthreads);
    free(ids);
    return rc;
}

/* ======================================================================
 * Neighbours of the attention call (the prologue).
 *
 * Rotary position embedding as the nanoGPT issue applies it to q and k
 * before the attention (RotaryEmbedding(dim = head_dim) and
 * apply_rotary_pos_emb; the class itself is not printed, so the plainest
 * reading is taken: the rotate-half form with base 10000): for a row of
 * head dim D at position p and each i < D/2, with theta = p * base^(-2i/D),
 *   out[i]       = x[i] cos(theta) - x[i + D/2] sin(theta)
 *   out[i + D/2] = x[i + D/2] cos(theta) + x[i] sin(theta).
 * x: (B, T, H, D) contiguous, positions pos0 + t.
 * ==================================================================== */
void oracle_rope(const double *x, int B, int T, int H, int D, int64_t pos0,
                 double base, double *out)
{
    const int half = D / 2;
    for (int b = 0; b < B; ++b)
        for (int t = 0; t < T; ++t) {
            const double pos = (double)(pos0 + t);
            for (int h = 0; h < H; ++h) {
                const int64_t row = (((int64_t)b * T + t) * H + h) * D;
                for (int i = 0; i < half; ++i) {
                    const double theta = pos * pow(base, -2.0 * (double)i / (double)D);
                    const double c = cos(theta), s = sin(theta);
                    const double x1 = x[row + i], x2 = x[row + i + half];
                    out[row + i] = x1 * c - x2 * s;
                    out[row + i + half] = x2 * c + x1 * s;
                }
            }
        }
}

/* DIFF V2's projected lambda ("a projected lambda for each token and each
 * head"): lam[n, i] = sum_c x[n, c] w[c, i] for every token n; x (N, C),
 * w (C, P), out (N, P). */
void oracle_lambda_proj(const double *x, const double *w, int64_t N, int C,
                        int P, double *out)
{
    for (int64_t n = 0; n < N; ++n)
        for (int i = 0; i < P; ++i) {
            double acc = 0.0;
            for (int c = 0; c < C; ++c)
                acc += x[n * C + c] * w[(int64_t)c * P + i];
            out[n * P + i] = acc;
        }
}
