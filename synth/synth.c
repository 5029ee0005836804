/*
 * synth.c -- seeded synthetic inputs for the verification step.
 *
 * This module only makes inputs: target logits, draft distributions q, draft
 * tokens and uniforms.  It holds none of the verification arithmetic (no
 * accept test, no residual, no inverse-CDF draw); drafts are drawn from q by
 * an exponential race (argmin_i E_i / q_i, E_i ~ Exp(1)), which is exact in
 * distribution and shares nothing with the method's sampler.
 *
 * Random numbers: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11), key = the 64-bit seed, counter =
 * (index lo, index hi, stream id, 0).  One stream per tensor, so a sequence's
 * inputs do not depend on how many sequences or threads are generated.
 *
 * Recipe per sequence b, row j (target logits) and position k (drafts):
 *   z_{j,i}  = fp32(sigma * N(0,1) + bias_i),  bias_i = -zipf_s * ln(i + 1),
 *              rounded to bf16 (nearest, ties to even) when dtype is bf16
 *   top-p (if top_p > 0): keep the smallest set of highest-probability ids
 *              (ties: lower id first) of softmax(z_j / T) whose mass reaches
 *              top_p; set the other logits to -inf
 *   d_{k,i}  = z_{k,i} + draft_sigma * N(0,1);  q_k = softmax(d_k / Tq) in
 *              fp64, restricted to its own top-p nucleus and renormalised if
 *              top_p > 0, stored as fp32
 *   x_k      ~ q_k (the stored fp32 values, as weights), exponential race
 *   one-hot drafts (no q): x_k = argmax_i z_{k,i} (lowest id on ties) with
 *              probability onehot_p, else uniform over [0, V)
 *   u_{b,k}  = (r >> 8) * 2^-24 in [0, 1), k = 0..K (u[K] = final draw)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ST_TARGET = 1, ST_DRAFT_NOISE = 2, ST_DRAFT_RACE = 3, ST_UNIFORM = 4,
       ST_ONEHOT = 5 };

/* ------------------------------------------------------------ Philox4x32-10 */

#define PH_M0 0xD2511F53u
#define PH_M1 0xCD9E8D57u
#define PH_W0 0x9E3779B9u
#define PH_W1 0xBB67AE85u

void synth_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                         uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int r = 0; r < 10; ++r) {
        uint64_t p0 = (uint64_t)PH_M0 * c0;
        uint64_t p1 = (uint64_t)PH_M1 * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        uint32_t n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        uint32_t n3 = (uint32_t)p0;
        c0 = n0;
        c1 = n1;
        c2 = n2;
        c3 = n3;
        k0 += PH_W0;
        k1 += PH_W1;
    }
    out[0] = c0;
    out[1] = c1;
    out[2] = c2;
    out[3] = c3;
}

static void draw(uint64_t seed, uint32_t stream, uint64_t idx, uint32_t out[4])
{
    uint32_t ctr[4] = {(uint32_t)idx, (uint32_t)(idx >> 32), stream, 0u};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    synth_philox4x32_10(ctr, key, out);
}

/* 53-bit uniform in (0, 1] from two words */
static double unit_open0(uint32_t hi, uint32_t lo)
{
    uint64_t m = ((uint64_t)hi << 21) ^ (uint64_t)(lo >> 11);
    return ((double)m + 1.0) * (1.0 / 9007199254740992.0);
}

/* standard normal number `idx` of a stream (Box-Muller, two per counter) */
static double normal_at(uint64_t seed, uint32_t stream, uint64_t idx)
{
    uint32_t w[4];
    draw(seed, stream, idx >> 1, w);
    double u1 = unit_open0(w[0], w[1]);
    double u2 = unit_open0(w[2], w[3]);
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586 * u2;
    return (idx & 1) ? rad * sin(ang) : rad * cos(ang);
}

static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x7FFFFFu))
        return (uint16_t)((b >> 16) | 0x40u); /* quiet NaN */
    uint32_t lsb = (b >> 16) & 1u;
    return (uint16_t)((b + 0x7FFFu + lsb) >> 16);
}

static double bf16_to_f64(uint16_t h)
{
    uint32_t b = (uint32_t)h << 16;
    float f;
    memcpy(&f, &b, 4);
    return (double)f;
}

/* --------------------------------------------------------------- recipe */

typedef struct {
    int dtype;          /* 0 bf16, 1 fp32 */
    int32_t K, V;
    double sigma;       /* target noise std */
    double zipf_s;      /* bias_i = -zipf_s * ln(i+1) */
    double T;           /* target temperature (used for top-p of p) */
    double draft_sigma; /* draft noise std (dense drafts) */
    double Tq;          /* draft temperature; 0 => one-hot drafts, no q */
    double top_p;       /* 0 => none */
    double onehot_p;    /* probability a one-hot draft is the target argmax */
} synth_cfg_t;

typedef struct {
    double v;
    int32_t id;
} pv_t;

static int cmp_desc(const void *a, const void *b)
{
    const pv_t *x = (const pv_t *)a, *y = (const pv_t *)b;
    if (x->v > y->v)
        return -1;
    if (x->v < y->v)
        return 1;
    return (x->id > y->id) - (x->id < y->id);
}

/* Mark the top-p nucleus of probabilities w (V values): keep[i] = 1 for
 * members.  Ties in probability are ordered by lower id first. */
static void nucleus(const double *w, int32_t V, double top_p, pv_t *tmp,
                    unsigned char *keep)
{
    for (int32_t i = 0; i < V; ++i) {
        tmp[i].v = w[i];
        tmp[i].id = i;
        keep[i] = 0;
    }
    qsort(tmp, (size_t)V, sizeof(pv_t), cmp_desc);
    double acc = 0.0;
    for (int32_t r = 0; r < V; ++r) {
        keep[tmp[r].id] = 1;
        acc += tmp[r].v;
        if (acc >= top_p)
            break;
    }
}

static void softmax64(const double *x, int32_t V, double *out)
{
    double m = -INFINITY;
    for (int32_t i = 0; i < V; ++i)
        if (x[i] > m)
            m = x[i];
    double s = 0.0;
    for (int32_t i = 0; i < V; ++i) {
        out[i] = isfinite(x[i]) || x[i] > 0 ? exp(x[i] - m) : 0.0;
        s += out[i];
    }
    for (int32_t i = 0; i < V; ++i)
        out[i] /= s;
}

typedef struct {
    const synth_cfg_t *c;
    uint64_t seed;
    int64_t b0;           /* global index of the first sequence generated */
    int64_t nb;
    void *logits;
    float *q;
    int32_t *tokens;
    float *u;
    int64_t r0, r1;       /* range of local sequences for this thread */
    int failed;
} job_t;

static void *run(void *arg)
{
    job_t *J = (job_t *)arg;
    const synth_cfg_t *c = J->c;
    int32_t K = c->K, V = c->V;
    double *zr = (double *)malloc(sizeof(double) * (size_t)V);
    double *zu = (double *)malloc(sizeof(double) * (size_t)V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    pv_t *tmp = (pv_t *)malloc(sizeof(pv_t) * (size_t)V);
    unsigned char *keep = (unsigned char *)malloc((size_t)V);
    if (!zr || !zu || !w || !tmp || !keep) {
        J->failed = 1;
        goto done;
    }
    for (int64_t lb = J->r0; lb < J->r1; ++lb) {
        int64_t gb = J->b0 + lb; /* global sequence index */
        for (int32_t j = 0; j <= K; ++j) {
            int64_t grow = gb * (K + 1) + j;
            int64_t lrow = lb * (K + 1) + j;
            for (int32_t i = 0; i < V; ++i) {
                double n = normal_at(J->seed, ST_TARGET,
                                     (uint64_t)(grow * (int64_t)V + i));
                float f = (float)(c->sigma * n - c->zipf_s * log((double)i + 1.0));
                if (c->dtype == 0) {
                    uint16_t h = f32_to_bf16_rne(f);
                    ((uint16_t *)J->logits)[lrow * V + i] = h;
                    zr[i] = bf16_to_f64(h);
                } else {
                    ((float *)J->logits)[lrow * V + i] = f;
                    zr[i] = (double)f;
                }
                zu[i] = zr[i];
            }
            if (c->top_p > 0.0) {
                for (int32_t i = 0; i < V; ++i)
                    w[i] = zr[i] / c->T;
                softmax64(w, V, w);
                nucleus(w, V, c->top_p, tmp, keep);
                for (int32_t i = 0; i < V; ++i) {
                    if (keep[i])
                        continue;
                    zr[i] = -INFINITY;
                    if (c->dtype == 0)
                        ((uint16_t *)J->logits)[lrow * V + i] = 0xFF80u;
                    else
                        ((float *)J->logits)[lrow * V + i] = -INFINITY;
                }
            }
            if (j == K)
                continue;
            /* draft position k = j */
            int64_t gpos = gb * K + j, lpos = lb * K + j;
            if (c->Tq > 0.0) {
                for (int32_t i = 0; i < V; ++i) {
                    double n = normal_at(J->seed, ST_DRAFT_NOISE,
                                         (uint64_t)(gpos * (int64_t)V + i));
                    /* the draft sees the unmasked target logits */
                    double zt = zu[i];
                    w[i] = (zt + c->draft_sigma * n) / c->Tq;
                }
                softmax64(w, V, w);
                if (c->top_p > 0.0) {
                    nucleus(w, V, c->top_p, tmp, keep);
                    double s = 0.0;
                    for (int32_t i = 0; i < V; ++i)
                        if (keep[i])
                            s += w[i];
                    for (int32_t i = 0; i < V; ++i)
                        w[i] = keep[i] ? w[i] / s : 0.0;
                }
                float *qrow = J->q + lpos * V;
                for (int32_t i = 0; i < V; ++i)
                    qrow[i] = (float)w[i];
                /* exponential race on the stored weights */
                double best = INFINITY;
                int32_t arg = -1;
                for (int32_t i = 0; i < V; ++i) {
                    if (!(qrow[i] > 0.0f))
                        continue;
                    uint32_t r[4];
                    draw(J->seed, ST_DRAFT_RACE,
                         (uint64_t)(gpos * (int64_t)V + i), r);
                    double e = -log(unit_open0(r[0], r[1]));
                    double key = e / (double)qrow[i];
                    if (key < best) {
                        best = key;
                        arg = i;
                    }
                }
                J->tokens[lpos] = arg;
            } else {
                uint32_t r[4];
                draw(J->seed, ST_ONEHOT, (uint64_t)gpos, r);
                double coin = unit_open0(r[0], r[1]);
                if (coin <= c->onehot_p) {
                    int32_t arg = 0;
                    for (int32_t i = 1; i < V; ++i)
                        if (zu[i] > zu[arg])
                            arg = i;
                    J->tokens[lpos] = arg;
                } else {
                    J->tokens[lpos] =
                        (int32_t)(((uint64_t)r[2] * (uint64_t)V) >> 32);
                }
            }
        }
        for (int32_t k = 0; k <= K; ++k) {
            uint32_t r[4];
            draw(J->seed, ST_UNIFORM, (uint64_t)(gb * (K + 1) + k), r);
            J->u[lb * (K + 1) + k] = (float)(r[0] >> 8) * (1.0f / 16777216.0f);
        }
    }
done:
    free(zr);
    free(zu);
    free(w);
    free(tmp);
    free(keep);
    return NULL;
}

/* Generate sequences [b0, b0 + nb) of the global stream for `seed`.
 * logits: [nb, K+1, V] uint16 (bf16) or fp32; q: [nb, K, V] fp32 (ignored and
 * may be NULL for one-hot drafts); tokens: [nb, K]; u: [nb, K+1].
 * Returns 0 on success. */
int synth_generate(const synth_cfg_t *c, uint64_t seed, int64_t b0,
                   int64_t nb, void *logits, float *q, int32_t *tokens,
                   float *u, int nthreads)
{
    if (!c || !logits || !tokens || !u || c->K < 0 || c->V < 1 || nb < 0 ||
        (c->Tq > 0.0 && c->K > 0 && !q) || !(c->T > 0.0))
        return -1;
    if (nb == 0)
        return 0;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > nb)
        nthreads = (int)nb;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        job_t J = {c, seed, b0, nb, logits, q, tokens, u,
                   nb * t / nthreads, nb * (t + 1) / nthreads, 0};
        jobs[t] = J;
    }
    int *started = (int *)calloc((size_t)nthreads, sizeof(int));
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&th[t], NULL, run, &jobs[t]) == 0;
    run(&jobs[0]);
    int rc = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (started[t])
            pthread_join(th[t], NULL);
        else
            run(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].failed)
            rc = -1;
    free(started);
    free(jobs);
    free(th);
    return rc;
}

/* bf16 rounding exposed for the generator's own tests */
void synth_f32_to_bf16(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = f32_to_bf16_rne(in[i]);
}
