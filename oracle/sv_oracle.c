/*
 * sv_oracle.c -- plain fp64 CPU oracle for the speculative-sampling
 * verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * constant with the CUDA library; the two are compared on the same seeded
 * inputs.  It is deliberately slow and literal: every sum runs sequentially
 * in token-id order, nothing is blocked, fused or reordered.
 *
 * What it computes, and where each step is defined:
 *
 *  (1) p_j = softmax(z_j / T) for every one of the K+1 target rows.
 *      "推测解码采样验证优化策略 —— 深度调研报告", part 1 section 4
 *      (实现逻辑, verify(): softmax of target_logits / temperature), and
 *      "推测解码：草稿、验证与实际加速", section 接受与拒绝怎样保住分布
 *      (p already carries the temperature; q arrives already processed).
 *  (2) Row j verifies draft x_{j+1}; row K is only used for the extra token.
 *      "推测解码：草稿、验证与实际加速", section 候选已知，验证才能并行
 *      (the equation listing p_1 .. p_4 and the offset between logits and
 *      candidates).
 *  (3) Accept draft x with probability a(x) = min(1, p(x)/q(x)), tested
 *      left to right as  u_k < a(x_k).
 *      Same page, section 接受与拒绝怎样保住分布 (equation for a(x)) and
 *      section 算完三个 token 的全部概率 (the replay accepts when the draw is
 *      strictly below the threshold).
 *  (4) At the first rejection, emit one token drawn from
 *      r(x) = max(0, p(x) - q(x)) / sum_y max(0, p(y) - q(y)); later drafts are
 *      discarded.  If every draft is accepted, emit one extra token from
 *      p_{K+1}.  Same page, sections 接受与拒绝怎样保住分布 (equation for r(x))
 *      and 候选已知，验证才能并行; "投机采样", section 机制：起草-验证-接受
 *      (n in [1, gamma+1]).
 *  (5) Drawing from a distribution w with a uniform u: walk the token ids in
 *      ascending order and return the first id whose cumulative mass exceeds
 *      u * sum(w).  "推测解码：草稿、验证与实际加速", section
 *      算完三个 token 的全部概率 (the sampler of the replay, which uses the
 *      final draw for the correction or the extra token).
 *  (6) A deterministic draft (n-gram / prompt lookup) is the case
 *      q = delta_x: then a(x) = min(1, p(x)) and r is p with x removed.
 *      Follows from (3)-(4) with q one-hot ("推测解码采样验证优化策略", part 1
 *      section 1 on prompt lookup; "投机采样", 变体谱系 table, N-gram row).
 *
 * Readings taken where the pages are silent or disagree (also listed in the
 * design notes):
 *  - the accept test is  u < a  (one page writes <=, the replay uses <);
 *  - the correction / extra token always uses the final uniform u[K];
 *  - if rounding leaves no id with t < C(i), the last id of positive mass is
 *    returned;
 *  - if the residual mass is not positive after a rejection (impossible in
 *    exact arithmetic) the token is drawn from p and a status bit is set;
 *  - a sequence with an invalid input (u outside [0,1), token outside [0,V),
 *    q(x) <= 0 or non-finite, a logit row with NaN/+inf or no finite entry)
 *    emits nothing: num_emitted = 0, tokens and flags -1, probabilities 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Per-sequence status bits reported by the oracle. */
enum {
    ORC_BAD_U = 1,
    ORC_BAD_TOKEN = 2,
    ORC_BAD_Q = 4,
    ORC_BAD_ROW = 8,
    ORC_DEGENERATE_RESIDUAL = 16
};

/* ---------------------------------------------------------------- helpers */

static double bf16_bits_to_double(uint16_t h)
{
    uint32_t bits = (uint32_t)h << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double logit_at(const void *logits, int dtype, int64_t idx)
{
    if (dtype == 0)
        return bf16_bits_to_double(((const uint16_t *)logits)[idx]);
    return (double)((const float *)logits)[idx];
}

/* Step (1): p = softmax(z / T) over one row.  Returns 0 if the row has a
 * NaN or +inf entry or no finite entry (then p is left undefined). */
static int softmax_row(const void *logits, int dtype, int64_t row_off,
                       int32_t V, double T, double *p)
{
    double m = -INFINITY;
    for (int32_t i = 0; i < V; ++i) {
        double z = logit_at(logits, dtype, row_off + i);
        if (isnan(z) || (isinf(z) && z > 0))
            return 0;
        double zt = z / T;
        if (zt > m)
            m = zt;
    }
    if (!isfinite(m))
        return 0;
    double s = 0.0;
    for (int32_t i = 0; i < V; ++i) {
        double zt = logit_at(logits, dtype, row_off + i) / T;
        p[i] = exp(zt - m); /* exp(-inf) = 0 for masked entries */
        s += p[i];
    }
    for (int32_t i = 0; i < V; ++i)
        p[i] /= s;
    return 1;
}

/* Step (5): first id (ascending) with t < C(i), t = u * sum(w).  If rounding
 * leaves none, the last id with positive mass.  *Z_out receives sum(w). */
static int32_t inverse_cdf(const double *w, int32_t V, double u, double *Z_out)
{
    double Z = 0.0;
    for (int32_t i = 0; i < V; ++i)
        Z += w[i];
    *Z_out = Z;
    double t = u * Z;
    double C = 0.0;
    for (int32_t i = 0; i < V; ++i) {
        C += w[i];
        if (t < C)
            return i;
    }
    for (int32_t i = V - 1; i >= 0; --i)
        if (w[i] > 0.0)
            return i;
    return 0;
}

/* The distribution the final token is drawn from at survivor row j.
 * rejected: r = max(0, p - q) (q one-hot on x when Q is NULL);
 * bonus:    r = p. */
static void survivor_weights(const double *p, const double *q, int onehot,
                             int32_t x, int rejected, int32_t V, double *w)
{
    for (int32_t i = 0; i < V; ++i) {
        if (!rejected) {
            w[i] = p[i];
        } else {
            double qi = onehot ? (i == x ? 1.0 : 0.0) : q[i];
            double d = p[i] - qi;
            w[i] = d > 0.0 ? d : 0.0;
        }
    }
}

/* ------------------------------------------------- one sequence, probs in */

typedef struct {
    int32_t *out_tokens;   /* [K+1] */
    int32_t *num_emitted;  /* [1]   */
    int8_t *accept_flags;  /* [K]   */
    double *accept_prob;   /* [K]   */
    double *residual_mass; /* [1]   */
    int32_t *status;       /* [1]   */
} seq_out_t;

/* P: K+1 rows of p (fp64); Q: K rows of q or NULL (one-hot drafts);
 * rows_ok: validity of each of the K+1 rows (NULL = all valid). */
static void verify_sequence(const double *P, const double *Q,
                            const int32_t *tok, const double *u,
                            const int *rows_ok, int32_t K, int32_t V,
                            double *w_scratch, seq_out_t o)
{
    int32_t st = 0;
    for (int32_t k = 0; k <= K; ++k)
        if (!(u[k] >= 0.0 && u[k] < 1.0))
            st |= ORC_BAD_U;
    for (int32_t k = 0; k < K; ++k) {
        if (tok[k] < 0 || tok[k] >= V) {
            st |= ORC_BAD_TOKEN;
        } else if (Q) {
            double qx = Q[(int64_t)k * V + tok[k]];
            if (!(qx > 0.0) || !isfinite(qx))
                st |= ORC_BAD_Q;
        }
    }
    if (rows_ok)
        for (int32_t j = 0; j <= K; ++j)
            if (!rows_ok[j])
                st |= ORC_BAD_ROW;

    for (int32_t k = 0; k <= K; ++k)
        o.out_tokens[k] = -1;
    for (int32_t k = 0; k < K; ++k) {
        o.accept_flags[k] = -1;
        o.accept_prob[k] = 0.0;
    }
    *o.residual_mass = 0.0;
    *o.num_emitted = 0;
    if (st) {
        *o.status = st;
        return;
    }

    /* accept probability of every draft (also of those never reached) */
    for (int32_t k = 0; k < K; ++k) {
        double px = P[(int64_t)k * V + tok[k]];
        double qx = Q ? Q[(int64_t)k * V + tok[k]] : 1.0;
        double a = px / qx;
        o.accept_prob[k] = a < 1.0 ? a : 1.0;
    }

    /* steps (3)-(4): left to right, stop at the first rejection */
    int32_t jstar = K;
    for (int32_t k = 0; k < K; ++k) {
        if (u[k] < o.accept_prob[k]) {
            o.out_tokens[k] = tok[k];
            o.accept_flags[k] = 1;
        } else {
            o.accept_flags[k] = 0;
            jstar = k;
            break;
        }
    }

    int rejected = jstar < K;
    const double *prow = P + (int64_t)jstar * V;
    survivor_weights(prow, rejected && Q ? Q + (int64_t)jstar * V : NULL,
                     rejected && !Q, rejected ? tok[jstar] : -1, rejected, V,
                     w_scratch);
    double Z;
    int32_t y = inverse_cdf(w_scratch, V, u[K], &Z);
    if (rejected && !(Z > 0.0)) {
        st |= ORC_DEGENERATE_RESIDUAL;
        double Zp;
        y = inverse_cdf(prow, V, u[K], &Zp);
    }
    o.out_tokens[jstar] = y;
    *o.residual_mass = rejected ? Z : 0.0;
    *o.num_emitted = jstar + 1;
    *o.status = st;
}

/* --------------------------------------------------------- thread fan-out */

typedef struct {
    /* common inputs */
    const void *logits;
    int dtype;
    const float *qf;
    const double *pd, *qd, *ud;
    const int32_t *tokens;
    const float *uf;
    double T;
    int64_t B;
    int32_t K, V;
    /* outputs */
    int32_t *out_tokens, *num_emitted, *status;
    int8_t *accept_flags;
    double *accept_prob, *residual_mass;
    /* work split */
    int64_t b0, b1;
    int from_logits;
    int failed;
} job_t;

static seq_out_t outputs_of(const job_t *J, int64_t b)
{
    seq_out_t o;
    o.out_tokens = J->out_tokens + b * (J->K + 1);
    o.num_emitted = J->num_emitted + b;
    o.accept_flags = J->accept_flags + b * J->K;
    o.accept_prob = J->accept_prob + b * J->K;
    o.residual_mass = J->residual_mass + b;
    o.status = J->status + b;
    return o;
}

static void *run_job(void *arg)
{
    job_t *J = (job_t *)arg;
    int32_t K = J->K, V = J->V;
    double *P = NULL, *Q = NULL, *w = NULL, *u = NULL;
    int *ok = NULL;
    w = (double *)malloc(sizeof(double) * (size_t)V);
    u = (double *)malloc(sizeof(double) * (size_t)(K + 1));
    ok = (int *)malloc(sizeof(int) * (size_t)(K + 1));
    if (J->from_logits) {
        P = (double *)malloc(sizeof(double) * (size_t)(K + 1) * (size_t)V);
        if (J->qf && K > 0)
            Q = (double *)malloc(sizeof(double) * (size_t)K * (size_t)V);
    }
    if (!w || !u || !ok || (J->from_logits && !P) ||
        (J->from_logits && J->qf && K > 0 && !Q)) {
        J->failed = 1;
        goto done;
    }
    for (int64_t b = J->b0; b < J->b1; ++b) {
        const int32_t *tok = J->tokens + b * K;
        if (J->from_logits) {
            for (int32_t j = 0; j <= K; ++j)
                ok[j] = softmax_row(J->logits, J->dtype,
                                    (b * (K + 1) + j) * (int64_t)V, V, J->T,
                                    P + (int64_t)j * V);
            if (Q)
                for (int64_t e = 0; e < (int64_t)K * V; ++e)
                    Q[e] = (double)J->qf[b * K * (int64_t)V + e];
            for (int32_t k = 0; k <= K; ++k)
                u[k] = (double)J->uf[b * (K + 1) + k];
            verify_sequence(P, J->qf ? Q : NULL, tok, u, ok, K, V, w,
                            outputs_of(J, b));
        } else {
            const double *Pb = J->pd + b * (K + 1) * (int64_t)V;
            const double *Qb = J->qd ? J->qd + b * K * (int64_t)V : NULL;
            verify_sequence(Pb, Qb, tok, J->ud + b * (K + 1), NULL, K, V, w,
                            outputs_of(J, b));
        }
    }
done:
    free(P);
    free(Q);
    free(w);
    free(u);
    free(ok);
    return NULL;
}

static int fan_out(job_t proto, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if ((int64_t)nthreads > proto.B)
        nthreads = (int)(proto.B > 0 ? proto.B : 1);
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].b0 = proto.B * t / nthreads;
        jobs[t].b1 = proto.B * (t + 1) / nthreads;
    }
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, run_job, &jobs[t]) != 0)
            jobs[t].failed = 2; /* run it inline below instead */
    run_job(&jobs[0]);
    int rc = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (jobs[t].failed == 2) {
            jobs[t].failed = 0;
            run_job(&jobs[t]);
        } else {
            pthread_join(th[t], NULL);
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].failed)
            rc = -1;
    free(jobs);
    free(th);
    return rc;
}

/* ------------------------------------------------------------ entry points */

/* Verification from target logits.
 * logits: [B, K+1, V], dtype 0 = bf16 bit patterns (uint16), 1 = fp32.
 * q: [B, K, V] fp32, or NULL for one-hot drafts.  tokens: [B, K] int32.
 * u: [B, K+1] fp32, u[:, K] is the final draw.  T > 0.
 * Outputs (host): out_tokens [B, K+1], num_emitted [B], accept_flags [B, K],
 * accept_prob [B, K] fp64, residual_mass [B] fp64, status [B].
 * Returns 0, or -1 on bad arguments / allocation failure. */
int sv_oracle_verify(const void *logits, int dtype, const float *q,
                     const int32_t *tokens, const float *u, double T,
                     int64_t B, int32_t K, int32_t V, int32_t *out_tokens,
                     int32_t *num_emitted, int8_t *accept_flags,
                     double *accept_prob, double *residual_mass,
                     int32_t *status, int nthreads)
{
    if (!logits || !tokens || !u || !out_tokens || !num_emitted ||
        !accept_flags || !accept_prob || !residual_mass || !status)
        return -1;
    if (B < 0 || K < 0 || V < 1 || !(T > 0.0) || !isfinite(T) ||
        (dtype != 0 && dtype != 1))
        return -1;
    job_t J;
    memset(&J, 0, sizeof J);
    J.logits = logits;
    J.dtype = dtype;
    J.qf = q;
    J.tokens = tokens;
    J.uf = u;
    J.T = T;
    J.B = B;
    J.K = K;
    J.V = V;
    J.out_tokens = out_tokens;
    J.num_emitted = num_emitted;
    J.accept_flags = accept_flags;
    J.accept_prob = accept_prob;
    J.residual_mass = residual_mass;
    J.status = status;
    J.from_logits = 1;
    if (B == 0)
        return 0;
    return fan_out(J, nthreads);
}

/* Verification from probabilities given directly (fp64): p [B, K+1, V],
 * q [B, K, V] or NULL (one-hot), u [B, K+1] fp64.  Same outputs. */
int sv_oracle_verify_probs(const double *p, const double *q,
                           const int32_t *tokens, const double *u, int64_t B,
                           int32_t K, int32_t V, int32_t *out_tokens,
                           int32_t *num_emitted, int8_t *accept_flags,
                           double *accept_prob, double *residual_mass,
                           int32_t *status, int nthreads)
{
    if (!p || !tokens || !u || !out_tokens || !num_emitted || !accept_flags ||
        !accept_prob || !residual_mass || !status)
        return -1;
    if (B < 0 || K < 0 || V < 1)
        return -1;
    job_t J;
    memset(&J, 0, sizeof J);
    J.pd = p;
    J.qd = q;
    J.ud = u;
    J.tokens = tokens;
    J.B = B;
    J.K = K;
    J.V = V;
    J.out_tokens = out_tokens;
    J.num_emitted = num_emitted;
    J.accept_flags = accept_flags;
    J.accept_prob = accept_prob;
    J.residual_mass = residual_mass;
    J.status = status;
    J.from_logits = 0;
    if (B == 0)
        return 0;
    return fan_out(J, nthreads);
}

/* Diagnostics for one sequence b of a logits input: the softmax of row j
 * (p_out, V values) and the normalised distribution the final token would be
 * drawn from at row j (w_out, V values): the residual when `rejected` is 1,
 * p itself otherwise, each divided by its own sum; cdf_out (V values) is the
 * running sum of w_out taken in id order.  Any output pointer may be NULL.
 * Returns the unnormalised mass sum(w), or -1 if the row is invalid. */
double sv_oracle_row_dists(const void *logits, int dtype, const float *q,
                           const int32_t *tokens, double T, int64_t b,
                           int32_t K, int32_t V, int32_t j, int rejected,
                           double *p_out, double *w_out, double *cdf_out)
{
    if (!logits || !tokens || V < 1 || K < 0 || j < 0 || j > K ||
        (rejected && j >= K) || !(T > 0.0))
        return -1.0;
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    double *qr = NULL;
    double Z = -1.0;
    if (!p || !w)
        goto out;
    if (!softmax_row(logits, dtype, (b * (K + 1) + j) * (int64_t)V, V, T, p))
        goto out;
    if (rejected && q) {
        qr = (double *)malloc(sizeof(double) * (size_t)V);
        if (!qr)
            goto out;
        for (int32_t i = 0; i < V; ++i)
            qr[i] = (double)q[(b * K + j) * (int64_t)V + i];
    }
    int32_t x = rejected ? tokens[b * K + j] : -1;
    survivor_weights(p, qr, rejected && !q, x, rejected, V, w);
    Z = 0.0;
    for (int32_t i = 0; i < V; ++i)
        Z += w[i];
    {
        double C = 0.0;
        for (int32_t i = 0; i < V; ++i) {
            C += w[i];
            if (p_out)
                p_out[i] = p[i];
            if (w_out)
                w_out[i] = Z > 0.0 ? w[i] / Z : 0.0;
            if (cdf_out)
                cdf_out[i] = Z > 0.0 ? C / Z : 0.0;
        }
    }
out:
    free(p);
    free(w);
    free(qr);
    return Z;
}

/* ------------------------------------------------ top-k / top-p filtering
 *
 * (7) The target distribution p carries the target's own sampling
 *     processing -- temperature, top-k, top-p -- before any accept test, and
 *     q must match what the draft actually used ("推测解码：草稿、验证与实际加速",
 *     section 接受与拒绝怎样保住分布).  The pages name these steps but define
 *     neither top-k nor top-p; the reading taken here:
 *       - order the ids by p = softmax(z / T) descending, equal p by
 *         ascending id (ids with a -inf logit have p = 0 and are never kept);
 *       - top-k (k >= 1): keep the first min(k, #finite) ids of that order;
 *         k <= 0 keeps every finite id;
 *       - top-p (0 < top_p < 1): of those, keep the shortest prefix whose
 *         mass reaches top_p times the mass of the top-k set (the id that
 *         crosses the threshold is kept); top_p >= 1 keeps the top-k set
 *         (top_p <= 0 or NaN is rejected);
 *       - every other logit becomes -inf and kept logits are copied
 *         unchanged, so softmax(z' / T) is the renormalised filtered p.
 *     Masses are fp64 exp(z/T - max) summed sequentially in that order.
 */

typedef struct {
    double z;   /* logit (the order of z/T, T > 0) */
    int32_t id;
} ranked_t;

static int ranked_cmp(const void *a, const void *b)
{
    const ranked_t *x = (const ranked_t *)a, *y = (const ranked_t *)b;
    if (x->z > y->z)
        return -1;
    if (x->z < y->z)
        return 1;
    return (x->id > y->id) - (x->id < y->id);
}

/* One row: the finite ids in filter order (rank[0..n)), their cumulative
 * masses cum[0..n) (unnormalised, exp(z/T - max)), the top-k count and the
 * top-p target mass.  Returns the number of finite ids, -1 for a bad row
 * (NaN, +inf or no finite logit). */
static int32_t filter_rank_row(const void *logits, int dtype, int64_t off, int32_t V, double T,
                               int32_t top_k, double top_p, ranked_t *rank, double *cum,
                               int32_t *n_topk, double *tau)
{
    int32_t n = 0;
    double m = -INFINITY;
    for (int32_t i = 0; i < V; ++i) {
        double z = logit_at(logits, dtype, off + i);
        if (isnan(z) || (isinf(z) && z > 0))
            return -1;
        if (isinf(z))
            continue;
        rank[n].z = z;
        rank[n].id = i;
        ++n;
        if (z / T > m)
            m = z / T;
    }
    if (n == 0)
        return -1;
    qsort(rank, (size_t)n, sizeof(ranked_t), ranked_cmp);
    double acc = 0.0;
    for (int32_t r = 0; r < n; ++r) {
        acc += exp(rank[r].z / T - m);
        cum[r] = acc;
    }
    const int32_t nk = (top_k >= 1 && top_k < n) ? top_k : n;
    *n_topk = nk;
    *tau = (top_p > 0.0 && top_p < 1.0) ? top_p * cum[nk - 1] : cum[nk - 1];
    return n;
}

/* How many ids of the order are kept: the shortest prefix (within the
 * top-k count) whose cumulative mass reaches tau. */
static int32_t filter_kept(const double *cum, int32_t nk, double tau)
{
    int32_t r = 0;
    while (r < nk - 1 && cum[r] < tau)
        ++r;
    return r + 1;
}

typedef struct {
    const void *logits;
    int dtype;
    int32_t V;
    double T, top_p;
    int32_t top_k;
    void *out;
    int32_t *kept;
    int32_t *status;
    int64_t r0, r1;
    int failed;
} filter_job_t;

static void *filter_job(void *arg)
{
    filter_job_t *J = (filter_job_t *)arg;
    const int32_t V = J->V;
    ranked_t *rank = (ranked_t *)malloc((size_t)V * sizeof(ranked_t));
    double *cum = (double *)malloc((size_t)V * sizeof(double));
    if (!rank || !cum) {
        J->failed = 1;
        free(rank);
        free(cum);
        return NULL;
    }
    for (int64_t row = J->r0; row < J->r1; ++row) {
        const int64_t off = row * (int64_t)V;
        int32_t nk = 0;
        double tau = 0.0;
        const int32_t n = filter_rank_row(J->logits, J->dtype, off, V, J->T, J->top_k, J->top_p,
                                          rank, cum, &nk, &tau);
        /* copy the row; then mask what is not kept */
        if (J->dtype == 0)
            memcpy((uint16_t *)J->out + off, (const uint16_t *)J->logits + off, (size_t)V * 2);
        else
            memcpy((float *)J->out + off, (const float *)J->logits + off, (size_t)V * 4);
        if (n < 0) {
            J->kept[row] = 0;
            J->status[row] = ORC_BAD_ROW;
            continue;
        }
        const int32_t kept = (J->top_p < 1.0) ? filter_kept(cum, nk, tau) : nk;
        for (int32_t r = kept; r < n; ++r) {
            const int32_t i = rank[r].id;
            if (J->dtype == 0)
                ((uint16_t *)J->out)[off + i] = 0xFF80u; /* bf16 -inf */
            else
                ((float *)J->out)[off + i] = -INFINITY;
        }
        J->kept[row] = kept;
        J->status[row] = 0;
    }
    free(rank);
    free(cum);
    return NULL;
}

/* Filter `rows` logit rows of V entries (dtype 0 = bf16 bits, 1 = fp32) at
 * temperature T with top_k / top_p as in (7).  out: the filtered rows, same
 * dtype; kept[row]: ids kept (0 for a bad row); status[row]: ORC_BAD_ROW for
 * a row with NaN, +inf or no finite logit (copied unchanged).  Returns 0. */
int sv_oracle_filter_logits(const void *logits, int dtype, int64_t rows, int32_t V, double T,
                            int32_t top_k, double top_p, void *out, int32_t *kept,
                            int32_t *status, int nthreads)
{
    if (!logits || !out || !kept || !status || rows < 0 || V < 1 || !(T > 0.0) || !(top_p > 0.0))
        return -1;
    if (nthreads < 1)
        nthreads = 1;
    if ((int64_t)nthreads > rows)
        nthreads = (int)(rows > 0 ? rows : 1);
    filter_job_t *jobs = (filter_job_t *)calloc((size_t)nthreads, sizeof(filter_job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    for (int t = 0; t < nthreads; ++t) {
        filter_job_t J = {logits, dtype, V, T, top_p, top_k, out, kept, status,
                          rows * t / nthreads, rows * (t + 1) / nthreads, 0};
        jobs[t] = J;
    }
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, filter_job, &jobs[t]) != 0)
            jobs[t].failed = 2;
    filter_job(&jobs[0]);
    int rc = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (jobs[t].failed == 2) {
            jobs[t].failed = 0;
            filter_job(&jobs[t]);
        } else {
            pthread_join(th[t], NULL);
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].failed)
            rc = -1;
    free(jobs);
    free(th);
    return rc;
}

/* One row's filter order for parity checks: the finite ids in order
 * (ids[0..n)), the cumulative masses of that order (cum[0..n)), the top-k
 * count and the top-p target mass.  Returns n, or -1 for a bad row. */
int32_t sv_oracle_filter_order(const void *logits, int dtype, int64_t row, int32_t V, double T,
                               int32_t top_k, double top_p, int32_t *ids, double *cum,
                               int32_t *n_topk, double *tau)
{
    ranked_t *rank = (ranked_t *)malloc((size_t)V * sizeof(ranked_t));
    if (!rank)
        return -1;
    const int32_t n = filter_rank_row(logits, dtype, row * (int64_t)V, V, T, top_k, top_p, rank, cum,
                                      n_topk, tau);
    for (int32_t r = 0; r < n; ++r)
        ids[r] = rank[r].id;
    free(rank);
    return n;
}

/* ------------------------------------------------------------------ */
/* The target's LM head, for the fused LM-head path: logits = h W^T.
 * "推测解码采样验证优化策略 —— 深度调研报告", part 1 section 6 (扩展性与安全性)
 * names fusing the verification into the target's last layer; the layer
 * itself is the plain product of the last hidden states h [M, d] with the
 * output embedding W [V, d].  Each entry is summed in fp64, sequentially in
 * k, from the bf16 inputs (every bf16 value and every product of two is
 * exact in fp64). */

double sv_oracle_lm_head_entry(const uint16_t *h, const uint16_t *W, int32_t d, int64_t row, int64_t col)
{
    double s = 0.0;
    for (int32_t k = 0; k < d; ++k)
        s += bf16_bits_to_double(h[row * d + k]) * bf16_bits_to_double(W[col * d + k]);
    return s;
}

int sv_oracle_lm_head(const uint16_t *h, const uint16_t *W, int64_t M, int32_t d, int32_t V, double *out)
{
    if (M < 0 || d < 1 || V < 1 || (M > 0 && (!h || !W || !out)))
        return 1;
    for (int64_t i = 0; i < M; ++i)
        for (int32_t v = 0; v < V; ++v)
            out[i * V + v] = sv_oracle_lm_head_entry(h, W, d, i, v);
    return 0;
}

/* fp64 -> bf16 bits, rounded once to the nearest representable value, ties
 * to the even significand (bf16: 8 significant bits).  Finite inputs below
 * the bf16 overflow threshold only (logits). */
void sv_oracle_bf16_round(const double *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) {
        const double v = x[i];
        if (v == 0.0) {
            out[i] = signbit(v) ? 0x8000u : 0u;
            continue;
        }
        int e;
        const double m = frexp(v, &e);              /* v = m 2^e, 0.5 <= |m| < 1 */
        const double r = nearbyint(ldexp(m, 8));    /* 8 significant bits, ties to even */
        const float f = (float)ldexp(r, e - 8);     /* exact: r has 8 bits */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        out[i] = (uint16_t)(u >> 16);               /* exact: the low 16 bits are zero */
    }
}

/* ------------------------------------------------ tree (multi-candidate)
 *
 * Verification of a candidate tree by multi-step speculative sampling
 * (SpecInfer, Miao et al., "SpecInfer: Accelerating Large Language Model
 * Serving with Tree-based Speculative Inference and Verification", ASPLOS
 * 2024, the multi-step speculative sampling of its verification section).
 * The pages fix what a tree must satisfy -- it commits one contiguous path
 * and keeps the target distribution, and the chain's single-candidate
 * correction cannot be applied to it as it stands ("推测解码：草稿、验证与
 * 实际加速", section 链、树与自推测) -- but give no rule; this is the
 * published rule taken for it.
 *
 * Nodes 0..N-1 of one sequence; node 0 is the committed prefix (no token),
 * parent[i] < i for i >= 1, and the children of a node are its nodes in
 * increasing index order, drafted i.i.d. from that node's draft
 * distribution q_v.  p_v = softmax(z_v / T) is the target's next-token
 * distribution after node v's path.  From v = 0:
 *   r = p_v; for each child c of v in order: accept c (token x) iff
 *   u[c] < min(1, r(x) / q_v(x)); on acceptance commit x and continue at c;
 *   on rejection r = max(0, r - q_v) / sum(max(0, r - q_v)).
 *   If every child is rejected, draw the final token from r with u[0]; if v
 *   has no children, draw it from p_v with u[0] (the draw as in step (5)).
 * Readings: the acceptance uniform of node c is u[c] and the final draw
 * uses u[0]; a residual with no positive mass (impossible in exact
 * arithmetic) ends the walk with the final token drawn from p_v and a
 * status bit; a sequence with an invalid input (parent outside [0, i) for
 * node i >= 1, a token outside [0, V), q_v(x) <= 0 or non-finite for a
 * drafted token x, u outside [0, 1), a bad logit row) emits nothing.
 */
enum { ORC_BAD_TREE = 64 };

/* P, Q: N rows of p and q (fp64); rows_ok: validity of each row (NULL =
 * all valid).  out_tokens / out_nodes: [N]; accept_prob: [N] (-1 where the
 * node was not tested). */
static void tree_sequence(const double *P, const double *Q, const int32_t *parent,
                          const int32_t *tok, const double *u, const int *rows_ok,
                          int32_t N, int32_t V, double *r, double *w,
                          int32_t *out_tokens, int32_t *out_nodes, int32_t *num_emitted,
                          double *accept_prob, int32_t *status)
{
    int32_t st = 0;
    for (int32_t i = 0; i < N; ++i)
        if (!(u[i] >= 0.0 && u[i] < 1.0))
            st |= ORC_BAD_U;
    for (int32_t i = 1; i < N; ++i) {
        if (parent[i] < 0 || parent[i] >= i) {
            st |= ORC_BAD_TREE;
        } else if (tok[i] < 0 || tok[i] >= V) {
            st |= ORC_BAD_TOKEN;
        } else {
            double qx = Q[(int64_t)parent[i] * V + tok[i]];
            if (!(qx > 0.0) || !isfinite(qx))
                st |= ORC_BAD_Q;
        }
    }
    if (rows_ok)
        for (int32_t i = 0; i < N; ++i)
            if (!rows_ok[i])
                st |= ORC_BAD_ROW;
    for (int32_t i = 0; i < N; ++i) {
        out_tokens[i] = -1;
        out_nodes[i] = -1;
        accept_prob[i] = -1.0;
    }
    *num_emitted = 0;
    if (st) {
        *status = st;
        return;
    }

    int32_t v = 0, len = 0, y = -1;
    for (;;) {
        const double *pv = P + (int64_t)v * V;
        const double *qv = Q + (int64_t)v * V;
        for (int32_t i = 0; i < V; ++i)
            r[i] = pv[i];
        int has_child = 0, next = -1, degenerate = 0;
        for (int32_t c = v + 1; c < N; ++c) {
            if (parent[c] != v)
                continue;
            has_child = 1;
            double a = r[tok[c]] / qv[tok[c]];
            a = a < 1.0 ? a : 1.0;
            accept_prob[c] = a;
            if (u[c] < a) {
                next = c;
                break;
            }
            double Z = 0.0;
            for (int32_t i = 0; i < V; ++i) {
                double d = r[i] - qv[i];
                r[i] = d > 0.0 ? d : 0.0;
                Z += r[i];
            }
            if (!(Z > 0.0)) {
                degenerate = 1;
                break;
            }
            for (int32_t i = 0; i < V; ++i)
                r[i] /= Z;
        }
        if (next >= 0) {
            out_tokens[len] = tok[next];
            out_nodes[len] = next;
            ++len;
            v = next;
            continue;
        }
        double Z;
        if (degenerate) {
            st |= ORC_DEGENERATE_RESIDUAL;
            y = inverse_cdf(pv, V, u[0], &Z);
        } else {
            (void)has_child; /* leaf: r = p_v; all rejected: r is the residual */
            for (int32_t i = 0; i < V; ++i)
                w[i] = r[i];
            y = inverse_cdf(w, V, u[0], &Z);
        }
        break;
    }
    out_tokens[len] = y;
    *num_emitted = len + 1;
    *status = st;
}

/* From probabilities: p, q [B, N, V] fp64, u [B, N] fp64. */
int sv_oracle_tree_verify_probs(const double *p, const double *q, const int32_t *parent,
                                const int32_t *tokens, const double *u, int64_t B, int32_t N,
                                int32_t V, int32_t *out_tokens, int32_t *out_nodes,
                                int32_t *num_emitted, double *accept_prob, int32_t *status)
{
    if (B < 0 || N < 1 || V < 1)
        return 1;
    double *r = malloc(sizeof(double) * (size_t)V);
    double *w = malloc(sizeof(double) * (size_t)V);
    if (!r || !w) {
        free(r);
        free(w);
        return 2;
    }
    for (int64_t b = 0; b < B; ++b)
        tree_sequence(p + b * N * (int64_t)V, q + b * N * (int64_t)V, parent + b * N,
                      tokens + b * N, u + b * N, NULL, N, V, r, w, out_tokens + b * N,
                      out_nodes + b * N, num_emitted + b, accept_prob + b * N, status + b);
    free(r);
    free(w);
    return 0;
}

/* From logits (bf16 bits or fp32) [B, N, V], q fp32 [B, N, V], u fp32 [B, N]:
 * p_v = softmax(z_v / T) in fp64 for every node row. */
int sv_oracle_tree_verify(const void *logits, int dtype, const float *q, const int32_t *parent,
                          const int32_t *tokens, const float *u, double T, int64_t B, int32_t N,
                          int32_t V, int32_t *out_tokens, int32_t *out_nodes, int32_t *num_emitted,
                          double *accept_prob, int32_t *status)
{
    if (B < 0 || N < 1 || V < 1 || !(T > 0.0))
        return 1;
    size_t rows = (size_t)N * (size_t)V;
    double *P = malloc(sizeof(double) * rows);
    double *Q = malloc(sizeof(double) * rows);
    double *ud = malloc(sizeof(double) * (size_t)N);
    int *ok = malloc(sizeof(int) * (size_t)N);
    double *r = malloc(sizeof(double) * (size_t)V);
    double *w = malloc(sizeof(double) * (size_t)V);
    if (!P || !Q || !ud || !ok || !r || !w) {
        free(P); free(Q); free(ud); free(ok); free(r); free(w);
        return 2;
    }
    for (int64_t b = 0; b < B; ++b) {
        for (int32_t i = 0; i < N; ++i) {
            ok[i] = softmax_row(logits, dtype, (b * N + i) * (int64_t)V, V, T, P + (int64_t)i * V);
            ud[i] = (double)u[b * N + i];
        }
        for (size_t k = 0; k < rows; ++k)
            Q[k] = (double)q[(size_t)b * rows + k];
        tree_sequence(P, Q, parent + b * N, tokens + b * N, ud, ok, N, V, r, w,
                      out_tokens + b * N, out_nodes + b * N, num_emitted + b,
                      accept_prob + b * N, status + b);
    }
    free(P); free(Q); free(ud); free(ok); free(r); free(w);
    return 0;
}
