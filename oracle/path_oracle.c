/*
 * PaTH attention oracle: plain fp64 CPU code, written straight from the
 * definition of the method.
 *
 * TEST INFRASTRUCTURE ONLY. Only tests/, the package's smoke() check and the
 * CPU-baseline leg of bench.py may load this library. The CUDA product path
 * shares no code with it and never calls it.
 *
 * Sources (web pages on PaTH attention):
 *  [KO] "거리에서 경로로, PaTH Attention" (iplexlaw.co.kr review),
 *       §3 핵심 원리 (per-token H = I - beta w w^T; logit k_j^T(H_{j+1}...H_i)q_i,
 *       order matters), §4 (softmax over the logits, weighted sum of V,
 *       PaTH-FoX adds a forget gate), §9 (decode updates the cached keys in place).
 *  [JA] "技術要約: PaTH Attention" (gist.science), §2 手法 "コアメカニズム"
 *       (logit formula, product s = j+1..i, H_s = I - beta_s w_s w_s^T),
 *       §2 "拡張: PaTH-FoX" (additive data-dependent forget gate),
 *       §3 "推論" (in-place key update with the current transition).
 *
 * Readings where the pages are silent (same list as the design notes):
 *  - softmax scale sigma multiplies the whole PaTH logit; the FoX bias
 *    sum_{s=j+1..i} log f_s is added after scaling, unscaled;
 *  - the product covers s = j+1..i: H_i is applied to q_i first, H_j is not
 *    applied; j = i uses the identity; the attention is causal (j <= i);
 *  - decode step t with N cached keys: first k_j <- H_t k_j for every j < N,
 *    then append (k_t, v_t) untransformed, then attend with q_t over N+1 keys.
 *
 * Every function computes the definition directly: no blocking, no UT
 * transform, no fusion. Cost O(L^2 d) per head.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* x <- H x with H = I - beta w w^T  ([KO] §3, [JA] §2 "データ依存の遷移行列"). */
static void apply_transition(double *x, const double *w, double beta, int d)
{
    double dot = 0.0;
    for (int c = 0; c < d; ++c)
        dot += w[c] * x[c];
    const double a = beta * dot;
    for (int c = 0; c < d; ++c)
        x[c] -= a * w[c];
}

/*
 * Logits of query row i against keys j = i, i-1, ..., 0 of one head:
 *   logit[j] = scale * k_j^T (H_{j+1} ... H_i) q_i  [+ sum_{s=j+1..i} log f_s]
 * The running vector x starts at q_i; once key j is scored, H_j is applied so
 * that x = H_j ... H_i q_i when key j-1 is scored ([JA] §2 formula; [KO] §3).
 */
static void row_logits(const double *q_i, const double *K, const double *W,
                       const double *beta, const double *log_f, int i, int d,
                       double scale, double *logit, double *x)
{
    memcpy(x, q_i, (size_t)d * sizeof(double));
    double bias = 0.0;
    for (int j = i; j >= 0; --j) {
        const double *k_j = K + (size_t)j * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += k_j[c] * x[c];
        logit[j] = scale * dot + bias;
        apply_transition(x, W + (size_t)j * d, beta[j], d);
        if (log_f)
            bias += log_f[j];
    }
}

/* Causal softmax over logit[0..n-1] and the weighted sum of V rows ([KO] §4). */
static void softmax_combine(const double *logit, const double *V, int n, int d,
                            double *p, double *out, double *lse)
{
    double m = -INFINITY;
    for (int j = 0; j < n; ++j)
        if (logit[j] > m)
            m = logit[j];
    double z = 0.0;
    for (int j = 0; j < n; ++j) {
        p[j] = exp(logit[j] - m);
        z += p[j];
    }
    for (int c = 0; c < d; ++c)
        out[c] = 0.0;
    for (int j = 0; j < n; ++j) {
        const double pj = p[j] / z;
        const double *v_j = V + (size_t)j * d;
        for (int c = 0; c < d; ++c)
            out[c] += pj * v_j[c];
    }
    if (lse)
        *lse = m + log(z);
}

/* ---------------------------------------------------------------- threads */

typedef struct {
    const double *q, *k, *v, *w, *beta, *log_f;
    int L, d;
    double scale;
    const int64_t *rows; /* (head, i) pairs, or NULL for every row */
    int64_t nrows;
    double *out, *lse;
    int64_t next; /* shared work counter */
    pthread_mutex_t mu;
} fwd_job;

static int64_t take(fwd_job *job, int64_t chunk)
{
    pthread_mutex_lock(&job->mu);
    int64_t r = job->next;
    job->next += chunk;
    pthread_mutex_unlock(&job->mu);
    return r;
}

static void *fwd_worker(void *arg)
{
    fwd_job *job = (fwd_job *)arg;
    const int L = job->L, d = job->d;
    double *logit = (double *)malloc((size_t)L * sizeof(double));
    double *p = (double *)malloc((size_t)L * sizeof(double));
    double *x = (double *)malloc((size_t)d * sizeof(double));
    for (;;) {
        const int64_t start = take(job, 16);
        if (start >= job->nrows)
            break;
        const int64_t stop = start + 16 < job->nrows ? start + 16 : job->nrows;
        for (int64_t r = start; r < stop; ++r) {
            int64_t head, i;
            if (job->rows) {
                head = job->rows[2 * r];
                i = job->rows[2 * r + 1];
            } else {
                head = r / L;
                i = r % L;
            }
            const size_t hb = (size_t)head * L;
            row_logits(job->q + (hb + i) * d, job->k + hb * d, job->w + hb * d,
                       job->beta + hb, job->log_f ? job->log_f + hb : NULL,
                       (int)i, d, job->scale, logit, x);
            softmax_combine(logit, job->v + hb * d, (int)i + 1, d, p,
                            job->out + (size_t)r * d,
                            job->lse ? job->lse + r : NULL);
        }
    }
    free(logit);
    free(p);
    free(x);
    return NULL;
}

static int resolve_threads(int nthreads)
{
    if (nthreads > 0)
        return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static void run_job(fwd_job *job, int nthreads)
{
    nthreads = resolve_threads(nthreads);
    pthread_mutex_init(&job->mu, NULL);
    job->next = 0;
    pthread_t *tid = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t)
        pthread_create(&tid[t], NULL, fwd_worker, job);
    for (int t = 0; t < nthreads; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&job->mu);
}

/* ---------------------------------------------------------------- exports */

/*
 * Full forward. Tensors are contiguous (nh, L, d) with nh = B*H heads;
 * beta and log_f are (nh, L); log_f may be NULL (plain PaTH) or the per-token
 * log forget gate (PaTH-FoX). out is (nh, L, d); lse (nh, L) may be NULL.
 * nthreads <= 0 uses every online core. Returns the thread count used.
 */
int oracle_path_fwd(const double *q, const double *k, const double *v,
                    const double *w, const double *beta, const double *log_f,
                    int nh, int L, int d, double scale, double *out, double *lse,
                    int nthreads)
{
    fwd_job job = {q, k, v, w, beta, log_f, L, d, scale, NULL,
                   (int64_t)nh * L, out, lse, 0};
    run_job(&job, nthreads);
    return resolve_threads(nthreads);
}

/*
 * The same forward for a list of sampled rows: rows holds nrows pairs
 * (head, i); out is (nrows, d), lse (nrows). Costs O(i d) per row, so it can
 * check sampled outputs of workloads too large for the full forward.
 */
int oracle_path_rows(const double *q, const double *k, const double *v,
                     const double *w, const double *beta, const double *log_f,
                     int nh, int L, int d, double scale, const int64_t *rows,
                     int64_t nrows, double *out, double *lse, int nthreads)
{
    (void)nh;
    fwd_job job = {q, k, v, w, beta, log_f, L, d, scale, rows, nrows, out, lse, 0};
    run_job(&job, nthreads);
    return resolve_threads(nthreads);
}

/* Full logit matrix of one head: logits[i*L + j] for j <= i, -inf above. */
void oracle_path_logits(const double *q, const double *k, const double *w,
                        const double *beta, const double *log_f, int L, int d,
                        double scale, double *logits)
{
    double *x = (double *)malloc((size_t)d * sizeof(double));
    for (int i = 0; i < L; ++i) {
        double *row = logits + (size_t)i * L;
        row_logits(q + (size_t)i * d, k, w, beta, log_f, i, d, scale, row, x);
        for (int j = i + 1; j < L; ++j)
            row[j] = -INFINITY;
    }
    free(x);
}

/*
 * The transport used for every logit: x = H_{j+1} ... H_i q for one head,
 * applying H_i first. Exposed so that tests can pin its invariants.
 */
void oracle_path_transport(const double *q, const double *w, const double *beta,
                           int i, int j, int d, double *x)
{
    memcpy(x, q, (size_t)d * sizeof(double));
    for (int s = i; s > j; --s)
        apply_transition(x, w + (size_t)s * d, beta[s], d);
}

/*
 * One decode step for nh independent heads ([KO] §9, [JA] §3 "推論"):
 *   k_j <- H_t k_j for every cached j < len (in place in the fp64 cache),
 *   append k_t, v_t at index len, then attend with q_t over len+1 keys.
 * Kc, Vc are (nh, cap, d); q, k, v, w are (nh, d); beta (nh); out (nh, d).
 * log_f (nh) may be NULL; with it the cache keeps per-key running biases in
 * cbias (nh, cap): cbias_j <- cbias_j + log f_t for j < len, cbias_len = 0,
 * so that key j carries sum_{s=j+1..t} log f_s.
 */
void oracle_path_decode_step(const double *q, const double *k, const double *v,
                             const double *w, const double *beta,
                             const double *log_f, double *Kc, double *Vc,
                             double *cbias, int nh, int len, int cap, int d,
                             double scale, double *out)
{
    double *logit = (double *)malloc((size_t)(len + 1) * sizeof(double));
    double *p = (double *)malloc((size_t)(len + 1) * sizeof(double));
    for (int h = 0; h < nh; ++h) {
        double *K = Kc + (size_t)h * cap * d;
        double *V = Vc + (size_t)h * cap * d;
        const double *w_t = w + (size_t)h * d;
        for (int j = 0; j < len; ++j)
            apply_transition(K + (size_t)j * d, w_t, beta[h], d);
        memcpy(K + (size_t)len * d, k + (size_t)h * d, (size_t)d * sizeof(double));
        memcpy(V + (size_t)len * d, v + (size_t)h * d, (size_t)d * sizeof(double));
        if (log_f) {
            double *cb = cbias + (size_t)h * cap;
            for (int j = 0; j < len; ++j)
                cb[j] += log_f[h];
            cb[len] = 0.0;
        }
        const double *q_t = q + (size_t)h * d;
        for (int j = 0; j <= len; ++j) {
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += q_t[c] * K[(size_t)j * d + c];
            logit[j] = scale * dot + (log_f ? cbias[(size_t)h * cap + j] : 0.0);
        }
        softmax_combine(logit, V, len + 1, d, p, out + (size_t)h * d, NULL);
    }
    free(logit);
    free(p);
}

/*
 * Producer of w and beta from the token activations ([KO] §3: a low-dimensional linear
 * projection and a short convolution of size 3 give w, which is then L2-normalised, and
 * beta is 2 sigmoid; [JA] §2: beta_s = 2 sigmoid(u^T x_s + b); [JA] §6: beta needs
 * clipping in bf16).
 *   x (B, L, D) activations; w_down (R, D) and w_up (H*d, R): the projection
 *   x -> w_up (w_down x); conv (H*d, 3) depthwise causal taps, conv[c][2] on token t,
 *   conv[c][1] on t-1, conv[c][0] on t-2 (zero before the first token);
 *   u (H, D), bias (H): beta_t,h = min(2 sigmoid(u_h . x_t + bias_h), beta_max).
 *   w_out (B, H, L, d): per head, the convolved projection divided by max(norm, eps);
 *   beta_out (B, H, L).
 * Computed directly: projection of every token, then the convolution, then the norm.
 */
void oracle_wbeta_produce(const double *x, const double *w_down, const double *w_up,
                          const double *conv, const double *u, const double *bias,
                          double beta_max, int B, int L, int D, int R, int H, int d,
                          double eps, double *w_out, double *beta_out)
{
    const int C = H * d;
    double *z = (double *)malloc((size_t)L * R * sizeof(double));
    double *y = (double *)malloc((size_t)L * C * sizeof(double));
    double *yc = (double *)malloc((size_t)C * sizeof(double));
    for (int b = 0; b < B; ++b) {
        const double *xb = x + (size_t)b * L * D;
        for (int t = 0; t < L; ++t) {
            for (int r = 0; r < R; ++r) {
                double acc = 0.0;
                for (int c = 0; c < D; ++c)
                    acc += w_down[(size_t)r * D + c] * xb[(size_t)t * D + c];
                z[(size_t)t * R + r] = acc;
            }
            for (int ch = 0; ch < C; ++ch) {
                double acc = 0.0;
                for (int r = 0; r < R; ++r)
                    acc += w_up[(size_t)ch * R + r] * z[(size_t)t * R + r];
                y[(size_t)t * C + ch] = acc;
            }
        }
        for (int t = 0; t < L; ++t) {
            for (int ch = 0; ch < C; ++ch) {
                double acc = conv[(size_t)ch * 3 + 2] * y[(size_t)t * C + ch];
                if (t >= 1)
                    acc += conv[(size_t)ch * 3 + 1] * y[(size_t)(t - 1) * C + ch];
                if (t >= 2)
                    acc += conv[(size_t)ch * 3 + 0] * y[(size_t)(t - 2) * C + ch];
                yc[ch] = acc;
            }
            for (int h = 0; h < H; ++h) {
                double ss = 0.0;
                for (int c = 0; c < d; ++c)
                    ss += yc[h * d + c] * yc[h * d + c];
                const double n = sqrt(ss);
                const double den = n > eps ? n : eps;
                double *wo = w_out + (((size_t)b * H + h) * L + t) * d;
                for (int c = 0; c < d; ++c)
                    wo[c] = yc[h * d + c] / den;
                double a = bias[h];
                for (int c = 0; c < D; ++c)
                    a += u[(size_t)h * D + c] * xb[(size_t)t * D + c];
                double be = 2.0 / (1.0 + exp(-a));
                if (be > beta_max)
                    be = beta_max;
                beta_out[((size_t)b * H + h) * L + t] = be;
            }
        }
    }
    free(z);
    free(y);
    free(yc);
}

/* ---------------------------------------------------------------- backward */

/*
 * Gradients of the forward above for one head, by reverse mode through the
 * per-row sweep of row_logits (the pages give no backward pass; this is the
 * chain rule applied to the definition, step by step).
 *
 * Forward for row i: x_i = q_i; for j = i, i-1, ..., 0: logit_ij =
 * scale * k_j . x_j + bias_ij, then x_{j-1} = H_j x_j; softmax over j <= i;
 * out_i = sum_j p_ij v_j. With dout_i given:
 *   dp_ij = dout_i . v_j,  D_i = sum_j p_ij dp_ij,  dS_ij = p_ij (dp_ij - D_i)
 *   dv_j += p_ij dout_i
 * and, walking back from j = 0 to j = i with g the gradient of x_j:
 *   g += scale dS_ij k_j,   dk_j += scale dS_ij x_j;
 *   through x_j = H_{j+1} x_{j+1}, H = I - beta w w^T, input u = x_{j+1}:
 *     dbeta_{j+1} -= (w.g)(w.u),  dw_{j+1} -= beta ((w.u) g + (w.g) u),
 *     g <- H g (the gradient of x_{j+1});
 *   at j = i, dq_i += g.
 * The FoX bias sum_{s=j+1..i} log f_s gives dlog_f_s += dS_ij for j < s <= i.
 * xs holds the row's x_j (L * d), the other buffers L each.
 */
static void head_backward(const double *Q, const double *K, const double *V,
                          const double *W, const double *beta, const double *log_f,
                          const double *dO, int L, int d, double scale,
                          double *dQ, double *dK, double *dV, double *dW,
                          double *dbeta, double *dlogf, double *xs, double *logit,
                          double *p, double *g)
{
    for (int i = 0; i < L; ++i) {
        const double *q_i = Q + (size_t)i * d;
        const double *do_i = dO + (size_t)i * d;
        /* forward sweep, keeping x_j */
        memcpy(xs + (size_t)i * d, q_i, (size_t)d * sizeof(double));
        double bias = 0.0;
        for (int j = i; j >= 0; --j) {
            double *x_j = xs + (size_t)j * d;
            if (j < i) {
                memcpy(x_j, xs + (size_t)(j + 1) * d, (size_t)d * sizeof(double));
                apply_transition(x_j, W + (size_t)(j + 1) * d, beta[j + 1], d);
            }
            double dot = 0.0;
            for (int c = 0; c < d; ++c)
                dot += K[(size_t)j * d + c] * x_j[c];
            logit[j] = bias + scale * dot;
            if (log_f)
                bias += log_f[j];
        }
        /* softmax and its gradient */
        double m = -INFINITY;
        for (int j = 0; j <= i; ++j)
            if (logit[j] > m)
                m = logit[j];
        double z = 0.0;
        for (int j = 0; j <= i; ++j) {
            p[j] = exp(logit[j] - m);
            z += p[j];
        }
        double Dsum = 0.0;
        for (int j = 0; j <= i; ++j) {
            p[j] /= z;
            double dp = 0.0;
            for (int c = 0; c < d; ++c)
                dp += do_i[c] * V[(size_t)j * d + c];
            logit[j] = dp; /* logit[] now holds dp_ij */
            Dsum += p[j] * dp;
        }
        /* reverse sweep */
        for (int c = 0; c < d; ++c)
            g[c] = 0.0;
        double gate_acc = 0.0;
        for (int j = 0; j <= i; ++j) {
            const double dS = p[j] * (logit[j] - Dsum);
            const double *x_j = xs + (size_t)j * d;
            const double *k_j = K + (size_t)j * d;
            for (int c = 0; c < d; ++c) {
                dV[(size_t)j * d + c] += p[j] * do_i[c];
                dK[(size_t)j * d + c] += scale * dS * x_j[c];
                g[c] += scale * dS * k_j[c];
            }
            if (log_f) {
                gate_acc += dS; /* sum of dS_ij' over j' <= j: the gradient of log f_{j+1} */
                if (j < i)
                    dlogf[j + 1] += gate_acc;
            }
            if (j < i) {
                const double *w = W + (size_t)(j + 1) * d;
                const double b = beta[j + 1];
                const double *u = xs + (size_t)(j + 1) * d;
                double wu = 0.0, wg = 0.0;
                for (int c = 0; c < d; ++c) {
                    wu += w[c] * u[c];
                    wg += w[c] * g[c];
                }
                dbeta[j + 1] -= wg * wu;
                for (int c = 0; c < d; ++c)
                    dW[(size_t)(j + 1) * d + c] -= b * (wu * g[c] + wg * u[c]);
                for (int c = 0; c < d; ++c)
                    g[c] -= b * wg * w[c];
            }
        }
        for (int c = 0; c < d; ++c)
            dQ[(size_t)i * d + c] += g[c];
    }
}

typedef struct {
    const double *q, *k, *v, *w, *beta, *log_f, *dout;
    int nh, L, d;
    double scale;
    double *dq, *dk, *dv, *dw, *dbeta, *dlogf;
    int next;
    pthread_mutex_t mu;
} bwd_job;

static void *bwd_worker(void *arg)
{
    bwd_job *job = (bwd_job *)arg;
    const int L = job->L, d = job->d;
    double *xs = (double *)malloc((size_t)L * d * sizeof(double));
    double *logit = (double *)malloc((size_t)L * sizeof(double));
    double *p = (double *)malloc((size_t)L * sizeof(double));
    double *g = (double *)malloc((size_t)d * sizeof(double));
    for (;;) {
        pthread_mutex_lock(&job->mu);
        const int h = job->next++;
        pthread_mutex_unlock(&job->mu);
        if (h >= job->nh)
            break;
        const size_t td = (size_t)h * L * d, t1 = (size_t)h * L;
        head_backward(job->q + td, job->k + td, job->v + td, job->w + td, job->beta + t1,
                      job->log_f ? job->log_f + t1 : NULL, job->dout + td, L, d, job->scale,
                      job->dq + td, job->dk + td, job->dv + td, job->dw + td,
                      job->dbeta + t1, job->dlogf ? job->dlogf + t1 : NULL, xs, logit, p, g);
    }
    free(xs);
    free(logit);
    free(p);
    free(g);
    return NULL;
}

/*
 * Backward of oracle_path_fwd for the loss sum(dout * out): gradients with
 * respect to q, k, v, w, beta and (PaTH-FoX) log_f, all (nh, L, d) or (nh, L),
 * zeroed here first. dlogf may be NULL when log_f is. Heads run in parallel.
 * Returns the thread count used.
 */
int oracle_path_bwd(const double *q, const double *k, const double *v, const double *w,
                    const double *beta, const double *log_f, const double *dout, int nh,
                    int L, int d, double scale, double *dq, double *dk, double *dv,
                    double *dw, double *dbeta, double *dlogf, int nthreads)
{
    const size_t n = (size_t)nh * L * d, n1 = (size_t)nh * L;
    memset(dq, 0, n * sizeof(double));
    memset(dk, 0, n * sizeof(double));
    memset(dv, 0, n * sizeof(double));
    memset(dw, 0, n * sizeof(double));
    memset(dbeta, 0, n1 * sizeof(double));
    if (dlogf)
        memset(dlogf, 0, n1 * sizeof(double));
    bwd_job job = {q, k, v, w, beta, log_f, dout, nh, L, d, scale,
                   dq, dk, dv, dw, dbeta, log_f ? dlogf : NULL, 0};
    nthreads = resolve_threads(nthreads);
    if (nthreads > nh)
        nthreads = nh;
    pthread_mutex_init(&job.mu, NULL);
    pthread_t *tid = (pthread_t *)malloc((size_t)nthreads * sizeof(pthread_t));
    for (int t = 0; t < nthreads; ++t)
        pthread_create(&tid[t], NULL, bwd_worker, &job);
    for (int t = 0; t < nthreads; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&job.mu);
    return nthreads;
}
