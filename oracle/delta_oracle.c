/*
 * delta_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct float64 CPU implementation of the forward
 * pass of delta-rule linear attention (DeltaNet, Gated DeltaNet, Gated
 * DeltaProduct).  It exists to check the CUDA library against; only the test
 * suite, the smoke check and the bench's CPU-baseline leg may load it.  It
 * shares no code, header or table with the CUDA path.
 *
 * What it computes -- the recurrence itself, token by token, in the order the
 * pages state it:
 *
 *   "DeltaProduct: 通过 Householder 乘积增强线性 RNN 的状态追踪" (reading
 *   notes), section 2.6 "Gated DeltaProduct" conceptual pseudo-code:
 *       H = g_i * H                      (gate once per token, g = 1 if absent)
 *       for j in 1..n_h:
 *           error = v_ij - H^T k_ij       (prediction error)
 *           H     = H + beta_ij * outer(k_ij, error)
 *       output_i = H^T q_i               (readout after the token's update)
 *   with H the [dk, dv] state (section 2.1: H_i in R^{n x d}, keys in R^n).
 *
 *   "08 · linear 路线（三）：delta rule 与 DPLR 统一框架", section 2.3, the
 *   recurrent reference form (the decode path): read v_old = S^T k, write only
 *   the residual beta * k (v - v_old)^T, then read out with q after the write.
 *   For n_h = 1 and g = 1 the loop above is exactly that form; section 1.2's
 *   S_t = (I - beta k k^T) S_{t-1} + beta k v^T is the same update expanded.
 *
 * Readings taken where the pages are silent:
 *   - no query scale (callers pre-scale q);
 *   - the gate is the linear gate g in [0,1] (g = 0 is an exact reset);
 *   - nothing is normalised or clamped here: inputs are used as given.
 *
 * Inputs arrive as float32 arrays: every value the GPU library sees (bf16 or
 * fp32) is exactly representable in float32, so the oracle consumes the very
 * same numbers.  All arithmetic is float64.
 *
 * Layouts (row-major, contiguous):
 *   q    [B, T, H, dk]          k    [B, T, n_h, H, dk]
 *   v    [B, T, n_h, H, dv]     beta [B, T, n_h, H]
 *   g    [B, T, H] or NULL      h0   [B, H, dk, dv] or NULL (=> zero state;
 *                                float32, or float64 for the decode carry)
 *   out  [B, T, H, dv] (f64)    hT   [B, H, dk, dv] (f64) or NULL
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const float *q, *k, *v, *beta, *g, *h0;
    const double *h0d;      /* float64 initial state (decode carry), or NULL */
    double *out, *hT;
    int64_t B, H, T, dk, dv, n_h;
    int64_t next;           /* next (b,h) pair to process */
    pthread_mutex_t lock;
    int failed;
} job_t;

/* One independent (b, h) sequence: the whole recurrence for that head. */
static int run_head(job_t *J, int64_t b, int64_t h, double *S, double *e)
{
    const int64_t H = J->H, T = J->T, dk = J->dk, dv = J->dv, n_h = J->n_h;

    if (J->h0) {
        const float *src = J->h0 + (b * H + h) * dk * dv;
        for (int64_t i = 0; i < dk * dv; ++i) S[i] = (double)src[i];
    } else if (J->h0d) {
        memcpy(S, J->h0d + (b * H + h) * dk * dv, sizeof(double) * (size_t)(dk * dv));
    } else {
        memset(S, 0, sizeof(double) * (size_t)(dk * dv));
    }

    for (int64_t t = 0; t < T; ++t) {
        /* gate once per token, before the sub-steps */
        if (J->g) {
            const double gt = (double)J->g[(b * T + t) * H + h];
            for (int64_t i = 0; i < dk * dv; ++i) S[i] *= gt;
        }
        /* n_h Householder sub-steps in execution order */
        for (int64_t j = 0; j < n_h; ++j) {
            const int64_t row = ((b * T + t) * n_h + j) * H + h;
            const float *kk = J->k + row * dk;
            const float *vv = J->v + row * dv;
            const double bb = (double)J->beta[row];
            /* e = v - S^T k */
            for (int64_t c = 0; c < dv; ++c) {
                double acc = 0.0;
                for (int64_t d = 0; d < dk; ++d) acc += S[d * dv + c] * (double)kk[d];
                e[c] = (double)vv[c] - acc;
            }
            /* S += beta * k e^T */
            for (int64_t d = 0; d < dk; ++d) {
                const double s = bb * (double)kk[d];
                for (int64_t c = 0; c < dv; ++c) S[d * dv + c] += s * e[c];
            }
        }
        /* out_t = S^T q_t, after the token's update */
        const float *qq = J->q + ((b * T + t) * H + h) * dk;
        double *oo = J->out + ((b * T + t) * H + h) * dv;
        for (int64_t c = 0; c < dv; ++c) {
            double acc = 0.0;
            for (int64_t d = 0; d < dk; ++d) acc += S[d * dv + c] * (double)qq[d];
            oo[c] = acc;
        }
    }

    if (J->hT) {
        double *dst = J->hT + (b * H + h) * dk * dv;
        memcpy(dst, S, sizeof(double) * (size_t)(dk * dv));
    }
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)(J->dk * J->dv));
    double *e = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!S || !e) {
        pthread_mutex_lock(&J->lock);
        J->failed = 1;
        pthread_mutex_unlock(&J->lock);
        free(S);
        free(e);
        return NULL;
    }
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t idx = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (idx >= J->B * J->H) break;
        run_head(J, idx / J->H, idx % J->H, S, e);
    }
    free(S);
    free(e);
    return NULL;
}

static int run_all(const float *q, const float *k, const float *v,
                   const float *beta, const float *g, const float *h0,
                   const double *h0d, double *out, double *hT,
                   int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv,
                   int64_t n_h, int nthreads)
{
    if (!q || !k || !v || !beta || !out) return -1;
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0 || n_h <= 0) return -1;

    job_t J;
    J.q = q; J.k = k; J.v = v; J.beta = beta; J.g = g; J.h0 = h0; J.h0d = h0d;
    J.out = out; J.hT = hT;
    J.B = B; J.H = H; J.T = T; J.dk = dk; J.dv = dv; J.n_h = n_h;
    J.next = 0;
    J.failed = 0;
    pthread_mutex_init(&J.lock, NULL);

    int64_t pairs = B * H;
    int n = nthreads > 0 ? nthreads : 1;
    if ((int64_t)n > pairs) n = pairs > 0 ? (int)pairs : 1;

    if (n == 1) {
        worker(&J);
    } else {
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n);
        if (!tid) {
            worker(&J);
        } else {
            int started = 0;
            for (int i = 0; i < n; ++i) {
                if (pthread_create(&tid[i], NULL, worker, &J) != 0) break;
                ++started;
            }
            if (started == 0) worker(&J);
            for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
            free(tid);
        }
    }
    pthread_mutex_destroy(&J.lock);
    return J.failed ? -2 : 0;
}

/*
 * delta_oracle_fwd: returns 0 on success, -1 on bad arguments, -2 if a worker
 * could not allocate its scratch state.  nthreads <= 0 means one thread.
 */
int delta_oracle_fwd(const float *q, const float *k, const float *v,
                     const float *beta, const float *g, const float *h0,
                     double *out, double *hT,
                     int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv,
                     int64_t n_h, int nthreads)
{
    return run_all(q, k, v, beta, g, h0, NULL, out, hT, B, H, T, dk, dv, n_h, nthreads);
}

/*
 * delta_oracle_fwd_state64: the same, with the initial state given in
 * float64 (NULL => zero), so that a state carried from one call to the next
 * (the decode path) is never rounded.
 */
int delta_oracle_fwd_state64(const float *q, const float *k, const float *v,
                             const float *beta, const float *g, const double *h0,
                             double *out, double *hT,
                             int64_t B, int64_t H, int64_t T, int64_t dk, int64_t dv,
                             int64_t n_h, int nthreads)
{
    return run_all(q, k, v, beta, g, NULL, h0, out, hT, B, H, T, dk, dv, n_h, nthreads);
}
