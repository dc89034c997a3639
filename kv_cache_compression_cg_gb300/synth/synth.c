/*
 * synth.c - seeded synthetic KV-cache generator.
 *
 * Produces fp16 K and V tensors [L][T][C] standing in for a model's KV cache
 * (no trained weights are available). It holds none of the codec's arithmetic
 * and is shared by the CUDA tests, the CPU oracle tests and the benchmark,
 * which therefore all see byte-identical inputs.
 *
 * Random numbers: SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used as a counter-based
 * generator: draw(key, i) is the SplitMix64 output for state key at step i.
 * Every value is keyed by (seed, kv, layer, channel, token, draw), so any
 * (kv, layer) slice is generated on its own and the result does not depend on
 * the thread count.
 *
 * Normal variates come from the Box-Muller transform; ln, exp, sin and cos are
 * evaluated here from their power series with only +, -, *, / (compiled
 * without fused multiply-add), so the bytes are the same on every IEEE-754
 * machine. double -> fp16 conversion rounds to nearest-even and saturates at
 * +-65504.
 *
 * Value models (per (kv, layer) slice, per channel c):
 *   sigma_c = exp(sigma_log * N(0,1)) (LogNormal(0, sigma_log)); a set of
 *   round(outlier_frac * C) channels, drawn without replacement, has sigma_c
 *   multiplied by outlier_scale.
 *   AR1:       x_0 ~ N(0, sigma_c^2 / (1 - rho^2)), x_t = rho x_{t-1} + sigma_c z_t
 *   STUDENT_T: x_t = sigma_c * Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3) (nu = 3)
 *   UNIFORM:   x_t ~ U[0, 1) (no sigma)
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "synth_core.h"

/* sigma_c of one (kv, layer) slice: LogNormal(0, sigma_log) per channel, and
 * round(outlier_frac * C) channels drawn without replacement (partial
 * Fisher-Yates) scaled by outlier_scale. */
int syn_slice_sigma(const syn_params *p, int kv, int layer, double *sigma)
{
    const int C = p->C;
    uint64_t key = slice_key(p, kv, layer);
    uint64_t key_sigma = sm64(key, 1), key_out = sm64(key, 2);
    int *perm = (int *)malloc(sizeof(int) * C);
    if (!perm)
        return -1;
    for (int c = 0; c < C; c++) {
        sigma[c] = syn_exp(p->sigma_log * syn_normal(key_sigma, (uint64_t)c));
        perm[c] = c;
    }
    int n_out = (int)nearbyint(p->outlier_frac * (double)C);
    for (int i = 0; i < n_out; i++) {
        uint64_t j = (uint64_t)i + sm64(key_out, (uint64_t)i) % (uint64_t)(C - i);
        int tmp = perm[i];
        perm[i] = perm[j];
        perm[j] = tmp;
        sigma[perm[i]] *= p->outlier_scale;
    }
    free(perm);
    return 0;
}

/* One (kv, layer) slice into out[t * C + c]. */
static int syn_fill_slice(const syn_params *p, int kv, int layer, uint16_t *out)
{
    const int T = p->T, C = p->C;
    uint64_t key = slice_key(p, kv, layer);
    uint64_t key_val = sm64(key, 3);

    if (p->kind == SYN_UNIFORM) {
        for (int t = 0; t < T; t++)
            for (int c = 0; c < C; c++)
                out[(int64_t)t * C + c] =
                    syn_to_half(u01(sm64(key_val, elem_ctr(c, t))));
        return 0;
    }

    double *sigma = (double *)malloc(sizeof(double) * C);
    double *state = (double *)malloc(sizeof(double) * C);
    if (!sigma || !state || syn_slice_sigma(p, kv, layer, sigma) != 0) {
        free(sigma); free(state);
        return -1;
    }
    if (p->kind == SYN_AR1) {
        double stat = sqrt(1.0 - p->rho * p->rho);
        for (int t = 0; t < T; t++)
            for (int c = 0; c < C; c++) {
                double x = syn_ar1_next(p, key_val, c, t, sigma[c], stat, state[c]);
                state[c] = x;
                out[(int64_t)t * C + c] = syn_to_half(x);
            }
    } else { /* SYN_STUDENT_T, nu = 3 */
        for (int t = 0; t < T; t++)
            for (int c = 0; c < C; c++)
                out[(int64_t)t * C + c] = syn_to_half(syn_student_value(key_val, c, t, sigma[c]));
    }
    free(sigma);
    free(state);
    return 0;
}

typedef struct syn_job {
    const syn_params *p;
    uint16_t *k, *v;
    int64_t layer_stride;
    int next_total;
    int *next;
    pthread_mutex_t *mu;
    int err;
} syn_job;

static void *syn_worker(void *arg)
{
    syn_job *j = (syn_job *)arg;
    for (;;) {
        pthread_mutex_lock(j->mu);
        int idx = (*j->next)++;
        pthread_mutex_unlock(j->mu);
        if (idx >= j->next_total)
            break;
        int kv = idx / j->p->L, layer = idx % j->p->L;
        uint16_t *dst = (kv ? j->v : j->k) + (int64_t)layer * j->layer_stride;
        if (syn_fill_slice(j->p, kv, layer, dst) != 0)
            j->err = -1;
    }
    return NULL;
}

/* Fill K and V ([L][T][C], layers layer_stride elements apart) with nthreads
 * workers over the 2*L slices. Returns 0 on success. */
int syn_generate(const syn_params *p, uint16_t *k, uint16_t *v,
                 int64_t layer_stride, int nthreads)
{
    if (!p || p->L < 1 || p->T < 1 || p->C < 1 || !k || !v)
        return -1;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 2 * p->L)
        nthreads = 2 * p->L;
    pthread_mutex_t mu = PTHREAD_MUTEX_INITIALIZER;
    int next = 0;
    syn_job *jobs = (syn_job *)calloc((size_t)nthreads, sizeof(syn_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs); free(th);
        return -1;
    }
    for (int i = 0; i < nthreads; i++) {
        jobs[i] = (syn_job){p, k, v, layer_stride, 2 * p->L, &next, &mu, 0};
        pthread_create(&th[i], NULL, syn_worker, &jobs[i]);
    }
    int err = 0;
    for (int i = 0; i < nthreads; i++) {
        pthread_join(th[i], NULL);
        err |= jobs[i].err;
    }
    free(jobs);
    free(th);
    return err;
}

/* Tokens [t0, t1) of one (kv, layer) slice into out[(t - t0) * C + c]; the
 * AR(1) recurrence still runs from token 0. */
int syn_generate_slice_range(const syn_params *p, int kv, int layer, int t0, int t1,
                             uint16_t *out)
{
    if (!p || kv < 0 || kv > 1 || layer < 0 || layer >= p->L || t0 < 0 || t1 < t0 || t1 > p->T || !out)
        return -1;
    const int C = p->C;
    uint64_t key_val = sm64(slice_key(p, kv, layer), 3);
    if (p->kind == SYN_UNIFORM) {
        for (int t = t0; t < t1; t++)
            for (int c = 0; c < C; c++)
                out[(int64_t)(t - t0) * C + c] = syn_to_half(u01(sm64(key_val, elem_ctr(c, t))));
        return 0;
    }
    double *sigma = (double *)malloc(sizeof(double) * C);
    double *state = (double *)calloc((size_t)C, sizeof(double));
    if (!sigma || !state || syn_slice_sigma(p, kv, layer, sigma) != 0) {
        free(sigma); free(state);
        return -1;
    }
    if (p->kind == SYN_AR1) {
        double stat = sqrt(1.0 - p->rho * p->rho);
        for (int t = 0; t < t1; t++)
            for (int c = 0; c < C; c++) {
                double x = syn_ar1_next(p, key_val, c, t, sigma[c], stat, state[c]);
                state[c] = x;
                if (t >= t0)
                    out[(int64_t)(t - t0) * C + c] = syn_to_half(x);
            }
    } else {
        for (int t = t0; t < t1; t++)
            for (int c = 0; c < C; c++)
                out[(int64_t)(t - t0) * C + c] = syn_to_half(syn_student_value(key_val, c, t, sigma[c]));
    }
    free(sigma);
    free(state);
    return 0;
}

/* One slice alone (for regenerating a sample on the host). */
int syn_generate_slice(const syn_params *p, int kv, int layer, uint16_t *out)
{
    if (!p || kv < 0 || kv > 1 || layer < 0 || layer >= p->L || !out)
        return -1;
    return syn_fill_slice(p, kv, layer, out);
}

/* Exposed for the generator's own checks. */
double syn_ln(double x) { return syn_log(x); }
double syn_expo(double x) { return syn_exp(x); }
void syn_cis2pi(double u, double *c, double *s) { syn_cis(u, c, s); }
uint16_t syn_half(double x) { return syn_to_half(x); }
uint64_t syn_splitmix(uint64_t key, uint64_t i) { return sm64(key, i); }
