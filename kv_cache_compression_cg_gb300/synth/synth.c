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
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { SYN_AR1 = 0, SYN_STUDENT_T = 1, SYN_UNIFORM = 2 };

typedef struct syn_params {
    int32_t kind;
    int32_t L, T, C;
    uint64_t seed;
    double rho;
    double sigma_log;
    double outlier_frac;
    double outlier_scale;
} syn_params;

/* ---------------------------------------------------------------- RNG */
static uint64_t sm64(uint64_t key, uint64_t i)
{
    uint64_t z = key + (i + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* uniform in (0, 1]: 53 random bits */
static double u01_open0(uint64_t x) { return ((double)(x >> 11) + 1.0) * 0x1p-53; }
/* uniform in [0, 1) */
static double u01(uint64_t x) { return (double)(x >> 11) * 0x1p-53; }

/* ------------------------------------------------- elementary functions */
static const double LN2_HI = 6.93147180369123816490e-01; /* 0x3FE62E42FEE00000 */
static const double LN2_LO = 1.90821492927058770002e-10;

/* ln(x), x > 0: x = m 2^e with m in [sqrt(1/2), sqrt(2)); with
 * s = (m-1)/(m+1), ln m = 2 (s + s^3/3 + s^5/5 + ...). */
static double syn_log(double x)
{
    int e;
    double m = frexp(x, &e); /* m in [0.5, 1) */
    if (m < 0.70710678118654752440) {
        m *= 2.0;
        e -= 1;
    }
    double s = (m - 1.0) / (m + 1.0);
    double s2 = s * s;
    double term = s, sum = 0.0;
    for (int k = 0; k < 14; k++) {
        sum = sum + term / (double)(2 * k + 1);
        term = term * s2;
    }
    return ((double)e * LN2_LO + 2.0 * sum) + (double)e * LN2_HI;
}

/* exp(x): x = n ln2 + r, |r| <= ln2/2, Taylor series of exp(r). */
static double syn_exp(double x)
{
    double n = nearbyint(x / 0.69314718055994530942);
    double r = (x - n * LN2_HI) - n * LN2_LO;
    double term = 1.0, sum = 1.0;
    for (int k = 1; k < 22; k++) {
        term = term * r / (double)k;
        sum = sum + term;
    }
    return ldexp(sum, (int)n);
}

/* sin and cos of pi/2 * f for f in [0, 1], Taylor series. */
static void syn_sincos_quarter(double f, double *s, double *c)
{
    double x = f * 1.57079632679489661923;
    double x2 = x * x;
    double ts = x, tc = 1.0, ss = 0.0, cc = 0.0;
    for (int k = 0; k < 14; k++) {
        ss = ss + ts;
        cc = cc + tc;
        ts = -ts * x2 / (double)((2 * k + 2) * (2 * k + 3));
        tc = -tc * x2 / (double)((2 * k + 1) * (2 * k + 2));
    }
    *s = ss;
    *c = cc;
}

/* (cos 2 pi u, sin 2 pi u) for u in [0, 1), by quadrant. */
static void syn_cis(double u, double *c, double *s)
{
    double v = u * 4.0; /* exact */
    int q = (int)v;
    double f = v - (double)q; /* exact */
    double sq, cq;
    syn_sincos_quarter(f, &sq, &cq);
    switch (q & 3) {
    case 0: *c = cq; *s = sq; break;
    case 1: *c = -sq; *s = cq; break;
    case 2: *c = -cq; *s = -sq; break;
    default: *c = sq; *s = -cq; break;
    }
}

/* Two independent N(0,1) from two uniforms (Box-Muller). */
static void syn_normal2(uint64_t key, uint64_t i, double *z0, double *z1)
{
    double u1 = u01_open0(sm64(key, 2 * i));
    double u2 = u01(sm64(key, 2 * i + 1));
    double rad = sqrt(-2.0 * syn_log(u1));
    double c, s;
    syn_cis(u2, &c, &s);
    *z0 = rad * c;
    *z1 = rad * s;
}

static double syn_normal(uint64_t key, uint64_t i)
{
    double a, b;
    syn_normal2(key, i, &a, &b);
    return a;
}

/* ------------------------------------------------- double -> fp16 bits */
static uint16_t syn_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (!(a < 65504.0))
        return sign | 0x7BFF; /* saturate (also catches NaN, none produced) */
    if (a < 0x1p-14) {
        double r = nearbyint(ldexp(a, 24)); /* subnormal units of 2^-24 */
        return sign | (uint16_t)r;          /* r == 1024 -> smallest normal */
    }
    int e;
    double m = frexp(a, &e); /* a = m 2^e, m in [0.5, 1) */
    int E = e - 1;           /* a = 1.f 2^E, E in [-14, 15] */
    double r = nearbyint(ldexp(m, 11)); /* in [1024, 2048] */
    if (r == 2048.0) {
        r = 1024.0;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7BFF;
    return sign | (uint16_t)(((E + 15) << 10) | ((int)r - 1024));
}

/* ------------------------------------------------------------ slices */
/* Per-element counter, independent of T so a token prefix of a tensor is the
 * prefix of the longer tensor. */
static uint64_t elem_ctr(int c, int t) { return ((uint64_t)c << 32) | (uint64_t)t; }

static uint64_t slice_key(const syn_params *p, int kv, int layer)
{
    uint64_t k0 = sm64(p->seed, 0);
    return sm64(k0, ((uint64_t)kv << 32) | (uint64_t)layer);
}

/* One (kv, layer) slice into out[t * C + c]. */
static int syn_fill_slice(const syn_params *p, int kv, int layer, uint16_t *out)
{
    const int T = p->T, C = p->C;
    uint64_t key = slice_key(p, kv, layer);
    uint64_t key_sigma = sm64(key, 1), key_out = sm64(key, 2);
    uint64_t key_val = sm64(key, 3);

    if (p->kind == SYN_UNIFORM) {
        for (int t = 0; t < T; t++)
            for (int c = 0; c < C; c++)
                out[(int64_t)t * C + c] =
                    syn_to_half(u01(sm64(key_val, elem_ctr(c, t))));
        return 0;
    }

    double *sigma = (double *)malloc(sizeof(double) * C);
    int *perm = (int *)malloc(sizeof(int) * C);
    double *state = (double *)malloc(sizeof(double) * C);
    if (!sigma || !perm || !state) {
        free(sigma); free(perm); free(state);
        return -1;
    }
    for (int c = 0; c < C; c++) {
        sigma[c] = syn_exp(p->sigma_log * syn_normal(key_sigma, (uint64_t)c));
        perm[c] = c;
    }
    int n_out = (int)nearbyint(p->outlier_frac * (double)C);
    for (int i = 0; i < n_out; i++) { /* partial Fisher-Yates */
        uint64_t j = (uint64_t)i + sm64(key_out, (uint64_t)i) % (uint64_t)(C - i);
        int tmp = perm[i];
        perm[i] = perm[j];
        perm[j] = tmp;
        sigma[perm[i]] *= p->outlier_scale;
    }

    if (p->kind == SYN_AR1) {
        double stat = sqrt(1.0 - p->rho * p->rho);
        for (int t = 0; t < T; t++)
            for (int c = 0; c < C; c++) {
                double z = syn_normal(key_val, elem_ctr(c, t));
                double x;
                if (t == 0)
                    x = sigma[c] * z / stat;
                else
                    x = p->rho * state[c] + sigma[c] * z;
                state[c] = x;
                out[(int64_t)t * C + c] = syn_to_half(x);
            }
    } else { /* SYN_STUDENT_T, nu = 3 */
        for (int t = 0; t < T; t++)
            for (int c = 0; c < C; c++) {
                uint64_t i = elem_ctr(c, t) * 2;
                double z0, z1, z2, z3;
                syn_normal2(key_val, i, &z0, &z1);
                syn_normal2(key_val, i + 1, &z2, &z3);
                double chi = (z1 * z1 + z2 * z2) + z3 * z3;
                double x = sigma[c] * z0 / sqrt(chi / 3.0);
                out[(int64_t)t * C + c] = syn_to_half(x);
            }
    }
    free(sigma);
    free(perm);
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
