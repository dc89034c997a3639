/*
 * synth_core.h - arithmetic of the seeded synthetic KV generator, shared by
 * the host generator (synth.c, gcc) and the device generator (synth_gpu.cu,
 * nvcc). Only +, -, *, / and sqrt (correctly rounded in IEEE-754 on both), the
 * exact helpers frexp/ldexp/nearbyint/fabs/signbit and integer operations are
 * used, and both builds disable fused multiply-add, so the host and the device
 * produce the same bytes. None of the codec's arithmetic is here.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <math.h>
#include <stdint.h>

#ifdef __CUDACC__
#define SYN_FN __host__ __device__ static inline
#else
#define SYN_FN static inline
#endif

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
SYN_FN uint64_t sm64(uint64_t key, uint64_t i)
{
    uint64_t z = key + (i + 1) * 0x9E3779B97F4A7C15ULL;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* uniform in (0, 1]: 53 random bits */
SYN_FN double u01_open0(uint64_t x) { return ((double)(x >> 11) + 1.0) * 0x1p-53; }
/* uniform in [0, 1) */
SYN_FN double u01(uint64_t x) { return (double)(x >> 11) * 0x1p-53; }

/* ------------------------------------------------- elementary functions */
/* Power series in Horner form. The coefficients are constant expressions
 * (1/(2k+1), 1/n!) folded at compile time with correct rounding, and only
 * +, -, *, / are used at run time, so results are identical on every IEEE-754
 * machine (compiled without fused multiply-add). */
#define SYN_LN2_HI 6.93147180369123816490e-01 /* 0x3FE62E42FEE00000 */
#define SYN_LN2_LO 1.90821492927058770002e-10
#define SYN_PI_4 0.78539816339744830962

/* ln(x), x > 0: x = m 2^e with m in [sqrt(1/2), sqrt(2)); with
 * s = (m-1)/(m+1), ln m = 2 (s + s^3/3 + s^5/5 + ...), |s| <= 0.172. */
SYN_FN double syn_log(double x)
{
    int e;
    double m = frexp(x, &e); /* m in [0.5, 1) */
    if (m < 0.70710678118654752440) {
        m *= 2.0;
        e -= 1;
    }
    double s = (m - 1.0) / (m + 1.0);
    double z = s * s;
    double p = 1.0 / 25.0;
    p = p * z + 1.0 / 23.0;
    p = p * z + 1.0 / 21.0;
    p = p * z + 1.0 / 19.0;
    p = p * z + 1.0 / 17.0;
    p = p * z + 1.0 / 15.0;
    p = p * z + 1.0 / 13.0;
    p = p * z + 1.0 / 11.0;
    p = p * z + 1.0 / 9.0;
    p = p * z + 1.0 / 7.0;
    p = p * z + 1.0 / 5.0;
    p = p * z + 1.0 / 3.0;
    p = p * z + 1.0;
    double ln_m = 2.0 * (s * p);
    return ((double)e * SYN_LN2_LO + ln_m) + (double)e * SYN_LN2_HI;
}

/* exp(x): x = n ln2 + r, |r| <= ln2/2, Taylor series of exp(r) to r^20. */
SYN_FN double syn_exp(double x)
{
    double n = nearbyint(x / 0.69314718055994530942);
    double r = (x - n * SYN_LN2_HI) - n * SYN_LN2_LO;
    double p = 1.0 / 2432902008176640000.0; /* 1/20! */
    p = p * r + 1.0 / 121645100408832000.0;
    p = p * r + 1.0 / 6402373705728000.0;
    p = p * r + 1.0 / 355687428096000.0;
    p = p * r + 1.0 / 20922789888000.0;
    p = p * r + 1.0 / 1307674368000.0;
    p = p * r + 1.0 / 87178291200.0;
    p = p * r + 1.0 / 6227020800.0;
    p = p * r + 1.0 / 479001600.0;
    p = p * r + 1.0 / 39916800.0;
    p = p * r + 1.0 / 3628800.0;
    p = p * r + 1.0 / 362880.0;
    p = p * r + 1.0 / 40320.0;
    p = p * r + 1.0 / 5040.0;
    p = p * r + 1.0 / 720.0;
    p = p * r + 1.0 / 120.0;
    p = p * r + 1.0 / 24.0;
    p = p * r + 1.0 / 6.0;
    p = p * r + 1.0 / 2.0;
    p = p * r + 1.0;
    p = p * r + 1.0;
    return ldexp(p, (int)n);
}

/* sin and cos of y in [0, pi/4]: Taylor series to y^17 and y^18. */
SYN_FN void syn_sincos_small(double y, double *s, double *c)
{
    double z = y * y;
    double ps = -1.0 / 355687428096000.0;  /* -1/17! */
    ps = ps * z + 1.0 / 1307674368000.0;   /* 1/15! */
    ps = ps * z - 1.0 / 6227020800.0;      /* -1/13! */
    ps = ps * z + 1.0 / 39916800.0;        /* 1/11! */
    ps = ps * z - 1.0 / 362880.0;          /* -1/9! */
    ps = ps * z + 1.0 / 5040.0;            /* 1/7! */
    ps = ps * z - 1.0 / 120.0;             /* -1/5! */
    ps = ps * z + 1.0 / 6.0;               /* 1/3! */
    *s = y - y * (z * ps);
    double pc = 1.0 / 6402373705728000.0;  /* 1/18! */
    pc = pc * z - 1.0 / 20922789888000.0;  /* -1/16! */
    pc = pc * z + 1.0 / 87178291200.0;     /* 1/14! */
    pc = pc * z - 1.0 / 479001600.0;       /* -1/12! */
    pc = pc * z + 1.0 / 3628800.0;         /* 1/10! */
    pc = pc * z - 1.0 / 40320.0;           /* -1/8! */
    pc = pc * z + 1.0 / 720.0;             /* 1/6! */
    pc = pc * z - 1.0 / 24.0;              /* -1/4! */
    pc = pc * z + 1.0 / 2.0;               /* 1/2! */
    *c = 1.0 - z * pc;
}

/* (cos 2 pi u, sin 2 pi u) for u in [0, 1): octant reduction, v = 8u. */
SYN_FN void syn_cis(double u, double *c, double *s)
{
    double v = u * 8.0; /* exact */
    int o = (int)v;
    double f = v - (double)o; /* exact, in [0, 1) */
    /* angle within the octant: (o + f) * pi/4; reflect odd octants */
    double y = (o & 1) ? (1.0 - f) * SYN_PI_4 : f * SYN_PI_4;
    double sy, cy;
    syn_sincos_small(y, &sy, &cy);
    /* for an odd octant the angle is (o + 1) pi/4 - y */
    double cs, sn;
    switch (o) {
    case 0: cs = cy; sn = sy; break;    /* y */
    case 1: cs = sy; sn = cy; break;    /* pi/2 - y */
    case 2: cs = -sy; sn = cy; break;   /* pi/2 + y */
    case 3: cs = -cy; sn = sy; break;   /* pi - y */
    case 4: cs = -cy; sn = -sy; break;  /* pi + y */
    case 5: cs = -sy; sn = -cy; break;  /* 3pi/2 - y */
    case 6: cs = sy; sn = -cy; break;   /* 3pi/2 + y */
    default: cs = cy; sn = -sy; break;  /* 2pi - y */
    }
    *c = cs;
    *s = sn;
}

/* Two independent N(0,1) from two uniforms (Box-Muller). */
SYN_FN void syn_normal2(uint64_t key, uint64_t i, double *z0, double *z1)
{
    double u1 = u01_open0(sm64(key, 2 * i));
    double u2 = u01(sm64(key, 2 * i + 1));
    double rad = sqrt(-2.0 * syn_log(u1));
    double c, s;
    syn_cis(u2, &c, &s);
    *z0 = rad * c;
    *z1 = rad * s;
}

SYN_FN double syn_normal(uint64_t key, uint64_t i)
{
    double a, b;
    syn_normal2(key, i, &a, &b);
    return a;
}

/* ------------------------------------------------- double -> fp16 bits */
SYN_FN uint16_t syn_to_half(double x)
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
SYN_FN uint64_t elem_ctr(int c, int t) { return ((uint64_t)c << 32) | (uint64_t)t; }

SYN_FN uint64_t slice_key(const syn_params *p, int kv, int layer)
{
    uint64_t k0 = sm64(p->seed, 0);
    return sm64(k0, ((uint64_t)kv << 32) | (uint64_t)layer);
}


/* AR(1) value at t: x_0 = sigma z_0 / sqrt(1 - rho^2), x_t = rho x_{t-1} + sigma z_t. */
SYN_FN double syn_ar1_next(const syn_params *p, uint64_t key_val, int c, int t, double sigma,
                           double stat, double prev)
{
    double z = syn_normal(key_val, elem_ctr(c, t));
    return t == 0 ? sigma * z / stat : p->rho * prev + sigma * z;
}

/* Student-t(3) value: sigma Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3). */
SYN_FN double syn_student_value(uint64_t key_val, int c, int t, double sigma)
{
    uint64_t i = elem_ctr(c, t) * 2;
    double z0, z1, z2, z3;
    syn_normal2(key_val, i, &z0, &z1);
    syn_normal2(key_val, i + 1, &z2, &z3);
    double chi = (z1 * z1 + z2 * z2) + z3 * z3;
    return sigma * z0 / sqrt(chi / 3.0);
}

#endif
