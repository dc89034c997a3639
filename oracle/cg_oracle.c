/*
 * cg_oracle.c - CPU oracle for the CacheGen KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY (see cg_oracle.h): slow, single-threaded, written
 * to be read against the page and the codec specification in cg_oracle.h.
 * Compiled with -O2 -ffp-contract=off so every binary32 operation is rounded
 * on its own.
 *
 * Each step follows the order the page gives: quantise [CG §2.3(1)], count
 * and build the CDF [CG §2.3(2)], code per chunk [CG §2.3(3), §1.2(3)], decode
 * [CG §2.4(1)] and dequantise [CG §2.4(2)].
 */
#include "cg_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORC_M 65536u

float orc_half_to_float(uint16_t h)
{
    /* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    float mag;
    if (e == 0)
        mag = ldexpf((float)f, -24); /* subnormal: f * 2^-24, exact */
    else if (e == 31)
        mag = f ? NAN : INFINITY;
    else
        mag = ldexpf((float)(f | 0x400), e - 25); /* 1.f * 2^(e-15) */
    return sign ? -mag : mag;
}

/* [CG §2.3(1)] torch_quant_vectorized on one group: MAX = bins // 2 - 1,
 * max1 = amax |x| over the group, factor = MAX / max1,
 * xq = round(x * factor + MAX). Arithmetic in binary32 (specification Q). */
int orc_quantize_group(const uint16_t *x, int64_t C, int bins, uint8_t *q,
                       uint16_t *max1_out)
{
    if (bins < 4 || bins > 256 || C < 1)
        return ORC_ERR_ARG;
    int MAX = bins / 2 - 1;
    float max1 = 0.0f;
    uint16_t max1_bits = 0;
    for (int64_t c = 0; c < C; c++) {
        float xv = orc_half_to_float(x[c]);
        if (!isfinite(xv))
            return ORC_ERR_NONFINITE;
        float a = fabsf(xv);
        if (a > max1) {
            max1 = a;
            max1_bits = (uint16_t)(x[c] & 0x7FFF);
        }
    }
    *max1_out = max1_bits;
    if (max1 == 0.0f) {
        /* all-zero group: every value sits at the offset MAX */
        for (int64_t c = 0; c < C; c++)
            q[c] = (uint8_t)MAX;
        return ORC_OK;
    }
    float factor = (float)MAX / max1;
    for (int64_t c = 0; c < C; c++) {
        float xv = orc_half_to_float(x[c]);
        float scaled = xv * factor;
        float y = scaled + (float)MAX;
        float r = rintf(y);
        if (r < 0.0f)
            r = 0.0f;
        if (r > (float)(2 * MAX))
            r = (float)(2 * MAX);
        q[c] = (uint8_t)r;
    }
    return ORC_OK;
}

/* [CG §2.4(2)] do_dequantize: t - MAX, to float, divide by MAX, times max1. */
float orc_dequantize_value(uint8_t q, int bins, uint16_t max1)
{
    int MAX = bins / 2 - 1;
    float centred = (float)((int)q - MAX);
    float unit = centred / (float)MAX;
    return unit * orc_half_to_float(max1);
}

/* [CG §2.3(2)] symbol frequencies -> CDF, normalised to a 16-bit total with
 * every symbol given a frequency of at least one (specification F). */
int orc_cdf_from_counts(const uint32_t *n, int A, uint32_t Tk, uint16_t *cdf)
{
    if (A < 2 || A > 256 || Tk < 1)
        return ORC_ERR_ARG;
    uint32_t f[256];
    uint64_t sum = 0;
    int best = 0;
    for (int s = 0; s < A; s++) {
        f[s] = 1u + (uint32_t)(((uint64_t)n[s] * (ORC_M - (uint32_t)A)) / Tk);
        sum += f[s];
        if (n[s] > n[best])
            best = s;
    }
    if (sum > ORC_M)
        return ORC_ERR_ARG; /* counts do not add up to Tk */
    f[best] += (uint32_t)(ORC_M - sum);
    uint32_t acc = 0;
    for (int s = 0; s < A; s++) {
        cdf[s] = (uint16_t)acc;
        acc += f[s];
    }
    return acc == ORC_M ? ORC_OK : ORC_ERR_ARG;
}

/* Carry into the bytes already emitted: the last byte gets +1; a 0xFF byte
 * turns into 0x00 and passes the carry on to the byte before it. */
static void orc_propagate_carry(uint8_t *out, int64_t pos)
{
    int64_t i = pos - 1;
    while (i >= 0 && out[i] == 0xFF) {
        out[i] = 0x00;
        i--;
    }
    if (i >= 0)
        out[i] = (uint8_t)(out[i] + 1);
}

static uint32_t orc_cdf_at(const uint16_t *row, int A, int s)
{
    return s >= A ? ORC_M : (uint32_t)row[s];
}

/* [CG §1.2(3)] arithmetic coding, in the range-coder form of specification R. */
int64_t orc_encode_stream(const uint8_t *sym, int64_t n, const uint16_t *cdf,
                          int64_t row_stride, int A, uint8_t *out, int64_t cap)
{
    if (A < 2 || n < 0 || cap < 0)
        return -1;
    uint32_t low = 0, range = 0xFFFFFFFFu;
    int64_t pos = 0;
    for (int64_t i = 0; i < n; i++) {
        const uint16_t *row = cdf + i * row_stride;
        int s = sym[i];
        if (s >= A)
            return -1;
        uint32_t lo = orc_cdf_at(row, A, s);
        uint32_t f = orc_cdf_at(row, A, s + 1) - lo;
        uint32_t r = range >> 16;
        uint32_t t = low + r * lo;
        if (t < low)
            orc_propagate_carry(out, pos);
        low = t;
        range = r * f;
        while (range < (1u << 24)) {
            if (pos >= cap)
                return -1;
            out[pos++] = (uint8_t)(low >> 24);
            low <<= 8;
            range <<= 8;
        }
    }
    uint32_t v = low + 0x00FFFFFFu;
    if (v < low)
        orc_propagate_carry(out, pos);
    if (pos >= cap)
        return -1;
    out[pos++] = (uint8_t)(v >> 24);
    return pos;
}

/* [CG §2.4(1)] decode_function_gpu: recover the integer symbols of one
 * stream with the CDFs sent alongside it (specification R, decoder side). */
int orc_decode_stream(const uint8_t *in, int64_t len, int64_t n,
                      const uint16_t *cdf, int64_t row_stride, int A,
                      uint8_t *sym, int64_t *consumed)
{
    if (A < 2 || n < 0 || len < 0)
        return ORC_ERR_ARG;
    int64_t pos = 0;
    uint32_t range = 0xFFFFFFFFu, code = 0;
    for (int b = 0; b < 4; b++) {
        uint32_t byte = pos < len ? in[pos] : 0;
        pos++;
        code = (code << 8) | byte;
    }
    for (int64_t i = 0; i < n; i++) {
        const uint16_t *row = cdf + i * row_stride;
        uint32_t r = range >> 16;
        int s = 0;
        for (int c = 1; c < A; c++)
            if ((uint64_t)r * row[c] <= code)
                s = c;
        uint32_t lo = orc_cdf_at(row, A, s);
        uint32_t f = orc_cdf_at(row, A, s + 1) - lo;
        sym[i] = (uint8_t)s;
        code -= r * lo;
        range = r * f;
        while (range < (1u << 24)) {
            uint32_t byte = pos < len ? in[pos] : 0;
            pos++;
            code = (code << 8) | byte;
            range <<= 8;
        }
    }
    if (consumed)
        *consumed = pos;
    return pos == len + 3 ? ORC_OK : ORC_ERR_CORRUPT;
}

int64_t orc_num_streams(int L, int T) { return 2 * (int64_t)L * T; }

static int orc_chunk_tokens(int T, int Tc, int k)
{
    int rest = T - k * Tc;
    return rest < Tc ? rest : Tc;
}

int64_t orc_cdf_elems(int L, int T, int C, int Tc, int A_k, int A_v)
{
    int64_t nch = (T + Tc - 1) / Tc;
    return nch * (int64_t)L * C * (A_k + A_v);
}

int64_t orc_cdf_offset(int L, int C, int A_k, int A_v, int k, int kv, int l,
                       int c)
{
    int64_t chunk = (int64_t)k * L * C * (A_k + A_v);
    int64_t tensor = kv ? (int64_t)L * C * A_k : 0;
    int A = kv ? A_v : A_k;
    return chunk + tensor + ((int64_t)l * C + c) * A;
}

int64_t orc_stream_id(int L, int T, int Tc, int k, int kv, int l, int tl)
{
    int Tck = orc_chunk_tokens(T, Tc, k);
    return 2 * (int64_t)L * Tc * k + ((int64_t)kv * L + l) * Tck + tl;
}

int orc_alphabet(const int32_t *bins, int L)
{
    int a = 0;
    for (int l = 0; l < L; l++)
        if (bins[l] > a)
            a = bins[l];
    return a;
}

static int orc_check_shape(int L, int T, int C)
{
    return L >= 1 && T >= 1 && C >= 1;
}

/* [CG §2.3(1)] with the layer-wise bins of [CG §2.2]: every (kv, l, t) group
 * is quantised with its layer's bins. */
int orc_quantize(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                 int64_t layer_stride, const int32_t *bins_k,
                 const int32_t *bins_v, uint8_t *sym, uint16_t *max1)
{
    if (!orc_check_shape(L, T, C))
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    for (int kv = 0; kv < 2; kv++) {
        const uint16_t *x = kv ? v : k;
        const int32_t *bins = kv ? bins_v : bins_k;
        for (int l = 0; l < L; l++)
            for (int t = 0; t < T; t++) {
                int64_t g = ((int64_t)kv * L + l) * T + t;
                int st = orc_quantize_group(
                    x + (int64_t)l * layer_stride + (int64_t)t * C, C, bins[l],
                    sym + g * C, max1 + g);
                if (st != ORC_OK)
                    return st;
            }
    }
    return ORC_OK;
}

/* [CG §2.3(2)] calculate_cdf, scoped per (chunk, kv, layer, channel) over the
 * chunk's tokens [CG §2.3(3)]. */
int orc_calculate_cdf(const uint8_t *sym, int L, int T, int C, int Tc,
                      int A_k, int A_v, uint16_t *cdf)
{
    if (!orc_check_shape(L, T, C) || Tc < 1)
        return ORC_ERR_ARG;
    int nch = (T + Tc - 1) / Tc;
    uint32_t n[256];
    for (int k = 0; k < nch; k++) {
        int Tk = orc_chunk_tokens(T, Tc, k);
        for (int kv = 0; kv < 2; kv++) {
            int A = kv ? A_v : A_k;
            for (int l = 0; l < L; l++)
                for (int c = 0; c < C; c++) {
                    memset(n, 0, sizeof n);
                    for (int tl = 0; tl < Tk; tl++) {
                        int64_t t = (int64_t)k * Tc + tl;
                        uint8_t s = sym[(((int64_t)kv * L + l) * T + t) * C + c];
                        if (s >= A)
                            return ORC_ERR_ARG;
                        n[s]++;
                    }
                    int st = orc_cdf_from_counts(
                        n, A, (uint32_t)Tk,
                        cdf + orc_cdf_offset(L, C, A_k, A_v, k, kv, l, c));
                    if (st != ORC_OK)
                        return st;
                }
        }
    }
    return ORC_OK;
}

/* [CG §2.3(3), §1.2(3)] code every (chunk, kv, layer, token) stream over its
 * channels and pack the streams in stream-id order. */
int orc_encode(const uint8_t *sym, const uint16_t *cdf, int L, int T, int C,
               int Tc, int A_k, int A_v, uint8_t *packed, uint64_t capacity,
               uint32_t *len, uint64_t *off)
{
    if (!orc_check_shape(L, T, C) || Tc < 1)
        return ORC_ERR_ARG;
    int nch = (T + Tc - 1) / Tc;
    int64_t cap = 2 * (int64_t)C + 8;
    uint8_t *buf = (uint8_t *)malloc((size_t)cap);
    if (!buf)
        return ORC_ERR_NOMEM;
    uint64_t total = 0;
    int status = ORC_OK;
    for (int k = 0; k < nch; k++) {
        int Tk = orc_chunk_tokens(T, Tc, k);
        for (int kv = 0; kv < 2; kv++) {
            int A = kv ? A_v : A_k;
            for (int l = 0; l < L; l++) {
                const uint16_t *rows =
                    cdf + orc_cdf_offset(L, C, A_k, A_v, k, kv, l, 0);
                for (int tl = 0; tl < Tk; tl++) {
                    int64_t t = (int64_t)k * Tc + tl;
                    int64_t sid = orc_stream_id(L, T, Tc, k, kv, l, tl);
                    const uint8_t *s =
                        sym + (((int64_t)kv * L + l) * T + t) * C;
                    int64_t n = orc_encode_stream(s, C, rows, A, A, buf, cap);
                    if (n < 0) {
                        free(buf);
                        return ORC_ERR_ARG;
                    }
                    off[sid] = total;
                    len[sid] = (uint32_t)n;
                    /* bytes at or past capacity are not written */
                    if (total + (uint64_t)n <= capacity) {
                        memcpy(packed + total, buf, (size_t)n);
                    } else {
                        if (total < capacity)
                            memcpy(packed + total, buf, (size_t)(capacity - total));
                        status = ORC_ERR_CAPACITY;
                    }
                    total += (uint64_t)n;
                }
            }
        }
    }
    off[orc_num_streams(L, T)] = total;
    free(buf);
    return status;
}

int orc_decode(const uint8_t *packed, const uint64_t *off, const uint32_t *len,
               const uint16_t *cdf, int L, int T, int C, int Tc, int A_k,
               int A_v, uint8_t *sym)
{
    if (!orc_check_shape(L, T, C) || Tc < 1)
        return ORC_ERR_ARG;
    int nch = (T + Tc - 1) / Tc;
    int status = ORC_OK;
    for (int k = 0; k < nch; k++) {
        int Tk = orc_chunk_tokens(T, Tc, k);
        for (int kv = 0; kv < 2; kv++) {
            int A = kv ? A_v : A_k;
            for (int l = 0; l < L; l++) {
                const uint16_t *rows =
                    cdf + orc_cdf_offset(L, C, A_k, A_v, k, kv, l, 0);
                for (int tl = 0; tl < Tk; tl++) {
                    int64_t t = (int64_t)k * Tc + tl;
                    int64_t sid = orc_stream_id(L, T, Tc, k, kv, l, tl);
                    int64_t used = 0;
                    int st = orc_decode_stream(
                        packed + off[sid], len[sid], C, rows, A, A,
                        sym + (((int64_t)kv * L + l) * T + t) * C, &used);
                    if (st != ORC_OK)
                        status = st;
                }
            }
        }
    }
    return status;
}

/* [CG §2.4(2)] do_dequantize over the whole tensor, output binary32. */
int orc_dequantize(const uint8_t *sym, const uint16_t *max1, int L, int T,
                   int C, const int32_t *bins_k, const int32_t *bins_v,
                   float *out_k, float *out_v)
{
    if (!orc_check_shape(L, T, C))
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    for (int kv = 0; kv < 2; kv++) {
        float *out = kv ? out_v : out_k;
        const int32_t *bins = kv ? bins_v : bins_k;
        for (int l = 0; l < L; l++)
            for (int t = 0; t < T; t++) {
                int64_t g = ((int64_t)kv * L + l) * T + t;
                for (int c = 0; c < C; c++)
                    out[((int64_t)l * T + t) * C + c] = orc_dequantize_value(
                        sym[g * C + c], bins[l], max1[g]);
            }
    }
    return ORC_OK;
}

int orc_compress(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                 int Tc, int64_t layer_stride, const int32_t *bins_k,
                 const int32_t *bins_v, uint16_t *max1, uint16_t *cdf,
                 uint8_t *packed, uint64_t capacity, uint32_t *len,
                 uint64_t *off)
{
    if (!orc_check_shape(L, T, C) || Tc < 1)
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    uint8_t *sym = (uint8_t *)malloc((size_t)(2 * (int64_t)L * T * C));
    if (!sym)
        return ORC_ERR_NOMEM;
    int st = orc_quantize(k, v, L, T, C, layer_stride, bins_k, bins_v, sym,
                          max1);
    int A_k = orc_alphabet(bins_k, L), A_v = orc_alphabet(bins_v, L);
    if (st == ORC_OK)
        st = orc_calculate_cdf(sym, L, T, C, Tc, A_k, A_v, cdf);
    if (st == ORC_OK)
        st = orc_encode(sym, cdf, L, T, C, Tc, A_k, A_v, packed, capacity, len,
                        off);
    free(sym);
    return st;
}

int orc_decompress(const uint8_t *packed, const uint64_t *off,
                   const uint32_t *len, const uint16_t *cdf,
                   const uint16_t *max1, int L, int T, int C, int Tc,
                   const int32_t *bins_k, const int32_t *bins_v, float *out_k,
                   float *out_v)
{
    if (!orc_check_shape(L, T, C) || Tc < 1)
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    uint8_t *sym = (uint8_t *)malloc((size_t)(2 * (int64_t)L * T * C));
    if (!sym)
        return ORC_ERR_NOMEM;
    int A_k = orc_alphabet(bins_k, L), A_v = orc_alphabet(bins_v, L);
    int st = orc_decode(packed, off, len, cdf, L, T, C, Tc, A_k, A_v, sym);
    if (st == ORC_OK)
        st = orc_dequantize(sym, max1, L, T, C, bins_k, bins_v, out_k, out_v);
    free(sym);
    return st;
}

/* ---- format 2: side information as symbol counts (specification S, F2) ---- */

int orc_alphabet_v2(int bins)
{
    return 2 * (bins / 2 - 1) + 1;
}

/* Bytes of one chunk's records of one tensor: C records per layer. */
static int64_t orc_rec_tensor_bytes(int L, int C, const int32_t *bins)
{
    int64_t b = 0;
    for (int l = 0; l < L; l++)
        b += (int64_t)C * orc_alphabet_v2(bins[l]);
    return b;
}

int64_t orc_rec_bytes(int L, int T, int C, int Tc, const int32_t *bins_k,
                      const int32_t *bins_v)
{
    if (!orc_check_shape(L, T, C) || Tc < 1)
        return -1;
    if (!bins_v)
        bins_v = bins_k;
    int64_t nch = (T + Tc - 1) / Tc;
    return nch * (orc_rec_tensor_bytes(L, C, bins_k) +
                  orc_rec_tensor_bytes(L, C, bins_v));
}

int64_t orc_rec_offset(int L, int C, const int32_t *bins_k,
                       const int32_t *bins_v, int k, int kv, int l, int c)
{
    if (!bins_v)
        bins_v = bins_k;
    int64_t per_k = orc_rec_tensor_bytes(L, C, bins_k);
    int64_t o = (int64_t)k * (per_k + orc_rec_tensor_bytes(L, C, bins_v));
    if (kv)
        o += per_k;
    const int32_t *bins = kv ? bins_v : bins_k;
    for (int j = 0; j < l; j++)
        o += (int64_t)C * orc_alphabet_v2(bins[j]);
    return o + (int64_t)c * orc_alphabet_v2(bins[l]);
}

/* The mode: the largest count, the smallest symbol on ties. */
static int orc_mode(const uint32_t *n, int A)
{
    int best = 0;
    for (int s = 1; s < A; s++)
        if (n[s] > n[best])
            best = s;
    return best;
}

int orc_record_from_counts(const uint32_t *n, int A, uint8_t *rec)
{
    if (A < 2 || A > 256)
        return ORC_ERR_ARG;
    int m = orc_mode(n, A);
    rec[0] = (uint8_t)m;
    int i = 1;
    for (int s = 0; s < A; s++) {
        if (s == m)
            continue;
        if (n[s] > 255)
            return ORC_ERR_ARG;
        rec[i++] = (uint8_t)n[s];
    }
    return ORC_OK;
}

int orc_counts_from_record(const uint8_t *rec, int A, uint32_t Tk, uint32_t *n)
{
    if (A < 2 || A > 256 || Tk < 1)
        return ORC_ERR_ARG;
    int m = rec[0];
    if (m >= A)
        return ORC_ERR_CORRUPT;
    uint32_t others = 0;
    int i = 1;
    for (int s = 0; s < A; s++) {
        if (s == m)
            continue;
        n[s] = rec[i++];
        others += n[s];
    }
    if (others > Tk)
        return ORC_ERR_CORRUPT;
    n[m] = Tk - others;
    return ORC_OK;
}

/* F with the remainder given to `mode` rather than to the argmax. */
int orc_cdf_from_counts_mode(const uint32_t *n, int A, uint32_t Tk, int mode,
                             uint16_t *cdf)
{
    if (A < 2 || A > 256 || Tk < 1 || mode < 0 || mode >= A)
        return ORC_ERR_ARG;
    uint32_t f[256];
    uint64_t sum = 0;
    for (int s = 0; s < A; s++) {
        f[s] = 1u + (uint32_t)(((uint64_t)n[s] * (ORC_M - (uint32_t)A)) / Tk);
        sum += f[s];
    }
    if (sum > ORC_M)
        return ORC_ERR_ARG;
    f[mode] += (uint32_t)(ORC_M - sum);
    uint32_t acc = 0;
    for (int s = 0; s < A; s++) {
        cdf[s] = (uint16_t)acc;
        acc += f[s];
    }
    return acc == ORC_M ? ORC_OK : ORC_ERR_ARG;
}

/* [CG §2.3(1)-(3), §1.2(3)] format 2: quantise, count per (chunk, kv, layer,
 * channel), store the counts as records, build each CDF over the layer's own
 * alphabet and code the streams as in format 1. */
/* Format 2 coding of given symbols: counts -> records and CDFs -> streams. */
static int orc_code_v2(const uint8_t *sym, int L, int T, int C, int Tc,
                       const int32_t *bins_k, const int32_t *bins_v,
                       uint8_t *rec, uint8_t *packed, uint64_t capacity,
                       uint32_t *len, uint64_t *off)
{
    uint16_t *rows = (uint16_t *)malloc((size_t)C * 256 * sizeof(uint16_t));
    int64_t cap1 = 2 * (int64_t)C + 8;
    uint8_t *buf = (uint8_t *)malloc((size_t)cap1);
    if (!rows || !buf) {
        free(rows), free(buf);
        return ORC_ERR_NOMEM;
    }
    int status = ORC_OK;
    int nch = (T + Tc - 1) / Tc;
    uint64_t total = 0;
    for (int kc = 0; kc < nch; kc++) {
        int Tk = orc_chunk_tokens(T, Tc, kc);
        for (int kv = 0; kv < 2; kv++) {
            const int32_t *bins = kv ? bins_v : bins_k;
            for (int l = 0; l < L; l++) {
                int A = orc_alphabet_v2(bins[l]);
                /* counts -> record and CDF row per channel */
                for (int c = 0; c < C; c++) {
                    uint32_t n[256] = {0};
                    for (int tl = 0; tl < Tk; tl++) {
                        int64_t t = (int64_t)kc * Tc + tl;
                        n[sym[(((int64_t)kv * L + l) * T + t) * C + c]]++;
                    }
                    uint8_t *r = rec + orc_rec_offset(L, C, bins_k, bins_v, kc, kv, l, c);
                    int st = orc_record_from_counts(n, A, r);
                    if (st == ORC_OK)
                        st = orc_cdf_from_counts_mode(n, A, (uint32_t)Tk, r[0],
                                                      rows + (int64_t)c * A);
                    if (st != ORC_OK) {
                        free(rows), free(buf);
                        return st;
                    }
                }
                /* one stream per token of the chunk */
                for (int tl = 0; tl < Tk; tl++) {
                    int64_t t = (int64_t)kc * Tc + tl;
                    int64_t sid = orc_stream_id(L, T, Tc, kc, kv, l, tl);
                    const uint8_t *s = sym + (((int64_t)kv * L + l) * T + t) * C;
                    int64_t n = orc_encode_stream(s, C, rows, A, A, buf, cap1);
                    if (n < 0) {
                        free(rows), free(buf);
                        return ORC_ERR_ARG;
                    }
                    off[sid] = total;
                    len[sid] = (uint32_t)n;
                    if (total + (uint64_t)n <= capacity) {
                        memcpy(packed + total, buf, (size_t)n);
                    } else {
                        if (total < capacity)
                            memcpy(packed + total, buf, (size_t)(capacity - total));
                        status = ORC_ERR_CAPACITY;
                    }
                    total += (uint64_t)n;
                }
            }
        }
    }
    off[orc_num_streams(L, T)] = total;
    free(rows), free(buf);
    return status;
}

int orc_compress_v2(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                    int Tc, int64_t layer_stride, const int32_t *bins_k,
                    const int32_t *bins_v, uint16_t *max1, uint8_t *rec,
                    uint8_t *packed, uint64_t capacity, uint32_t *len,
                    uint64_t *off)
{
    return orc_compress_ex(k, v, L, T, C, Tc, 1, 2, layer_stride, bins_k,
                           bins_v, max1, rec, packed, capacity, len, off);
}

/* Format 2 decoding: records -> CDFs -> symbols [2][L][T][C]. */
static int orc_decode_v2(const uint8_t *packed, const uint64_t *off,
                         const uint32_t *len, const uint8_t *rec, int L, int T,
                         int C, int Tc, const int32_t *bins_k,
                         const int32_t *bins_v, uint8_t *sym)
{
    uint16_t *rows = (uint16_t *)malloc((size_t)C * 256 * sizeof(uint16_t));
    if (!rows)
        return ORC_ERR_NOMEM;
    int status = ORC_OK;
    int nch = (T + Tc - 1) / Tc;
    for (int kc = 0; kc < nch; kc++) {
        int Tk = orc_chunk_tokens(T, Tc, kc);
        for (int kv = 0; kv < 2; kv++) {
            const int32_t *bins = kv ? bins_v : bins_k;
            for (int l = 0; l < L; l++) {
                int A = orc_alphabet_v2(bins[l]);
                for (int c = 0; c < C; c++) {
                    const uint8_t *r = rec + orc_rec_offset(L, C, bins_k, bins_v, kc, kv, l, c);
                    uint32_t n[256];
                    int st = orc_counts_from_record(r, A, (uint32_t)Tk, n);
                    if (st == ORC_OK)
                        st = orc_cdf_from_counts_mode(n, A, (uint32_t)Tk, r[0],
                                                      rows + (int64_t)c * A);
                    if (st != ORC_OK) {
                        free(rows);
                        return st;
                    }
                }
                for (int tl = 0; tl < Tk; tl++) {
                    int64_t t = (int64_t)kc * Tc + tl;
                    int64_t sid = orc_stream_id(L, T, Tc, kc, kv, l, tl);
                    int64_t used = 0;
                    int st = orc_decode_stream(
                        packed + off[sid], len[sid], C, rows, A, A,
                        sym + (((int64_t)kv * L + l) * T + t) * C, &used);
                    if (st != ORC_OK)
                        status = st;
                }
            }
        }
    }
    free(rows);
    return status;
}

int orc_decompress_v2(const uint8_t *packed, const uint64_t *off,
                      const uint32_t *len, const uint8_t *rec,
                      const uint16_t *max1, int L, int T, int C, int Tc,
                      const int32_t *bins_k, const int32_t *bins_v,
                      float *out_k, float *out_v)
{
    return orc_decompress_ex(packed, off, len, rec, max1, L, T, C, Tc, 1, 2,
                             bins_k, bins_v, out_k, out_v);
}

/* ---- serving layouts: binary16 output ---------------------------------- */

/* binary32 -> binary16 bits, round to nearest, ties to even (IEEE 754):
 * finite values keep 11 significant bits (fewer below 2^-14, where the
 * spacing is 2^-24); too large values become infinity, NaN stays NaN. */
uint16_t orc_float_to_half(float x)
{
    uint32_t b;
    memcpy(&b, &x, 4);
    uint16_t sign = (uint16_t)((b >> 16) & 0x8000u);
    uint32_t e = (b >> 23) & 0xFFu;
    uint32_t m = b & 0x7FFFFFu;
    if (e == 0xFFu) /* infinity or NaN */
        return (uint16_t)(sign | 0x7C00u | (m ? 0x200u : 0u));
    int exp = (int)e - 127; /* unbiased; x = 1.m * 2^exp for normal x */
    if (e == 0)             /* binary32 subnormal: far below half's smallest */
        return sign;
    uint32_t sig = m | 0x800000u; /* 24-bit significand, value sig * 2^(exp-23) */
    /* half keeps the bits down to 2^-24 (subnormal range) or to 2^(exp-10) */
    int lsb = exp - 10 < -24 ? -24 : exp - 10; /* exponent of the last kept bit */
    int shift = lsb - (exp - 23);              /* bits of sig to drop, >= 13 */
    if (shift > 25)
        return sign; /* below half the smallest subnormal: rounds to zero */
    uint32_t kept = sig >> shift;
    uint32_t rest = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rest > half || (rest == half && (kept & 1u)))
        kept++; /* may carry into the next binade; handled by the sum below */
    /* value = kept * 2^lsb; encode: normal when lsb > -24 or kept >= 2^10 */
    uint32_t h;
    if (lsb == -24) {
        h = kept; /* subnormal (kept < 2^10) or, after rounding, 2^10 = smallest normal */
    } else {
        /* kept in [2^10, 2^11]; exponent field = lsb + 10 + 15 */
        uint32_t ef = (uint32_t)(lsb + 10 + 15);
        h = (ef << 10) + (kept - 0x400u); /* kept == 2^11 rolls into the next exponent */
    }
    if (h >= 0x7C00u)
        h = 0x7C00u; /* overflow to infinity */
    return (uint16_t)(sign | h);
}

/* [CG §2.4(2)] dequantisation with binary16 output: the binary32 value of D
 * rounded to nearest-even binary16 (no overflow: |x^| <= max1). */
int orc_dequantize_half(const uint8_t *sym, const uint16_t *max1, int L, int T,
                        int C, const int32_t *bins_k, const int32_t *bins_v,
                        uint16_t *out_k, uint16_t *out_v)
{
    if (!orc_check_shape(L, T, C))
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    for (int kv = 0; kv < 2; kv++) {
        uint16_t *out = kv ? out_v : out_k;
        const int32_t *bins = kv ? bins_v : bins_k;
        for (int l = 0; l < L; l++)
            for (int t = 0; t < T; t++) {
                int64_t g = ((int64_t)kv * L + l) * T + t;
                for (int c = 0; c < C; c++)
                    out[((int64_t)l * T + t) * C + c] = orc_float_to_half(
                        orc_dequantize_value(sym[g * C + c], bins[l], max1[g]));
            }
    }
    return ORC_OK;
}

/* ---- token-locality delta (specification G) ------------------------------ */

uint16_t orc_half_up(float m)
{
    if (!(m <= 65504.0f))
        return 0x7BFFu; /* above the largest finite binary16 */
    uint16_t h = orc_float_to_half(m); /* nearest; at most one step below m */
    if (h >= 0x7C00u)
        return 0x7BFFu;
    if (orc_half_to_float(h) < m)
        h++; /* the next binary16 up (positive values order like their bits) */
    return h;
}

void orc_floats_to_half(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_float_to_half(x[i]);
}

/* [CG §1.2(1)] QD: one non-anchor row, given its anchor's reconstruction. */
static int orc_quantize_delta_row(const uint16_t *x, const float *anchor, int C,
                                  int bins, float *d, uint8_t *q,
                                  uint16_t *max1_out)
{
    int MAX = bins / 2 - 1;
    float m = 0.0f;
    for (int c = 0; c < C; c++) {
        float xv = orc_half_to_float(x[c]);
        if (!isfinite(xv))
            return ORC_ERR_NONFINITE;
        d[c] = xv - anchor[c];
        if (fabsf(d[c]) > m)
            m = fabsf(d[c]);
    }
    uint16_t max1 = m == 0.0f ? 0 : orc_half_up(m);
    *max1_out = max1;
    if (max1 == 0) {
        for (int c = 0; c < C; c++)
            q[c] = (uint8_t)MAX;
        return ORC_OK;
    }
    float factor = (float)MAX / orc_half_to_float(max1);
    for (int c = 0; c < C; c++) {
        float scaled = d[c] * factor;
        float y = scaled + (float)MAX;
        float r = rintf(y);
        if (r < 0.0f)
            r = 0.0f;
        if (r > (float)(2 * MAX))
            r = (float)(2 * MAX);
        q[c] = (uint8_t)r;
    }
    return ORC_OK;
}

int orc_quantize_delta(const uint16_t *k, const uint16_t *v, int L, int T,
                       int C, int Tc, int G, int64_t layer_stride,
                       const int32_t *bins_k, const int32_t *bins_v,
                       uint8_t *sym, uint16_t *max1)
{
    if (!orc_check_shape(L, T, C) || Tc < 1 || G < 1)
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    float *anchor = (float *)malloc((size_t)C * sizeof(float));
    float *d = (float *)malloc((size_t)C * sizeof(float));
    if (!anchor || !d) {
        free(anchor), free(d);
        return ORC_ERR_NOMEM;
    }
    int st = ORC_OK;
    for (int kv = 0; kv < 2 && st == ORC_OK; kv++) {
        const uint16_t *x = kv ? v : k;
        const int32_t *bins = kv ? bins_v : bins_k;
        for (int l = 0; l < L && st == ORC_OK; l++) {
            if (bins[l] < 4 || bins[l] > 256) {
                st = ORC_ERR_ARG;
                break;
            }
            for (int t = 0; t < T && st == ORC_OK; t++) {
                int64_t g = ((int64_t)kv * L + l) * T + t;
                const uint16_t *row = x + (int64_t)l * layer_stride + (int64_t)t * C;
                int tl = t % Tc; /* position in the chunk */
                if (tl % G == 0) {
                    st = orc_quantize_group(row, C, bins[l], sym + g * C, max1 + g);
                    for (int c = 0; c < C && st == ORC_OK; c++)
                        anchor[c] = orc_dequantize_value(sym[g * C + c], bins[l], max1[g]);
                } else {
                    st = orc_quantize_delta_row(row, anchor, C, bins[l], d, sym + g * C,
                                                max1 + g);
                }
            }
        }
    }
    free(anchor), free(d);
    return st;
}

int orc_dequantize_delta(const uint8_t *sym, const uint16_t *max1, int L,
                         int T, int C, int Tc, int G, const int32_t *bins_k,
                         const int32_t *bins_v, float *out_k, float *out_v)
{
    if (!orc_check_shape(L, T, C) || Tc < 1 || G < 1)
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    for (int kv = 0; kv < 2; kv++) {
        float *out = kv ? out_v : out_k;
        const int32_t *bins = kv ? bins_v : bins_k;
        for (int l = 0; l < L; l++)
            for (int t = 0; t < T; t++) {
                int64_t g = ((int64_t)kv * L + l) * T + t;
                int tl = t % Tc;
                int64_t a = g - tl % G; /* the anchor's row */
                for (int c = 0; c < C; c++) {
                    float x = orc_dequantize_value(sym[g * C + c], bins[l], max1[g]);
                    if (a != g)
                        x = orc_dequantize_value(sym[a * C + c], bins[l], max1[a]) + x;
                    out[((int64_t)l * T + t) * C + c] = x;
                }
            }
    }
    return ORC_OK;
}

int orc_compress_ex(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                    int Tc, int G, int fmt, int64_t layer_stride,
                    const int32_t *bins_k, const int32_t *bins_v,
                    uint16_t *max1, void *side, uint8_t *packed,
                    uint64_t capacity, uint32_t *len, uint64_t *off)
{
    if (!orc_check_shape(L, T, C) || Tc < 1 || G < 1 || (fmt != 1 && fmt != 2) ||
        (fmt == 2 && Tc > 256))
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    uint8_t *sym = (uint8_t *)malloc((size_t)(2 * (int64_t)L * T * C));
    if (!sym)
        return ORC_ERR_NOMEM;
    int st = orc_quantize_delta(k, v, L, T, C, Tc, G, layer_stride, bins_k, bins_v, sym, max1);
    if (st == ORC_OK && fmt == 1) {
        int A_k = orc_alphabet(bins_k, L), A_v = orc_alphabet(bins_v, L);
        st = orc_calculate_cdf(sym, L, T, C, Tc, A_k, A_v, (uint16_t *)side);
        if (st == ORC_OK)
            st = orc_encode(sym, (const uint16_t *)side, L, T, C, Tc, A_k, A_v, packed,
                            capacity, len, off);
    } else if (st == ORC_OK) {
        st = orc_code_v2(sym, L, T, C, Tc, bins_k, bins_v, (uint8_t *)side, packed, capacity,
                         len, off);
    }
    free(sym);
    return st;
}

int orc_decompress_ex(const uint8_t *packed, const uint64_t *off,
                      const uint32_t *len, const void *side,
                      const uint16_t *max1, int L, int T, int C, int Tc, int G,
                      int fmt, const int32_t *bins_k, const int32_t *bins_v,
                      float *out_k, float *out_v)
{
    if (!orc_check_shape(L, T, C) || Tc < 1 || G < 1 || (fmt != 1 && fmt != 2) ||
        (fmt == 2 && Tc > 256))
        return ORC_ERR_ARG;
    if (!bins_v)
        bins_v = bins_k;
    uint8_t *sym = (uint8_t *)malloc((size_t)(2 * (int64_t)L * T * C));
    if (!sym)
        return ORC_ERR_NOMEM;
    int st;
    if (fmt == 1)
        st = orc_decode(packed, off, len, (const uint16_t *)side, L, T, C, Tc,
                        orc_alphabet(bins_k, L), orc_alphabet(bins_v, L), sym);
    else
        st = orc_decode_v2(packed, off, len, (const uint8_t *)side, L, T, C, Tc, bins_k,
                           bins_v, sym);
    if (st == ORC_OK)
        st = orc_dequantize_delta(sym, max1, L, T, C, Tc, G, bins_k, bins_v, out_k, out_v);
    free(sym);
    return st;
}

/* ---- format 3: compact count records ------------------------------------- */

static void orc_put_le(uint8_t *p, uint64_t v, int nbytes)
{
    for (int i = 0; i < nbytes; i++)
        p[i] = (uint8_t)(v >> (8 * i));
}

static uint64_t orc_get_le(const uint8_t *p, int nbytes)
{
    uint64_t v = 0;
    for (int i = 0; i < nbytes; i++)
        v |= (uint64_t)p[i] << (8 * i);
    return v;
}

/* Byte offsets of M, B and V in the side buffer; 0 when format 3 does not
 * apply to the shape. */
static int64_t orc_v3_layout(int L, int T, int C, int Tc, int64_t *offM,
                             int64_t *offB, int64_t *nslice)
{
    if (!orc_check_shape(L, T, C) || Tc < 1 || Tc > 256)
        return 0;
    int64_t nch = (T + Tc - 1) / Tc;
    int64_t ns = 2 * (int64_t)L * nch, nrec = ns * C;
    *nslice = ns;
    *offM = 8 * (ns + 1);
    *offB = (*offM + nrec + 3) / 4 * 4;
    return *offB + 4 * nrec; /* offV */
}

static int orc_v3_bins_ok(int L, const int32_t *bins_k, const int32_t *bins_v)
{
    for (int l = 0; l < L; l++)
        if (bins_k[l] < 4 || bins_v[l] < 4 || orc_alphabet_v2(bins_k[l]) > 32 ||
            orc_alphabet_v2(bins_v[l]) > 32)
            return 0;
    return 1;
}

int64_t orc_v3_fixed_bytes(int L, int T, int C, int Tc)
{
    int64_t offM, offB, ns;
    return orc_v3_layout(L, T, C, Tc, &offM, &offB, &ns);
}

int64_t orc_v3_max_bytes(int L, int T, int C, int Tc, const int32_t *bins_k,
                         const int32_t *bins_v)
{
    if (!bins_v)
        bins_v = bins_k;
    int64_t offM, offB, ns;
    int64_t offV = orc_v3_layout(L, T, C, Tc, &offM, &offB, &ns);
    if (offV == 0 || !orc_v3_bins_ok(L, bins_k, bins_v))
        return 0;
    int64_t per_chunk = 0;
    for (int l = 0; l < L; l++)
        per_chunk += (int64_t)C * (orc_alphabet_v2(bins_k[l]) - 1 + orc_alphabet_v2(bins_v[l]) - 1);
    return offV + per_chunk * ((T + Tc - 1) / Tc);
}

/* A record's byte 1 + i holds the count of the i-th symbol other than the
 * mode, in increasing order. */
static int orc_other_symbol(int i, int mode)
{
    return i < mode ? i : i + 1;
}

int64_t orc_records_to_v3(const uint8_t *rec, int L, int T, int C, int Tc,
                          const int32_t *bins_k, const int32_t *bins_v,
                          uint8_t *side, int64_t capacity)
{
    if (!bins_v)
        bins_v = bins_k;
    int64_t offM, offB, ns;
    int64_t offV = orc_v3_layout(L, T, C, Tc, &offM, &offB, &ns);
    if (offV == 0 || !orc_v3_bins_ok(L, bins_k, bins_v) || capacity < offV)
        return -ORC_ERR_ARG;
    memset(side, 0, (size_t)offV);
    int nch = (T + Tc - 1) / Tc;
    int64_t pos = 0; /* bytes of V so far */
    for (int kc = 0; kc < nch; kc++)
        for (int kv = 0; kv < 2; kv++)
            for (int l = 0; l < L; l++) {
                int64_t s = ((int64_t)kc * 2 + kv) * L + l;
                int A = orc_alphabet_v2((kv ? bins_v : bins_k)[l]);
                orc_put_le(side + 8 * s, (uint64_t)pos, 8);
                for (int c = 0; c < C; c++) {
                    const uint8_t *r = rec + orc_rec_offset(L, C, bins_k, bins_v, kc, kv, l, c);
                    int mode = r[0];
                    if (mode >= A)
                        return -ORC_ERR_CORRUPT;
                    uint32_t bits = 0;
                    for (int i = 0; i < A - 1; i++) {
                        if (r[1 + i] == 0)
                            continue;
                        bits |= 1u << orc_other_symbol(i, mode);
                        if (offV + pos >= capacity)
                            return -ORC_ERR_CAPACITY;
                        side[offV + pos++] = r[1 + i];
                    }
                    side[offM + s * C + c] = (uint8_t)mode;
                    orc_put_le(side + offB + 4 * (s * C + c), bits, 4);
                }
            }
    orc_put_le(side + 8 * ns, (uint64_t)pos, 8);
    return offV + pos;
}

int orc_v3_to_records(const uint8_t *side, int64_t nbytes, int L, int T, int C,
                      int Tc, const int32_t *bins_k, const int32_t *bins_v,
                      uint8_t *rec)
{
    if (!bins_v)
        bins_v = bins_k;
    int64_t offM, offB, ns;
    int64_t offV = orc_v3_layout(L, T, C, Tc, &offM, &offB, &ns);
    if (offV == 0 || !orc_v3_bins_ok(L, bins_k, bins_v))
        return ORC_ERR_ARG;
    if (nbytes < offV || orc_get_le(side, 8) != 0)
        return ORC_ERR_CORRUPT;
    uint64_t vtotal = orc_get_le(side + 8 * ns, 8);
    if (vtotal > (uint64_t)(nbytes - offV))
        return ORC_ERR_CORRUPT;
    int nch = (T + Tc - 1) / Tc;
    for (int kc = 0; kc < nch; kc++)
        for (int kv = 0; kv < 2; kv++)
            for (int l = 0; l < L; l++) {
                int64_t s = ((int64_t)kc * 2 + kv) * L + l;
                int A = orc_alphabet_v2((kv ? bins_v : bins_k)[l]);
                uint64_t pos = orc_get_le(side + 8 * s, 8);
                uint64_t end = orc_get_le(side + 8 * (s + 1), 8);
                if (pos > end || end > vtotal)
                    return ORC_ERR_CORRUPT;
                for (int c = 0; c < C; c++) {
                    uint8_t *r = rec + orc_rec_offset(L, C, bins_k, bins_v, kc, kv, l, c);
                    int mode = side[offM + s * C + c];
                    uint32_t bits = (uint32_t)orc_get_le(side + offB + 4 * (s * C + c), 4);
                    if (mode >= A || (A < 32 && (bits >> A) != 0) || ((bits >> mode) & 1u))
                        return ORC_ERR_CORRUPT;
                    r[0] = (uint8_t)mode;
                    for (int i = 0; i < A - 1; i++) {
                        int t = orc_other_symbol(i, mode);
                        r[1 + i] = 0;
                        if ((bits >> t) & 1u) {
                            if (pos >= end || side[offV + pos] == 0)
                                return ORC_ERR_CORRUPT;
                            r[1 + i] = side[offV + pos++];
                        }
                    }
                }
                if (pos != end)
                    return ORC_ERR_CORRUPT;
            }
    return ORC_OK;
}

int orc_compress_v3(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                    int Tc, int G, int64_t layer_stride, const int32_t *bins_k,
                    const int32_t *bins_v, uint16_t *max1, uint8_t *side,
                    int64_t side_capacity, int64_t *side_bytes,
                    uint8_t *packed, uint64_t capacity, uint32_t *len,
                    uint64_t *off)
{
    if (!bins_v)
        bins_v = bins_k;
    int64_t nrec = orc_rec_bytes(L, T, C, Tc, bins_k, bins_v);
    if (nrec <= 0 || orc_v3_fixed_bytes(L, T, C, Tc) == 0 || !orc_v3_bins_ok(L, bins_k, bins_v))
        return ORC_ERR_ARG;
    uint8_t *rec = (uint8_t *)malloc((size_t)nrec);
    if (!rec)
        return ORC_ERR_NOMEM;
    int st = orc_compress_ex(k, v, L, T, C, Tc, G, 2, layer_stride, bins_k, bins_v, max1, rec,
                             packed, capacity, len, off);
    if (st == ORC_OK || st == ORC_ERR_CAPACITY) {
        int64_t n = orc_records_to_v3(rec, L, T, C, Tc, bins_k, bins_v, side, side_capacity);
        if (n < 0)
            st = (int)-n;
        else
            *side_bytes = n;
    }
    free(rec);
    return st;
}

int orc_decompress_v3(const uint8_t *packed, const uint32_t *len,
                      const uint8_t *side, int64_t side_bytes,
                      const uint16_t *max1, int L, int T, int C, int Tc, int G,
                      const int32_t *bins_k, const int32_t *bins_v,
                      float *out_k, float *out_v)
{
    if (!bins_v)
        bins_v = bins_k;
    int64_t nrec = orc_rec_bytes(L, T, C, Tc, bins_k, bins_v);
    int64_t ns = orc_num_streams(L, T);
    if (nrec <= 0)
        return ORC_ERR_ARG;
    uint8_t *rec = (uint8_t *)malloc((size_t)nrec);
    uint64_t *off = (uint64_t *)malloc((size_t)(ns + 1) * sizeof(uint64_t));
    if (!rec || !off) {
        free(rec), free(off);
        return ORC_ERR_NOMEM;
    }
    /* the offsets are the exclusive scan of the lengths */
    off[0] = 0;
    for (int64_t i = 0; i < ns; i++)
        off[i + 1] = off[i] + len[i];
    int st = orc_v3_to_records(side, side_bytes, L, T, C, Tc, bins_k, bins_v, rec);
    if (st == ORC_OK)
        st = orc_decompress_ex(packed, off, len, rec, max1, L, T, C, Tc, G, 2, bins_k, bins_v,
                               out_k, out_v);
    free(rec), free(off);
    return st;
}
