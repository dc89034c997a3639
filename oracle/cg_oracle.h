/*
 * cg_oracle.h - CPU oracle for the CacheGen KV-cache codec.
 *
 * TEST INFRASTRUCTURE ONLY. This is the plain, slow, single-threaded reference
 * the CUDA library is checked against. Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load it. The product library never
 * links it, calls it or falls back to it, and it shares no source with it.
 *
 * Citation key used throughout:
 *   [CG] = web page "CacheGen 技术详解：KV Cache 的高效压缩与流式传输"
 *          (CacheGen as implemented in LMCache, forceinjection.github.io).
 *   [CG §2.3(1)] quantisation (torch_quant_vectorized), [CG §2.3(2)] CDF
 *   (calculate_cdf), [CG §2.3(3)] 256-token chunks, [CG §1.2(3)] arithmetic
 *   coding, [CG §2.4(1)] GPU decoding, [CG §2.4(2)] dequantisation
 *   (do_dequantize), [CG §2.2] layer-wise bins (QuantizationSpec).
 *
 * The page states the quantisation and dequantisation formulas but gives no
 * bit-stream format, CDF precision or coder constants. Those are fixed by the
 * codec specification restated below; both this oracle and the CUDA library
 * implement it independently.
 *
 * ---------------------------------------------------------------------------
 * Codec specification (format version 1)
 * ---------------------------------------------------------------------------
 * Shapes: K and V are fp16 [L][T][C]; tokens are cut into chunks of Tc tokens
 * (the last chunk may be shorter: Tc_k = min(Tc, T - k*Tc)); nch = ceil(T/Tc).
 *
 * Q  (quantise, per group (kv, layer l, token t), IEEE binary32, every
 *    operation rounded to nearest-even on its own, no fused multiply-add):
 *    MAX = bins_l / 2 - 1 (integer division); max1 = max_c |x_c| (an fp16
 *    value, stored as fp16); factor = (float)MAX / max1;
 *    y = (x * factor) + (float)MAX; q = rint(y) (ties to even), clamped to
 *    [0, 2*MAX]. A group with max1 == 0 gives q = MAX everywhere. Non-finite
 *    input is rejected. bins_l must lie in [4, 256].
 *
 * A  (alphabet width) A_K = max_l bins_k[l], A_V = max_l bins_v[l]; every
 *    CDF of that tensor has A symbols 0..A-1.
 *
 * F  (CDF, per (chunk k, kv, l, channel c), over the chunk's Tc_k tokens):
 *    n_s = count of q == s; f_s = 1 + floor(n_s * (65536 - A) / Tc_k);
 *    R = 65536 - sum f_s (0 <= R < A) is added to the symbol with the largest
 *    n_s (smallest s on ties); cdf[0] = 0, cdf[s+1] = cdf[s] + f_s; the A
 *    entries cdf[0..A-1] are stored as uint16 (cdf[A] = 65536 is implicit).
 *    Layout: cdf[k] = { K: [L][C][A_K], then V: [L][C][A_V] }.
 *
 * R  (range coder, one stream per (k, kv, l, t) over c = 0..C-1 ascending,
 *    each symbol coded with cdf[k][kv][l][c]):
 *    state low = 0, range = 0xFFFFFFFF (uint32).
 *    encode s: r = range >> 16; low' = low + r*cdf[s] (mod 2^32); if low' <
 *    low a carry adds one to the bytes already emitted (last byte first, 0xFF
 *    becomes 0x00 and the carry moves on); low = low'; range = r * f_s;
 *    while range < 2^24: emit low >> 24, low <<= 8, range <<= 8.
 *    flush: v = low + 0x00FFFFFF (carry as above if it wraps); emit v >> 24.
 *    decode: range = 0xFFFFFFFF, code = first 4 bytes big-endian; bytes at or
 *    past the stream's length read as 0. Per symbol: r = range >> 16;
 *    s = largest s with r*cdf[s] <= code; code -= r*cdf[s]; range = r*f_s;
 *    while range < 2^24: code = (code << 8) | next byte, range <<= 8.
 *    A valid stream of len bytes is consumed in exactly len + 3 bytes.
 *
 * P  (packing) stream id sid(k, kv, l, tl) = 2*L*Tc*k + (kv*L + l)*Tc_k + tl;
 *    streams are stored back to back in sid order, len[] is uint32 per
 *    stream, off[] the uint64 exclusive scan of len with off[nstreams] the
 *    total; nstreams = 2*L*T. With a capacity below the total, exactly the
 *    bytes at positions < capacity are written.
 *
 * D  (dequantise, binary32, no FMA): x^ = ((float)(q - MAX) / (float)MAX)
 *    * (float)max1.
 *
 * ---------------------------------------------------------------------------
 * Format version 2: side information as symbol counts
 * ---------------------------------------------------------------------------
 * The page sends, with each chunk, what the decoder needs to rebuild the
 * chunk's CDFs [CG §2.3(2), §2.4(1)]; format 2 sends the symbol counts the
 * CDFs are built from instead of the CDF entries. Q, R, P and D are as in
 * format 1; requires Tc <= 256.
 *
 * A2 (alphabet per (kv, l)): A = 2*MAX_l + 1, the symbols Q can produce.
 * S  (count record per (chunk k, kv, l, channel c), A bytes): byte 0 is the
 *    mode s* (largest n_s, smallest s on ties); bytes 1..A-1 are n_s for
 *    every s != s* in increasing s, one byte each (a count other than the
 *    mode's is at most Tc_k / 2 <= 128). The mode's count is Tc_k minus the
 *    others. Layout: rec[k] = { K: layer 0 [C][A_0], layer 1 [C][A_1], ...,
 *    then V likewise }.
 * F2 (CDF) F over the layer's A symbols, the remainder going to the record's
 *    mode byte.
 *
 * ---------------------------------------------------------------------------
 * Format version 3: compact count records
 * ---------------------------------------------------------------------------
 * Format 2's counts, stored without its zero bytes; the CDFs, and so the
 * streams, are format 2's. Requires Tc <= 256 and every A_l <= 32. Slices
 * s = (k*2 + kv)*L + l (nslice = 2*L*nch); records r = s*C + c
 * (nrec = nslice*C). One side buffer, little-endian:
 *   O  uint64 [nslice + 1] at byte 0: O[s] = offset of slice s's counts in
 *      V, O[nslice] = |V|;
 *   M  uint8 [nrec] at byte offM = 8*(nslice + 1): each record's mode;
 *   B  uint32 [nrec] at byte offB = offM + nrec rounded up to a multiple
 *      of 4: bit t set iff t != mode and n_t > 0 (t < A_l);
 *   V  uint8 at byte offV = offB + 4*nrec: for each record in order, its
 *      set bits' counts n_t in increasing t, one byte each.
 * Size offV + O[nslice]. Only the stream lengths travel with it (the
 * offsets are their exclusive scan).
 * ---------------------------------------------------------------------------
 * Token-locality delta: the change-based encoding of [CG §1.2(1)]
 * ---------------------------------------------------------------------------
 * The page's design codes each token's change from a nearby token rather than
 * its raw values, since neighbouring tokens' K/V are similar [CG §1.2(1)];
 * LMCache's code skips this step [CG §2.3(1)]. The page gives no group size,
 * anchor rule or precision; this specification reads it as follows. It
 * changes Q and D only (F, F2, S, R and P see symbols as before), so it
 * applies to either format. Group size G >= 1; G = 1 is plain Q and D.
 *
 * G  (groups) within chunk k the tokens tl = 0..Tc_k-1 form groups of G
 *    consecutive tokens from tl = 0; the first token of each group
 *    (tl % G == 0) is the group's anchor.
 * QA (anchor rows) exactly Q. The anchor's reconstruction is
 *    a^_c = D(q_a,c, max1_a), binary32, as the decoder will see it.
 * QD (other rows) d_c = x_c - a^_c (binary32, rounded once); m = max_c |d_c|;
 *    max1 = the smallest binary16 value >= m (stored as fp16; the largest
 *    finite binary16, 65504, if m exceeds it); then Q's steps on d with this
 *    max1: factor = (float)MAX / max1, y = (d * factor) + (float)MAX,
 *    q = rint(y) clamped to [0, 2*MAX]; max1 == 0 gives q = MAX.
 * DD (other rows) x^_c = a^_c + D(q_c, max1) (binary32, the sum rounded
 *    once); anchor rows are D. A binary16 output rounds x^ to nearest-even.
 */
#ifndef CG_ORACLE_H
#define CG_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    ORC_OK = 0,
    ORC_ERR_ARG = 1,
    ORC_ERR_NONFINITE = 2,
    ORC_ERR_CAPACITY = 3,
    ORC_ERR_CORRUPT = 4,
    ORC_ERR_NOMEM = 5
};

/* fp16 bits -> binary32 (exact). */
float orc_half_to_float(uint16_t h);

/* [CG §2.3(1)] one group of C fp16 values -> C symbols and the group's max1. */
int orc_quantize_group(const uint16_t *x, int64_t C, int bins, uint8_t *q,
                       uint16_t *max1);

/* [CG §2.4(2)] one symbol -> binary32, given the group's max1 (fp16 bits). */
float orc_dequantize_value(uint8_t q, int bins, uint16_t max1);

/* [CG §2.3(2)] counts of A symbols over Tk tokens -> A uint16 CDF entries. */
int orc_cdf_from_counts(const uint32_t *n, int A, uint32_t Tk, uint16_t *cdf);

/* [CG §1.2(3)] encode n symbols; symbol i uses the CDF row cdf + i*row_stride
 * (A entries). Writes at most cap bytes; returns the stream length or -1 when
 * cap is too small or an argument is bad. */
int64_t orc_encode_stream(const uint8_t *sym, int64_t n, const uint16_t *cdf,
                          int64_t row_stride, int A, uint8_t *out, int64_t cap);

/* [CG §2.4(1)] decode n symbols from a stream of len bytes. *consumed gets
 * the number of bytes the decoder read (len + 3 for a valid stream). */
int orc_decode_stream(const uint8_t *in, int64_t len, int64_t n,
                      const uint16_t *cdf, int64_t row_stride, int A,
                      uint8_t *sym, int64_t *consumed);

/* Size helpers. */
int64_t orc_num_streams(int L, int T);
int64_t orc_cdf_elems(int L, int T, int C, int Tc, int A_k, int A_v);
int64_t orc_cdf_offset(int L, int C, int A_k, int A_v, int k, int kv, int l,
                       int c);
int64_t orc_stream_id(int L, int T, int Tc, int k, int kv, int l, int tl);
int orc_alphabet(const int32_t *bins, int L);

/* Whole-tensor steps. k and v are fp16 [L][T][C] with layers layer_stride
 * elements apart (tokens C apart, channels contiguous). sym is uint8
 * [2][L][T][C], max1 fp16 [2][L][T]. bins_v == NULL means bins_v = bins_k. */
int orc_quantize(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                 int64_t layer_stride, const int32_t *bins_k,
                 const int32_t *bins_v, uint8_t *sym, uint16_t *max1);

int orc_calculate_cdf(const uint8_t *sym, int L, int T, int C, int Tc,
                      int A_k, int A_v, uint16_t *cdf);

int orc_encode(const uint8_t *sym, const uint16_t *cdf, int L, int T, int C,
               int Tc, int A_k, int A_v, uint8_t *packed, uint64_t capacity,
               uint32_t *len, uint64_t *off);

int orc_decode(const uint8_t *packed, const uint64_t *off, const uint32_t *len,
               const uint16_t *cdf, int L, int T, int C, int Tc, int A_k,
               int A_v, uint8_t *sym);

int orc_dequantize(const uint8_t *sym, const uint16_t *max1, int L, int T,
                   int C, const int32_t *bins_k, const int32_t *bins_v,
                   float *out_k, float *out_v);

/* Quantise -> CDF -> encode in one call (symbols kept in host scratch). */
int orc_compress(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                 int Tc, int64_t layer_stride, const int32_t *bins_k,
                 const int32_t *bins_v, uint16_t *max1, uint16_t *cdf,
                 uint8_t *packed, uint64_t capacity, uint32_t *len,
                 uint64_t *off);

/* Decode -> dequantise in one call. */
int orc_decompress(const uint8_t *packed, const uint64_t *off,
                   const uint32_t *len, const uint16_t *cdf,
                   const uint16_t *max1, int L, int T, int C, int Tc,
                   const int32_t *bins_k, const int32_t *bins_v, float *out_k,
                   float *out_v);

/* ---- format 2 ---------------------------------------------------------- */
/* A = 2*MAX + 1 for a layer with `bins` bins (specification A2). */
int orc_alphabet_v2(int bins);
/* Bytes of all count records / offset of record (k, kv, l, c). */
int64_t orc_rec_bytes(int L, int T, int C, int Tc, const int32_t *bins_k,
                      const int32_t *bins_v);
int64_t orc_rec_offset(int L, int C, const int32_t *bins_k,
                       const int32_t *bins_v, int k, int kv, int l, int c);
/* [CG §2.3(2)] counts of A symbols -> the A-byte record (S); error if a
 * non-mode count exceeds 255. */
int orc_record_from_counts(const uint32_t *n, int A, uint8_t *rec);
/* The record -> counts over Tk tokens; error if the mode byte is >= A or the
 * stored counts exceed Tk. */
int orc_counts_from_record(const uint8_t *rec, int A, uint32_t Tk, uint32_t *n);
/* F2: counts and the mode -> A uint16 CDF entries. */
int orc_cdf_from_counts_mode(const uint32_t *n, int A, uint32_t Tk, int mode,
                             uint16_t *cdf);
/* Quantise -> counts -> records and CDFs -> encode (format 2). */
int orc_compress_v2(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                    int Tc, int64_t layer_stride, const int32_t *bins_k,
                    const int32_t *bins_v, uint16_t *max1, uint8_t *rec,
                    uint8_t *packed, uint64_t capacity, uint32_t *len,
                    uint64_t *off);
/* Records -> CDFs -> decode -> dequantise (format 2). */
int orc_decompress_v2(const uint8_t *packed, const uint64_t *off,
                      const uint32_t *len, const uint8_t *rec,
                      const uint16_t *max1, int L, int T, int C, int Tc,
                      const int32_t *bins_k, const int32_t *bins_v,
                      float *out_k, float *out_v);

/* ---- serving layouts ---------------------------------------------------- */
/* binary32 -> binary16 bits, round to nearest, ties to even. */
uint16_t orc_float_to_half(float x);
/* D with binary16 output (each binary32 value rounded to nearest-even). */
int orc_dequantize_half(const uint8_t *sym, const uint16_t *max1, int L, int T,
                        int C, const int32_t *bins_k, const int32_t *bins_v,
                        uint16_t *out_k, uint16_t *out_v);

/* ---- format 3: compact count records ------------------------------------- */
/* Fixed part of the side buffer (offV) and its largest size; 0 when the
 * shape, the bins or Tc do not allow format 3. */
int64_t orc_v3_fixed_bytes(int L, int T, int C, int Tc);
int64_t orc_v3_max_bytes(int L, int T, int C, int Tc, const int32_t *bins_k,
                         const int32_t *bins_v);
/* Format 2 records -> format 3 side buffer (size returned, < 0 on error). */
int64_t orc_records_to_v3(const uint8_t *rec, int L, int T, int C, int Tc,
                          const int32_t *bins_k, const int32_t *bins_v,
                          uint8_t *side, int64_t capacity);
/* Format 3 side buffer (nbytes readable) -> format 2 records; an error for
 * a buffer that is not one the encoder can produce (offsets out of order or
 * past the buffer, a mode outside the alphabet, a bit at or past A or at the
 * mode, a slice whose bits disagree with its offsets). */
int orc_v3_to_records(const uint8_t *side, int64_t nbytes, int L, int T, int C,
                      int Tc, const int32_t *bins_k, const int32_t *bins_v,
                      uint8_t *rec);
/* Compress in format 3 (with token groups of G; 1: none): max1, side
 * buffer (size in *side_bytes), packed, len (and off). */
int orc_compress_v3(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                    int Tc, int G, int64_t layer_stride, const int32_t *bins_k,
                    const int32_t *bins_v, uint16_t *max1, uint8_t *side,
                    int64_t side_capacity, int64_t *side_bytes,
                    uint8_t *packed, uint64_t capacity, uint32_t *len,
                    uint64_t *off);
/* Decompress format 3 from the lengths alone (offsets rebuilt), binary32. */
int orc_decompress_v3(const uint8_t *packed, const uint32_t *len,
                      const uint8_t *side, int64_t side_bytes,
                      const uint16_t *max1, int L, int T, int C, int Tc, int G,
                      const int32_t *bins_k, const int32_t *bins_v,
                      float *out_k, float *out_v);

/* ---- token-locality delta (specification G) ------------------------------ */
/* The smallest binary16 value >= m (m finite, >= 0), as bits; 0x7BFF (the
 * largest finite binary16) when m > 65504. */
uint16_t orc_half_up(float m);
/* binary32 -> binary16 (round to nearest-even) over n values. */
void orc_floats_to_half(const float *x, int64_t n, uint16_t *out);
/* QA + QD over the whole tensor: symbols [2][L][T][C], max1 [2][L][T]. */
int orc_quantize_delta(const uint16_t *k, const uint16_t *v, int L, int T,
                       int C, int Tc, int G, int64_t layer_stride,
                       const int32_t *bins_k, const int32_t *bins_v,
                       uint8_t *sym, uint16_t *max1);
/* D on anchors, DD on the other rows; binary32 output [L][T][C]. */
int orc_dequantize_delta(const uint8_t *sym, const uint16_t *max1, int L,
                         int T, int C, int Tc, int G, const int32_t *bins_k,
                         const int32_t *bins_v, float *out_k, float *out_v);
/* Quantise with groups of G tokens (G = 1: plain Q) and code in format fmt
 * (1: side = uint16 CDF entries, 2: side = uint8 count records). */
int orc_compress_ex(const uint16_t *k, const uint16_t *v, int L, int T, int C,
                    int Tc, int G, int fmt, int64_t layer_stride,
                    const int32_t *bins_k, const int32_t *bins_v,
                    uint16_t *max1, void *side, uint8_t *packed,
                    uint64_t capacity, uint32_t *len, uint64_t *off);
/* The inverse of orc_compress_ex, binary32 output. */
int orc_decompress_ex(const uint8_t *packed, const uint64_t *off,
                      const uint32_t *len, const void *side,
                      const uint16_t *max1, int L, int T, int C, int Tc, int G,
                      int fmt, const int32_t *bins_k, const int32_t *bins_v,
                      float *out_k, float *out_v);

#ifdef __cplusplus
}
#endif
#endif
