/*
 * cachegen.h - C ABI of the GB300 (sm_103a) CacheGen KV-cache codec.
 *
 * Citation key: [CG] = web page "CacheGen 技术详解：KV Cache 的高效压缩与流式传输"
 * (CacheGen as implemented in LMCache). Sections cited: §2.2 layer-wise bins
 * (QuantizationSpec), §2.3(1) vectorised adaptive quantisation
 * (torch_quant_vectorized), §2.3(2) CDF computation (calculate_cdf),
 * §2.3(3) 256-token chunks, §1.2(3) GPU-parallel arithmetic coding,
 * §2.4(1) GPU-parallel decoding (decode_function_gpu), §2.4(2)
 * dequantisation (do_dequantize), §3.2 the (layers, 2, tokens, heads,
 * head_dim) fp16 KV layout.
 *
 * Conventions
 *  - Every data pointer is DEVICE memory owned by the caller, except the
 *    bins arrays (HOST int32, read during the call and not kept).
 *  - The library allocates nothing. Scratch comes from the caller through a
 *    workspace pointer sized with cg_workspace_bytes().
 *  - Every call is asynchronous on the caller's stream; nothing synchronises,
 *    so the calls can be captured in a CUDA graph and replayed.
 *  - fp16 values are passed as their IEEE binary16 bit patterns (uint16_t).
 *  - The return value reports argument and launch errors, detected on the
 *    host before (or at) launch. Errors that depend on the data are OR-ed as
 *    CG_FLAG_* bits into an optional device int32 status word, which the
 *    caller zeroes beforehand and reads after synchronising. Kernels never
 *    assert or trap.
 *
 * Codec specification (format version 1; the page gives the quantisation and
 * dequantisation formulas, this header fixes the rest):
 *  Q  per group (kv, layer l, token t): MAX = bins_l / 2 - 1;
 *     max1 = max_c |x_c| (kept as fp16); factor = (float)MAX / max1;
 *     q = rint((x * factor) + (float)MAX) in binary32 with every operation
 *     rounded on its own (ties to even), clamped to [0, 2*MAX]; a group with
 *     max1 = 0 gives q = MAX. bins_l in [4, 256].
 *  A  alphabet width A_K = max_l bins_k[l], A_V = max_l bins_v[l].
 *  F  per (chunk k, kv, l, channel c) over the chunk's Tc_k tokens: counts
 *     n_s; f_s = 1 + floor(n_s * (65536 - A) / Tc_k); the remainder
 *     65536 - sum f_s goes to the symbol with the largest count (smallest s
 *     on ties); cdf[s] = f_0 + ... + f_{s-1}, stored as uint16 cdf[0..A-1].
 *     Layout per chunk: K rows [L][C][A_K] then V rows [L][C][A_V].
 *  R  range coder, one stream per (k, kv, l, t) over channels c = 0..C-1,
 *     symbol c coded with row (k, kv, l, c): low = 0, range = 0xFFFFFFFF;
 *     r = range >> 16; low += r*cdf[s] (a wrap adds one to the bytes
 *     already emitted, 0xFF bytes turning to 0x00); range = r*f_s; while
 *     range < 2^24 emit low >> 24, shift low and range left by 8. Flush:
 *     emit (low + 0x00FFFFFF) >> 24 (carrying as above). The decoder reads
 *     bytes at or past the stream's length as 0 and consumes exactly
 *     len + 3 bytes of a valid stream.
 *  P  stream id sid(k, kv, l, tl) = 2*L*Tc*k + (kv*L + l)*Tc_k + tl with
 *     Tc_k = min(Tc, T - k*Tc); streams stored back to back in sid order;
 *     len[] uint32 per stream; off[] uint64 exclusive scan (off[nstreams]
 *     = total); nstreams = 2*L*T.
 *  D  x^ = ((float)(q - MAX) / (float)MAX) * (float)max1 in binary32.
 */
#ifndef CACHEGEN_GB300_H
#define CACHEGEN_GB300_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t cg_status;

/* Return codes. */
#define CG_OK 0
#define CG_ERR_INVALID_ARG 1 /* null pointer, bad shape or bins, misaligned */
#define CG_ERR_WORKSPACE 2   /* workspace smaller than cg_workspace_bytes() */
#define CG_ERR_CUDA 3        /* a kernel launch failed (cudaGetLastError) */

/* Device status bits (OR-ed into *status when status != NULL). */
#define CG_FLAG_NONFINITE 0x1 /* an input value was Inf or NaN (Q) */
#define CG_FLAG_CAPACITY 0x2  /* packed total exceeded capacity (P) */
#define CG_FLAG_CORRUPT 0x4   /* a stream did not decode in len + 3 bytes,
                                 or off/len point outside the buffer (R) */
#define CG_FLAG_BAD_SYMBOL 0x8 /* encode input symbol >= A */
#define CG_FLAG_TIMEOUT 0x10   /* a bounded wait for another CTA ran out;
                                  offsets and packed bytes are not valid */

/* Limits of this implementation. */
#define CG_MAX_LAYERS 1024
#define CG_MAX_CHUNK_TOKENS 1024
#define CG_MAX_CHANNELS 65536

/* Shape of one K (or V) tensor, fp16 [L][T][C]: channels contiguous, tokens
 * C elements apart, layers layer_stride elements apart (layer_stride = T*C
 * when contiguous; 2*T*C for K and V views of the [layers][2][tokens][heads]
 * [head_dim] layout of [CG §3.2], where C = heads*head_dim and V starts T*C
 * elements after K). chunk_tokens is the CDF and streaming unit [CG §2.3(3)]
 * (256 by default); the last chunk may be shorter. */
typedef struct cg_shape {
    int32_t L;
    int32_t T;
    int32_t C;
    int32_t chunk_tokens;
    int64_t layer_stride;
} cg_shape;

/* ---- sizes (host only, no device work) --------------------------------- */

/* 2*L*T, or 0 for an invalid shape. */
uint64_t cg_num_streams(const cg_shape *shape);

/* Number of uint16 CDF entries: nch * L * C * (A_K + A_V), or 0 when the
 * shape or the bins are invalid. bins_v == NULL means bins_v = bins_k. */
uint64_t cg_cdf_elems(const cg_shape *shape, const int32_t *bins_k,
                      const int32_t *bins_v);

/* Upper bound of the packed size: nstreams * (2*C + 8) bytes. With
 * capacity >= this bound CG_FLAG_CAPACITY cannot occur. */
uint64_t cg_max_compressed_bytes(const cg_shape *shape);

/* Bytes of device workspace cg_encode / cg_compress_chunk need (per-stream
 * staging plus scan partials); 0 for an invalid shape. */
uint64_t cg_workspace_bytes(const cg_shape *shape);

/* ---- steps ------------------------------------------------------------- */

/* [CG §2.3(1), §2.2] Quantise K and V (fp16 bits, see cg_shape) with the
 * layer-wise bins. Outputs: sym uint8 [2][L][T][C] (K then V), max1 fp16
 * bits [2][L][T]. k, v must be 2-byte aligned. Sets CG_FLAG_NONFINITE in
 * *status on Inf/NaN input (outputs then unspecified for those groups). */
cg_status cg_quantize(const uint16_t *k, const uint16_t *v,
                      const cg_shape *shape, const int32_t *bins_k,
                      const int32_t *bins_v, uint8_t *sym, uint16_t *max1,
                      int32_t *status, cudaStream_t stream);

/* [CG §2.3(2)] Per (chunk, kv, layer, channel) CDFs of the symbols
 * sym [2][L][T][C] (symbols must be < the tensor's A); output cdf has
 * cg_cdf_elems() uint16 entries in the layout of F above. */
cg_status cg_calculate_cdf(const uint8_t *sym, const cg_shape *shape,
                           const int32_t *bins_k, const int32_t *bins_v,
                           uint16_t *cdf, int32_t *status,
                           cudaStream_t stream);

/* [CG §1.2(3), §2.3(3)] Range-code every (chunk, kv, layer, token) stream of
 * sym with the given CDFs and pack them. Outputs: packed bytes (only
 * positions < capacity are written), len uint32 [nstreams], off uint64
 * [nstreams + 1] (the total is off[nstreams], on the device). workspace
 * must hold cg_workspace_bytes(shape) bytes, 256-byte aligned. */
cg_status cg_encode(const uint8_t *sym, const uint16_t *cdf,
                    const cg_shape *shape, const int32_t *bins_k,
                    const int32_t *bins_v, uint8_t *packed, uint64_t capacity,
                    uint32_t *len, uint64_t *off, void *workspace,
                    uint64_t workspace_bytes, int32_t *status,
                    cudaStream_t stream);

/* [CG §2.4(1)] Decode every stream back to symbols sym [2][L][T][C].
 * packed_bytes is the readable size of packed; bytes a stream would read at
 * or past its len (or past packed_bytes) read as 0. A stream not consumed in
 * exactly len + 3 bytes, or lying outside packed_bytes, sets
 * CG_FLAG_CORRUPT. */
cg_status cg_decode(const uint8_t *packed, uint64_t packed_bytes,
                    const uint64_t *off, const uint32_t *len,
                    const uint16_t *cdf, const cg_shape *shape,
                    const int32_t *bins_k, const int32_t *bins_v, uint8_t *sym,
                    int32_t *status, cudaStream_t stream);

/* [CG §2.4(2)] Dequantise sym [2][L][T][C] with max1 [2][L][T] into binary32
 * out_k, out_v, each [L][T][C] contiguous. */
cg_status cg_dequantize(const uint8_t *sym, const uint16_t *max1,
                        const cg_shape *shape, const int32_t *bins_k,
                        const int32_t *bins_v, float *out_k, float *out_v,
                        int32_t *status, cudaStream_t stream);

/* ---- fused ------------------------------------------------------------- */

/* Quantise -> CDF -> encode -> pack in one call (the serializer's to_bytes
 * [CG §2.1, §3.2]); same outputs as the steps above, without a symbol
 * tensor. workspace must hold cg_compress_workspace_bytes(shape) bytes,
 * 256-byte aligned. */
uint64_t cg_compress_workspace_bytes(const cg_shape *shape);

cg_status cg_compress_chunk(const uint16_t *k, const uint16_t *v,
                            const cg_shape *shape, const int32_t *bins_k,
                            const int32_t *bins_v, uint16_t *max1,
                            uint16_t *cdf, uint8_t *packed, uint64_t capacity,
                            uint32_t *len, uint64_t *off, void *workspace,
                            uint64_t workspace_bytes, int32_t *status,
                            cudaStream_t stream);

/* Decode fused with dequantisation (the deserializer [CG §2.4]): packed
 * streams -> binary32 out_k, out_v [L][T][C]. */
cg_status cg_decompress_chunk(const uint8_t *packed, uint64_t packed_bytes,
                              const uint64_t *off, const uint32_t *len,
                              const uint16_t *cdf, const uint16_t *max1,
                              const cg_shape *shape, const int32_t *bins_k,
                              const int32_t *bins_v, float *out_k,
                              float *out_v, int32_t *status,
                              cudaStream_t stream);

/* Compress without a workspace argument. The method itself has no counterpart: this
 * entry point exists for callers that cannot allocate device memory at all,
 * such as code living inside a host framework whose memory pool owns every
 * device byte and hands the codec only the tensors it works on, or a
 * latency-critical path that must not take cudaMalloc's implicit device
 * synchronisation. Inputs and outputs are as in cg_compress_chunk; the
 * scratch is a static device array inside the library of
 * CG_NOALLOC_WORKSPACE_BYTES (64 MiB, enough for one 256-token chunk of a
 * 32-layer, 1024-channel KV cache), which every GPU that loads the library
 * holds until the process exits.
 *  - Returns CG_ERR_WORKSPACE, doing nothing, when the shape needs more than
 *    CG_NOALLOC_WORKSPACE_BYTES (cg_compress_workspace_bytes(shape) >
 *    CG_NOALLOC_WORKSPACE_BYTES); CG_ERR_INVALID_ARG for an invalid shape.
 *  - Calls no allocating routine. The first call on each device looks the
 *    array's device address up (cudaGetSymbolAddress, with that device
 *    current) and caches it; make that first call before any stream capture.
 *    The cached address belongs to the device's primary context: after a
 *    cudaDeviceReset of that device it is stale, so do not call this entry
 *    point on a device that has been reset in the same process.
 *  - All calls on a device share the one array and it keeps the last call's
 *    contents (no byte of it is read before the same call wrote it). Calls
 *    that overlap on the GPU (other streams, other host threads) race on it:
 *    serialise them. */
#define CG_NOALLOC_WORKSPACE_BYTES (64ull << 20)

cg_status cg_compress_chunk_noalloc(const uint16_t *k, const uint16_t *v,
                                    const cg_shape *shape,
                                    const int32_t *bins_k,
                                    const int32_t *bins_v, uint16_t *max1,
                                    uint16_t *cdf, uint8_t *packed,
                                    uint64_t capacity, uint32_t *len,
                                    uint64_t *off, int32_t *status,
                                    cudaStream_t stream);

/* ---- format 2: side information as symbol counts ------------------------
 * The page sends, with each chunk, what the decoder needs to rebuild the
 * chunk's CDFs [CG §2.3(2), §2.4(1)]. Format 2 sends the symbol counts the
 * CDFs are built from instead of CDF entries, over each layer's own alphabet:
 *
 * A2 A = 2*MAX_l + 1 per (kv, layer): the symbols Q can produce.
 * S  count record per (chunk k, kv, l, channel c), A bytes: byte 0 is the
 *    mode s* (largest count, smallest s on ties), bytes 1..A-1 the counts of
 *    the other symbols in increasing s, one byte each (at most Tc_k / 2).
 *    Layout: rec[k] = { K: layer 0 [C][A_0], layer 1 [C][A_1], ..., then V }.
 * F2 CDF = F over the layer's A symbols, the remainder on the record's mode.
 * Q, R, P and D are format 1's. Requires chunk_tokens <= 256.
 */

/* Bytes of all count records, or 0 for an invalid shape, invalid bins or
 * chunk_tokens > 256. */
uint64_t cg_record_bytes(const cg_shape *shape, const int32_t *bins_k,
                         const int32_t *bins_v);

/* cg_compress_chunk in format 2: max1 as in format 1, rec gets the count
 * records (cg_record_bytes bytes), packed/len/off the streams coded with the
 * per-layer CDFs. Workspace: cg_compress_workspace_bytes. Any bins in
 * [4, 256] and any C; requires chunk_tokens <= 256. (Every layer alphabet
 * 2 MAX + 1 <= 64 (bins <= 65) with C % 8 == 0, k and v 16-byte aligned and
 * layer_stride % 8 == 0 takes one fused kernel; other shapes take the
 * quantise, count-and-code and pack steps, with the same output.) */
cg_status cg_compress_chunk_v2(const uint16_t *k, const uint16_t *v,
                               const cg_shape *shape, const int32_t *bins_k,
                               const int32_t *bins_v, uint16_t *max1,
                               uint8_t *rec, uint8_t *packed,
                               uint64_t capacity, uint32_t *len,
                               uint64_t *off, void *workspace,
                               uint64_t workspace_bytes, int32_t *status,
                               cudaStream_t stream);

/* cg_decompress_chunk in format 2: the CDFs come from the count records; a
 * record whose mode byte lies outside the alphabet or whose counts exceed the
 * chunk's tokens sets CG_FLAG_CORRUPT (its channel then decodes with an
 * all-ones count). */
cg_status cg_decompress_chunk_v2(const uint8_t *packed, uint64_t packed_bytes,
                                 const uint64_t *off, const uint32_t *len,
                                 const uint8_t *rec, const uint16_t *max1,
                                 const cg_shape *shape, const int32_t *bins_k,
                                 const int32_t *bins_v, float *out_k,
                                 float *out_v, int32_t *status,
                                 cudaStream_t stream);

/* ---- format 3: compact count records ------------------------------------
 * Format 2's counts without their zero bytes [CG §2.3(2)]: the CDFs, and so
 * the streams, are format 2's. Requires chunk_tokens <= 256 and every layer
 * alphabet A_l = 2*MAX_l + 1 <= 32. Slices s = (k*2 + kv)*L + l (nslice =
 * 2*L*nch), records r = s*C + c (nrec = nslice*C). One side buffer,
 * little-endian:
 * O  uint64 [nslice + 1] at byte 0: O[s] = offset of slice s's counts in V;
 *    O[nslice] = |V|;
 * M  uint8 [nrec] at byte offM = 8*(nslice + 1): each record's mode;
 * B  uint32 [nrec] at offB = offM + nrec rounded up to a multiple of 4:
 *    bit t set iff t != mode and the count of symbol t is > 0;
 * V  uint8 at offV = offB + 4*nrec (= cg_side3_fixed_bytes): for each record
 *    in order, the counts of its set bits in increasing t, one byte each.
 * Its size is offV + O[nslice]. Only the stream lengths travel with it: the
 * offsets are their exclusive scan, which the decompressor rebuilds.
 */

/* offV, or 0 when chunk_tokens > 256 or the shape is invalid. */
uint64_t cg_side3_fixed_bytes(const cg_shape *shape);
/* The largest side buffer for these bins (capacity to pass to
 * cg_compress_chunk_v3); 0 when format 3 does not apply. */
uint64_t cg_side3_max_bytes(const cg_shape *shape, const int32_t *bins_k,
                            const int32_t *bins_v);
/* Device workspace of cg_compress_chunk_v3 and cg_decompress_chunk_v3. */
uint64_t cg_workspace_bytes_v3(const cg_shape *shape, const int32_t *bins_k,
                               const int32_t *bins_v);

/* Compress in format 3 with token-locality groups of `group` (1: none):
 * max1, the side buffer (side_capacity >= cg_side3_max_bytes; its size is
 * cg_side3_fixed_bytes + O[nslice], the uint64 at byte 8*nslice), packed,
 * len and off. Requires chunk_tokens <= 256 and every layer alphabet
 * 2 MAX + 1 <= 32 (bins <= 33); side must be 8-byte aligned. */
cg_status cg_compress_chunk_v3(const uint16_t *k, const uint16_t *v,
                               const cg_shape *shape, const int32_t *bins_k,
                               const int32_t *bins_v, int32_t group,
                               uint16_t *max1, uint8_t *side,
                               uint64_t side_capacity, uint8_t *packed,
                               uint64_t capacity, uint32_t *len, uint64_t *off,
                               void *workspace, uint64_t workspace_bytes,
                               int32_t *status, cudaStream_t stream);

/* Decompress format 3 from the lengths (no offsets) and side_bytes of side
 * buffer, into out_k / out_v as cg_decompress_chunk_ex. A side buffer the
 * compressor cannot produce sets CG_FLAG_CORRUPT. */
cg_status cg_decompress_chunk_v3(const uint8_t *packed, uint64_t packed_bytes,
                                 const uint32_t *len, const uint8_t *side,
                                 uint64_t side_bytes, const uint16_t *max1,
                                 const cg_shape *shape, const int32_t *bins_k,
                                 const int32_t *bins_v, int32_t group,
                                 int out_dtype, void *out_k, void *out_v,
                                 int64_t out_layer_stride, void *workspace,
                                 uint64_t workspace_bytes, int32_t *status,
                                 cudaStream_t stream);

/* ---- serving layouts ----------------------------------------------------
 * Decompression straight into the layout a serving engine keeps its cache in
 * [CG §3.2] (K and V of a layer side by side: [L][2][T][C], i.e. out_v =
 * out_k + T*C and a layer stride of 2*T*C), as binary32 or as binary16 (each
 * binary32 value of D rounded to nearest, ties to even).
 */
#define CG_OUT_F32 0
#define CG_OUT_F16 1

/* Decode fused with dequantisation, either format (format 1: side = uint16
 * CDF entries; format 2: side = uint8 count records) and token-locality delta
 * group (1: none; see below), into out_k / out_v [L][T][C] of out_dtype with
 * layers out_layer_stride elements apart (>= T*C; tokens C apart, channels
 * contiguous). Requires chunk_tokens <= 256. Status bits as
 * cg_decompress_chunk / cg_decompress_chunk_v2. */
cg_status cg_decompress_chunk_ex(const uint8_t *packed, uint64_t packed_bytes,
                                 const uint64_t *off, const uint32_t *len,
                                 const void *side, const uint16_t *max1,
                                 const cg_shape *shape, const int32_t *bins_k,
                                 const int32_t *bins_v, int format,
                                 int32_t group, int out_dtype, void *out_k,
                                 void *out_v, int64_t out_layer_stride,
                                 int32_t *status, cudaStream_t stream);

/* ---- token-locality delta ------------------------------------------------
 * The page's design codes each token's change from a nearby token, since
 * neighbouring tokens' K/V are similar [CG §1.2(1)] (LMCache's code skips
 * this step, [CG §2.3(1)]). Read here as follows; it changes Q and D only
 * (F, S, F2, R, P code the symbols as before), for either format, with a
 * group size G >= 1 (G = 1: plain Q and D; G <= CG_MAX_CHUNK_TOKENS):
 *
 * G  within chunk k the tokens tl = 0..Tc_k-1 form groups of G consecutive
 *    tokens from tl = 0; the first of each group (tl % G == 0) is its anchor.
 * QA anchor rows: Q. The anchor's reconstruction a^_c = D(q_a,c, max1_a).
 * QD other rows: d_c = x_c - a^_c (binary32); max1 = the smallest binary16
 *    value >= max_c |d_c| (65504 when above it); q = Q's steps on d with that
 *    max1, clamped to [0, 2*MAX] (max1 == 0: q = MAX).
 * DD other rows: x^_c = a^_c + D(q_c, max1) in binary32; anchors: D. The
 *    binary16 output of cg_decompress_chunk_ex rounds x^ to nearest-even.
 * The decoder needs nothing beyond G: the anchors' symbols and max1 are in
 * the chunk.
 */

/* QA + QD over the whole tensor: outputs as cg_quantize (sym, max1). */
cg_status cg_quantize_delta(const uint16_t *k, const uint16_t *v,
                            const cg_shape *shape, const int32_t *bins_k,
                            const int32_t *bins_v, int32_t group, uint8_t *sym,
                            uint16_t *max1, int32_t *status,
                            cudaStream_t stream);

/* D / DD: sym, max1 as from cg_quantize_delta with the same group ->
 * binary32 out_k, out_v [L][T][C] contiguous (16-byte aligned). */
cg_status cg_dequantize_delta(const uint8_t *sym, const uint16_t *max1,
                              const cg_shape *shape, const int32_t *bins_k,
                              const int32_t *bins_v, int32_t group,
                              float *out_k, float *out_v, int32_t *status,
                              cudaStream_t stream);

/* Quantise (with the delta when group > 1) -> CDF or count records -> encode
 * -> pack, either format: side = uint16 CDF entries (format 1,
 * cg_cdf_elems) or uint8 count records (format 2, cg_record_bytes).
 * Workspace: cg_compress_workspace_bytes. Format 2 needs chunk_tokens <=
 * 256; format 1 takes any shape. Decode with
 * cg_decompress_chunk_ex and the same format and group (chunk_tokens <= 256),
 * or, in format 1 with any chunk size, cg_decode then cg_dequantize_delta. */
cg_status cg_compress_chunk_ex(const uint16_t *k, const uint16_t *v,
                               const cg_shape *shape, const int32_t *bins_k,
                               const int32_t *bins_v, int format,
                               int32_t group, uint16_t *max1, void *side,
                               uint8_t *packed, uint64_t capacity,
                               uint32_t *len, uint64_t *off, void *workspace,
                               uint64_t workspace_bytes, int32_t *status,
                               cudaStream_t stream);

/* Library version string ("cachegen-gb300 <formats> <options> <build>"). */
const char *cg_version(void);

#ifdef __cplusplus
}
#endif
#endif
