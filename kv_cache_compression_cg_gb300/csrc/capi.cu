// capi.cu - the C ABI of include/cachegen.h: argument checks on the host,
// workspace carving, and kernel launches on the caller's stream. Nothing here
// allocates or synchronises.
#include <cstring>

#include "cg_internal.cuh"

namespace {

using cg::Dims;
using cg::MaxTab;

constexpr uint64_t kAlign = 256;

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

bool shape_ok(const cg_shape *s) {
    if (!s) return false;
    if (s->L < 1 || s->L > CG_MAX_LAYERS) return false;
    if (s->T < 0) return false;
    if (s->C < 1 || s->C > CG_MAX_CHANNELS) return false;
    if (s->chunk_tokens < 1 || s->chunk_tokens > CG_MAX_CHUNK_TOKENS) return false;
    if (s->layer_stride < (int64_t)s->T * s->C) return false;
    return true;
}

bool bins_ok(const int32_t *b, int L) {
    if (!b) return false;
    for (int l = 0; l < L; l++)
        if (b[l] < 4 || b[l] > 256) return false;
    return true;
}

int alphabet(const int32_t *b, int L) {
    int a = 0;
    for (int l = 0; l < L; l++) a = b[l] > a ? b[l] : a;
    return a;
}

uint64_t stage_bytes_per_stream(int C) {
    // slack prefix, then up to 2*C + 8 stream bytes; the last word store may
    // run 3 bytes past the stream's end
    return cg::kStagePrefix + round_up(2ull * (uint64_t)C + 12ull, 16);
}

// Fill dims and the MAX table; false on invalid shape/bins.
bool prepare(const cg_shape *s, const int32_t *bins_k, const int32_t *bins_v, Dims &d, MaxTab *mt) {
    if (!shape_ok(s)) return false;
    if (!bins_v) bins_v = bins_k;
    if (!bins_ok(bins_k, s->L) || !bins_ok(bins_v, s->L)) return false;
    d.L = s->L;
    d.T = s->T;
    d.C = s->C;
    d.Tc = s->chunk_tokens;
    d.nch = (s->T + s->chunk_tokens - 1) / s->chunk_tokens;
    d.A[0] = alphabet(bins_k, s->L);
    d.A[1] = alphabet(bins_v, s->L);
    d.layer_stride = s->layer_stride;
    d.nstreams = 2LL * s->L * s->T;
    d.stage_bytes = (long long)stage_bytes_per_stream(s->C);
    d.G = 1;
    if (mt) {
        std::memset(mt, 0, sizeof(*mt));
        for (int l = 0; l < s->L; l++) {
            mt->v[0][l] = (unsigned char)(bins_k[l] / 2 - 1);
            mt->v[1][l] = (unsigned char)(bins_v[l] / 2 - 1);
        }
    }
    return true;
}

struct Workspace {
    uint8_t *stage;
    unsigned long long *partials;
    uint8_t *sym;
    unsigned long long *state;  // fused compress: two tickets, a look-back slot and a total per slice
};

uint64_t encode_ws_bytes(const Dims &d) {
    const uint64_t stage = round_up((uint64_t)d.nstreams * (uint64_t)d.stage_bytes, kAlign);
    const uint64_t parts = round_up(8ull * (uint64_t)(cg::scan_tiles(d.nstreams) + 1), kAlign);
    return stage + parts;
}

uint64_t sym_bytes(const Dims &d) { return round_up(2ull * d.L * (uint64_t)d.T * d.C, kAlign); }

uint64_t state_bytes(const Dims &d) { return round_up(8ull * (2ull + 4ull * d.L * d.nch), kAlign); }

Workspace carve(void *ws, const Dims &d, bool with_sym) {
    Workspace w;
    uint8_t *p = static_cast<uint8_t *>(ws);
    w.stage = p;
    p += round_up((uint64_t)d.nstreams * (uint64_t)d.stage_bytes, kAlign);
    w.partials = reinterpret_cast<unsigned long long *>(p);
    p += round_up(8ull * (uint64_t)(cg::scan_tiles(d.nstreams) + 1), kAlign);
    w.sym = with_sym ? p : nullptr;
    if (with_sym) p += sym_bytes(d);
    w.state = with_sym ? reinterpret_cast<unsigned long long *>(p) : nullptr;
    return w;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Format 2: layer alphabet 2*MAX + 1, records C * sum_l A_l per tensor and chunk.
uint64_t record_bytes(const Dims &d, const MaxTab &mt) {
    uint64_t per = 0;
    for (int kv = 0; kv < 2; kv++)
        for (int l = 0; l < d.L; l++) per += 2ull * mt.v[kv][l] + 1;
    return (uint64_t)d.nch * (uint64_t)d.C * per;
}

int max_alphabet_v2(const Dims &d, const MaxTab &mt) {
    int a = 0;
    for (int kv = 0; kv < 2; kv++)
        for (int l = 0; l < d.L; l++) a = 2 * mt.v[kv][l] + 1 > a ? 2 * mt.v[kv][l] + 1 : a;
    return a;
}

cg_status launched(cudaError_t e) { return e == cudaSuccess ? CG_OK : CG_ERR_CUDA; }

bool group_ok(int32_t g) { return g >= 1 && g <= CG_MAX_CHUNK_TOKENS; }

// Format 3: chunks of at most 256 tokens and every layer alphabet within a
// 32-bit presence mask.
bool v3_ok(const Dims &d, const MaxTab &mt) { return d.Tc <= 256 && max_alphabet_v2(d, mt) <= 32; }

uint64_t v3_fixed_bytes(const Dims &d) {
    long long offM, offB, offV;
    cg::v3_layout(d, offM, offB, offV);
    return (uint64_t)offV;
}

uint64_t v3_max_bytes(const Dims &d, const MaxTab &mt) {
    uint64_t per = 0;
    for (int kv = 0; kv < 2; kv++)
        for (int l = 0; l < d.L; l++) per += 2ull * mt.v[kv][l];  // A - 1 count bytes at most
    return v3_fixed_bytes(d) + (uint64_t)d.nch * (uint64_t)d.C * per;
}

// Format 3 scratch: compress = the fused compress workspace, the format 2
// records and the slice totals; decompress = offsets, scan partials and the
// records. One size covers both.
uint64_t v3_workspace_bytes(const Dims &d, const MaxTab &mt) {
    const uint64_t rec = round_up(record_bytes(d, mt), kAlign);
    const uint64_t comp = encode_ws_bytes(d) + sym_bytes(d) + state_bytes(d) + rec +
                          round_up(8ull * (2ull * d.L * d.nch + 1), kAlign);
    const uint64_t dec = round_up(8ull * (d.nstreams + 1), kAlign) +
                         round_up(8ull * (uint64_t)(cg::scan_tiles(d.nstreams) + 1), kAlign) + rec;
    return comp > dec ? comp : dec;
}

// Empty token range: only off[0] = 0 has to be written.
cg_status empty_offsets(uint64_t *off, cudaStream_t stream) {
    if (!off) return CG_OK;
    return launched(cudaMemsetAsync(off, 0, sizeof(uint64_t), stream));
}

}  // namespace

extern "C" {

uint64_t cg_num_streams(const cg_shape *shape) {
    return shape_ok(shape) ? 2ull * (uint64_t)shape->L * (uint64_t)shape->T : 0;
}

uint64_t cg_cdf_elems(const cg_shape *shape, const int32_t *bins_k, const int32_t *bins_v) {
    Dims d;
    if (!prepare(shape, bins_k, bins_v, d, nullptr)) return 0;
    return (uint64_t)d.nch * d.L * (uint64_t)d.C * (uint64_t)(d.A[0] + d.A[1]);
}

uint64_t cg_max_compressed_bytes(const cg_shape *shape) {
    if (!shape_ok(shape)) return 0;
    return 2ull * shape->L * (uint64_t)shape->T * (2ull * shape->C + 8ull);
}

uint64_t cg_workspace_bytes(const cg_shape *shape) {
    if (!shape_ok(shape)) return 0;
    Dims d;
    int32_t b[CG_MAX_LAYERS];
    for (int l = 0; l < shape->L; l++) b[l] = 4;
    prepare(shape, b, b, d, nullptr);
    return encode_ws_bytes(d);
}

uint64_t cg_compress_workspace_bytes(const cg_shape *shape) {
    if (!shape_ok(shape)) return 0;
    Dims d;
    int32_t b[CG_MAX_LAYERS];
    for (int l = 0; l < shape->L; l++) b[l] = 4;
    prepare(shape, b, b, d, nullptr);
    return encode_ws_bytes(d) + sym_bytes(d) + state_bytes(d);
}

const char *cg_version(void) { return "cachegen-gb300 formats-1,2,3 delta sm_103a"; }

cg_status cg_quantize(const uint16_t *k, const uint16_t *v, const cg_shape *shape,
                      const int32_t *bins_k, const int32_t *bins_v, uint8_t *sym, uint16_t *max1,
                      int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt)) return CG_ERR_INVALID_ARG;
    if (!k || !v || !sym || !max1 || !aligned(k, 2) || !aligned(v, 2) || !aligned(max1, 2))
        return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    return launched(cg::launch_quantize(k, v, d, mt, sym, max1, status, stream));
}

cg_status cg_calculate_cdf(const uint8_t *sym, const cg_shape *shape, const int32_t *bins_k,
                           const int32_t *bins_v, uint16_t *cdf, int32_t *status,
                           cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    if (!prepare(shape, bins_k, bins_v, d, nullptr)) return CG_ERR_INVALID_ARG;
    if (!sym || !cdf || !aligned(cdf, 2)) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    return launched(cg::launch_code_slices(sym, nullptr, cdf, nullptr, nullptr, d, 0, status, stream));
}

cg_status cg_encode(const uint8_t *sym, const uint16_t *cdf, const cg_shape *shape,
                    const int32_t *bins_k, const int32_t *bins_v, uint8_t *packed,
                    uint64_t capacity, uint32_t *len, uint64_t *off, void *workspace,
                    uint64_t workspace_bytes, int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    if (!prepare(shape, bins_k, bins_v, d, nullptr)) return CG_ERR_INVALID_ARG;
    if (!off) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return empty_offsets(off, stream);
    if (!sym || !cdf || !len || !workspace || (!packed && capacity > 0)) return CG_ERR_INVALID_ARG;
    if (!aligned(cdf, 2) || !aligned(len, 4) || !aligned(off, 8) || !aligned(workspace, kAlign))
        return CG_ERR_INVALID_ARG;
    if (workspace_bytes < encode_ws_bytes(d)) return CG_ERR_WORKSPACE;
    Workspace w = carve(workspace, d, false);
    cudaError_t e = cg::launch_code_slices(sym, cdf, nullptr, w.stage, len, d, 1, status, stream);
    if (e != cudaSuccess) return CG_ERR_CUDA;
    return launched(cg::launch_scan_and_pack(len, off, w.stage, packed, capacity, w.partials, d,
                                             status, stream));
}

cg_status cg_decode(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                    const uint32_t *len, const uint16_t *cdf, const cg_shape *shape,
                    const int32_t *bins_k, const int32_t *bins_v, uint8_t *sym, int32_t *status,
                    cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt)) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    if (!packed || !off || !len || !cdf || !sym) return CG_ERR_INVALID_ARG;
    if (!aligned(packed, 4) || !aligned(off, 8) || !aligned(len, 4) || !aligned(cdf, 2))
        return CG_ERR_INVALID_ARG;
    return launched(cg::launch_decode(packed, packed_bytes, off, len, cdf, nullptr, d, mt, 0, sym,
                                      nullptr, nullptr, status, stream));
}

cg_status cg_dequantize(const uint8_t *sym, const uint16_t *max1, const cg_shape *shape,
                        const int32_t *bins_k, const int32_t *bins_v, float *out_k, float *out_v,
                        int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    (void)status;
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt)) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    if (!sym || !max1 || !out_k || !out_v || !aligned(max1, 2) || !aligned(out_k, 16) ||
        !aligned(out_v, 16) || !aligned(sym, 4))
        return CG_ERR_INVALID_ARG;
    return launched(cg::launch_dequantize(sym, max1, d, mt, out_k, out_v, stream));
}

cg_status cg_compress_chunk(const uint16_t *k, const uint16_t *v, const cg_shape *shape,
                            const int32_t *bins_k, const int32_t *bins_v, uint16_t *max1,
                            uint16_t *cdf, uint8_t *packed, uint64_t capacity, uint32_t *len,
                            uint64_t *off, void *workspace, uint64_t workspace_bytes,
                            int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt)) return CG_ERR_INVALID_ARG;
    if (!off) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return empty_offsets(off, stream);
    if (!k || !v || !max1 || !cdf || !len || !workspace || (!packed && capacity > 0))
        return CG_ERR_INVALID_ARG;
    if (!aligned(k, 2) || !aligned(v, 2) || !aligned(max1, 2) || !aligned(cdf, 2) ||
        !aligned(len, 4) || !aligned(off, 8) || !aligned(workspace, kAlign))
        return CG_ERR_INVALID_ARG;
    if (workspace_bytes < encode_ws_bytes(d) + sym_bytes(d) + state_bytes(d)) return CG_ERR_WORKSPACE;
    Workspace w = carve(workspace, d, true);
    if (cg::compress_fused_applies(d, k, v))
        return launched(cg::launch_compress_fused(k, v, d, mt, max1, cdf, nullptr, w.stage, len, off, packed,
                                                  capacity, w.state, status, stream));
    if (cg::launch_quantize(k, v, d, mt, w.sym, max1, status, stream) != cudaSuccess) return CG_ERR_CUDA;
    if (cg::launch_code_slices(w.sym, nullptr, cdf, w.stage, len, d, 2, status, stream) != cudaSuccess)
        return CG_ERR_CUDA;
    return launched(cg::launch_scan_and_pack(len, off, w.stage, packed, capacity, w.partials, d,
                                             status, stream));
}

cg_status cg_decompress_chunk(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                              const uint32_t *len, const uint16_t *cdf, const uint16_t *max1,
                              const cg_shape *shape, const int32_t *bins_k, const int32_t *bins_v,
                              float *out_k, float *out_v, int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt)) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    if (!packed || !off || !len || !cdf || !max1 || !out_k || !out_v) return CG_ERR_INVALID_ARG;
    if (!aligned(packed, 4) || !aligned(off, 8) || !aligned(len, 4) || !aligned(cdf, 2) ||
        !aligned(max1, 2) || !aligned(out_k, 16) || !aligned(out_v, 16))
        return CG_ERR_INVALID_ARG;
    return launched(cg::launch_decode(packed, packed_bytes, off, len, cdf, max1, d, mt, 1, nullptr,
                                      out_k, out_v, status, stream));
}

uint64_t cg_record_bytes(const cg_shape *shape, const int32_t *bins_k, const int32_t *bins_v) {
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || d.Tc > 256) return 0;
    return record_bytes(d, mt);
}

cg_status cg_compress_chunk_v2(const uint16_t *k, const uint16_t *v, const cg_shape *shape,
                               const int32_t *bins_k, const int32_t *bins_v, uint16_t *max1, uint8_t *rec,
                               uint8_t *packed, uint64_t capacity, uint32_t *len, uint64_t *off,
                               void *workspace, uint64_t workspace_bytes, int32_t *status,
                               cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || d.Tc > 256) return CG_ERR_INVALID_ARG;
    if (!off) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return empty_offsets(off, stream);
    if (!k || !v || !max1 || !rec || !len || !workspace || (!packed && capacity > 0)) return CG_ERR_INVALID_ARG;
    if (!aligned(k, 2) || !aligned(v, 2) || !aligned(max1, 2) || !aligned(len, 4) || !aligned(off, 8) ||
        !aligned(workspace, kAlign))
        return CG_ERR_INVALID_ARG;
    if (workspace_bytes < encode_ws_bytes(d) + sym_bytes(d) + state_bytes(d)) return CG_ERR_WORKSPACE;
    // the fused kernel where its limits allow (with format 2's alphabet), else
    // the step path: quantise, then count -> records and CDF rows -> code
    Dims d2 = d;
    d2.A[0] = d2.A[1] = max_alphabet_v2(d, mt);
    Workspace w = carve(workspace, d, true);
    if (cg::compress_fused_applies(d2, k, v))
        return launched(cg::launch_compress_fused(k, v, d, mt, max1, nullptr, rec, w.stage, len, off, packed,
                                                  capacity, w.state, status, stream));
    if (cg::launch_quantize(k, v, d, mt, w.sym, max1, status, stream) != cudaSuccess) return CG_ERR_CUDA;
    if (cg::launch_code_slices(w.sym, nullptr, nullptr, w.stage, len, d, 2, status, stream, &mt, rec) !=
        cudaSuccess)
        return CG_ERR_CUDA;
    return launched(cg::launch_scan_and_pack(len, off, w.stage, packed, capacity, w.partials, d, status, stream));
}

cg_status cg_decompress_chunk_v2(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                                 const uint32_t *len, const uint8_t *rec, const uint16_t *max1,
                                 const cg_shape *shape, const int32_t *bins_k, const int32_t *bins_v,
                                 float *out_k, float *out_v, int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || d.Tc > 256) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    if (!packed || !off || !len || !rec || !max1 || !out_k || !out_v) return CG_ERR_INVALID_ARG;
    if (!aligned(packed, 4) || !aligned(off, 8) || !aligned(len, 4) || !aligned(max1, 2) ||
        !aligned(out_k, 16) || !aligned(out_v, 16))
        return CG_ERR_INVALID_ARG;
    return launched(cg::launch_decode_pipe(packed, packed_bytes, off, len, nullptr, rec, max1, d, mt, 1, out_k,
                                           out_v, (long long)d.T * d.C, status, stream));
}

cg_status cg_decompress_chunk_ex(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                                 const uint32_t *len, const void *side, const uint16_t *max1,
                                 const cg_shape *shape, const int32_t *bins_k, const int32_t *bins_v, int format,
                                 int32_t group, int out_dtype, void *out_k, void *out_v,
                                 int64_t out_layer_stride, int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || d.Tc > 256) return CG_ERR_INVALID_ARG;
    if ((format != 1 && format != 2) || (out_dtype != CG_OUT_F32 && out_dtype != CG_OUT_F16) || !group_ok(group))
        return CG_ERR_INVALID_ARG;
    d.G = group;
    if (out_layer_stride < (int64_t)d.T * d.C) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    const uintptr_t es = out_dtype == CG_OUT_F16 ? 2 : 4;
    if (!packed || !off || !len || !side || !max1 || !out_k || !out_v) return CG_ERR_INVALID_ARG;
    if (!aligned(packed, 4) || !aligned(off, 8) || !aligned(len, 4) || !aligned(max1, 2) ||
        !aligned(side, format == 1 ? 2 : 1) || !aligned(out_k, es) || !aligned(out_v, es))
        return CG_ERR_INVALID_ARG;
    const uint16_t *cdf = format == 1 ? static_cast<const uint16_t *>(side) : nullptr;
    const uint8_t *rec = format == 2 ? static_cast<const uint8_t *>(side) : nullptr;
    return launched(cg::launch_decode_pipe(packed, packed_bytes, off, len, cdf, rec, max1, d, mt,
                                           out_dtype == CG_OUT_F16 ? 2 : 1, out_k, out_v, out_layer_stride, status,
                                           stream));
}

cg_status cg_quantize_delta(const uint16_t *k, const uint16_t *v, const cg_shape *shape, const int32_t *bins_k,
                            const int32_t *bins_v, int32_t group, uint8_t *sym, uint16_t *max1, int32_t *status,
                            cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || !group_ok(group)) return CG_ERR_INVALID_ARG;
    if (!k || !v || !sym || !max1 || !aligned(k, 2) || !aligned(v, 2) || !aligned(max1, 2))
        return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    d.G = group;
    if (group == 1) return launched(cg::launch_quantize(k, v, d, mt, sym, max1, status, stream));
    return launched(cg::launch_quantize_delta(k, v, d, mt, sym, max1, status, stream));
}

cg_status cg_dequantize_delta(const uint8_t *sym, const uint16_t *max1, const cg_shape *shape,
                              const int32_t *bins_k, const int32_t *bins_v, int32_t group, float *out_k,
                              float *out_v, int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    (void)status;
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || !group_ok(group)) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    if (!sym || !max1 || !out_k || !out_v || !aligned(max1, 2) || !aligned(out_k, 16) || !aligned(out_v, 16) ||
        !aligned(sym, 4))
        return CG_ERR_INVALID_ARG;
    d.G = group;
    if (group == 1) return launched(cg::launch_dequantize(sym, max1, d, mt, out_k, out_v, stream));
    return launched(cg::launch_dequantize_delta(sym, max1, d, mt, out_k, out_v, stream));
}

cg_status cg_compress_chunk_ex(const uint16_t *k, const uint16_t *v, const cg_shape *shape, const int32_t *bins_k,
                               const int32_t *bins_v, int format, int32_t group, uint16_t *max1, void *side,
                               uint8_t *packed, uint64_t capacity, uint32_t *len, uint64_t *off, void *workspace,
                               uint64_t workspace_bytes, int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || !group_ok(group) || (format != 1 && format != 2))
        return CG_ERR_INVALID_ARG;
    if (format == 2 && d.Tc > 256) return CG_ERR_INVALID_ARG;
    if (!off) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return empty_offsets(off, stream);
    if (!k || !v || !max1 || !side || !len || !workspace || (!packed && capacity > 0)) return CG_ERR_INVALID_ARG;
    if (!aligned(k, 2) || !aligned(v, 2) || !aligned(max1, 2) || !aligned(side, format == 1 ? 2 : 1) ||
        !aligned(len, 4) || !aligned(off, 8) || !aligned(workspace, kAlign))
        return CG_ERR_INVALID_ARG;
    if (workspace_bytes < encode_ws_bytes(d) + sym_bytes(d) + state_bytes(d)) return CG_ERR_WORKSPACE;
    d.G = group;
    Workspace w = carve(workspace, d, true);
    uint16_t *cdf = format == 1 ? static_cast<uint16_t *>(side) : nullptr;
    uint8_t *rec = format == 2 ? static_cast<uint8_t *>(side) : nullptr;
    Dims df = d;  // the fused kernel's limits, with format 2's alphabet
    if (format == 2) df.A[0] = df.A[1] = max_alphabet_v2(d, mt);
    if (cg::compress_fused_applies(df, k, v))
        return launched(cg::launch_compress_fused(k, v, d, mt, max1, cdf, rec, w.stage, len, off, packed, capacity,
                                                  w.state, status, stream));
    cudaError_t e = group == 1 ? cg::launch_quantize(k, v, d, mt, w.sym, max1, status, stream)
                               : cg::launch_quantize_delta(k, v, d, mt, w.sym, max1, status, stream);
    if (e != cudaSuccess) return CG_ERR_CUDA;
    if (cg::launch_code_slices(w.sym, nullptr, cdf, w.stage, len, d, 2, status, stream, &mt, rec) != cudaSuccess)
        return CG_ERR_CUDA;
    return launched(cg::launch_scan_and_pack(len, off, w.stage, packed, capacity, w.partials, d, status, stream));
}

uint64_t cg_side3_fixed_bytes(const cg_shape *shape) {
    Dims d;
    int32_t b[CG_MAX_LAYERS];
    if (!shape_ok(shape)) return 0;
    for (int l = 0; l < shape->L; l++) b[l] = 4;
    prepare(shape, b, b, d, nullptr);
    return d.Tc <= 256 ? v3_fixed_bytes(d) : 0;
}

uint64_t cg_side3_max_bytes(const cg_shape *shape, const int32_t *bins_k, const int32_t *bins_v) {
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || !v3_ok(d, mt)) return 0;
    return v3_max_bytes(d, mt);
}

uint64_t cg_workspace_bytes_v3(const cg_shape *shape, const int32_t *bins_k, const int32_t *bins_v) {
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || !v3_ok(d, mt)) return 0;
    return v3_workspace_bytes(d, mt);
}

cg_status cg_compress_chunk_v3(const uint16_t *k, const uint16_t *v, const cg_shape *shape, const int32_t *bins_k,
                               const int32_t *bins_v, int32_t group, uint16_t *max1, uint8_t *side,
                               uint64_t side_capacity, uint8_t *packed, uint64_t capacity, uint32_t *len,
                               uint64_t *off, void *workspace, uint64_t workspace_bytes, int32_t *status,
                               cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || !v3_ok(d, mt) || !group_ok(group)) return CG_ERR_INVALID_ARG;
    if (!off) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return empty_offsets(off, stream);
    if (!k || !v || !max1 || !side || !len || !workspace || (!packed && capacity > 0)) return CG_ERR_INVALID_ARG;
    if (!aligned(k, 2) || !aligned(v, 2) || !aligned(max1, 2) || !aligned(side, 8) || !aligned(len, 4) ||
        !aligned(off, 8) || !aligned(workspace, kAlign))
        return CG_ERR_INVALID_ARG;
    if (side_capacity < v3_max_bytes(d, mt)) return CG_ERR_INVALID_ARG;
    if (workspace_bytes < v3_workspace_bytes(d, mt)) return CG_ERR_WORKSPACE;
    d.G = group;
    Dims d2 = d;  // the fused kernel's limits, with format 2's alphabet
    d2.A[0] = d2.A[1] = max_alphabet_v2(d, mt);
    Workspace w = carve(workspace, d, true);
    uint8_t *rec = static_cast<uint8_t *>(workspace) + encode_ws_bytes(d) + sym_bytes(d) + state_bytes(d);
    auto *totals = reinterpret_cast<unsigned long long *>(rec + round_up(record_bytes(d, mt), kAlign));
    if (cg::compress_fused_applies(d2, k, v)) {
        if (cg::launch_compress_fused(k, v, d, mt, max1, nullptr, rec, w.stage, len, off, packed, capacity, w.state,
                                      status, stream) != cudaSuccess)
            return CG_ERR_CUDA;
    } else {  // the step path (any C, unaligned inputs)
        cudaError_t e = group == 1 ? cg::launch_quantize(k, v, d, mt, w.sym, max1, status, stream)
                                   : cg::launch_quantize_delta(k, v, d, mt, w.sym, max1, status, stream);
        if (e != cudaSuccess) return CG_ERR_CUDA;
        if (cg::launch_code_slices(w.sym, nullptr, nullptr, w.stage, len, d, 2, status, stream, &mt, rec) !=
            cudaSuccess)
            return CG_ERR_CUDA;
        if (cg::launch_scan_and_pack(len, off, w.stage, packed, capacity, w.partials, d, status, stream) !=
            cudaSuccess)
            return CG_ERR_CUDA;
    }
    return launched(cg::launch_v3_pack(rec, d, mt, side, totals, stream));
}

cg_status cg_decompress_chunk_v3(const uint8_t *packed, uint64_t packed_bytes, const uint32_t *len,
                                 const uint8_t *side, uint64_t side_bytes, const uint16_t *max1,
                                 const cg_shape *shape, const int32_t *bins_k, const int32_t *bins_v,
                                 int32_t group, int out_dtype, void *out_k, void *out_v, int64_t out_layer_stride,
                                 void *workspace, uint64_t workspace_bytes, int32_t *status, cudaStream_t stream) {
    CG_TRACE_RANGE();
    Dims d;
    MaxTab mt;
    if (!prepare(shape, bins_k, bins_v, d, &mt) || !v3_ok(d, mt) || !group_ok(group)) return CG_ERR_INVALID_ARG;
    if (out_dtype != CG_OUT_F32 && out_dtype != CG_OUT_F16) return CG_ERR_INVALID_ARG;
    if (out_layer_stride < (int64_t)d.T * d.C) return CG_ERR_INVALID_ARG;
    if (d.T == 0) return CG_OK;
    const uintptr_t es = out_dtype == CG_OUT_F16 ? 2 : 4;
    if (!packed || !len || !side || !max1 || !out_k || !out_v || !workspace) return CG_ERR_INVALID_ARG;
    if (!aligned(packed, 4) || !aligned(len, 4) || !aligned(side, 8) || !aligned(max1, 2) || !aligned(out_k, es) ||
        !aligned(out_v, es) || !aligned(workspace, kAlign))
        return CG_ERR_INVALID_ARG;
    if (side_bytes < v3_fixed_bytes(d)) return CG_ERR_INVALID_ARG;
    if (workspace_bytes < v3_workspace_bytes(d, mt)) return CG_ERR_WORKSPACE;
    d.G = group;
    uint8_t *p = static_cast<uint8_t *>(workspace);
    auto *off = reinterpret_cast<uint64_t *>(p);
    p += round_up(8ull * (d.nstreams + 1), kAlign);
    auto *partials = reinterpret_cast<unsigned long long *>(p);
    p += round_up(8ull * (uint64_t)(cg::scan_tiles(d.nstreams) + 1), kAlign);
    uint8_t *rec = p;
    if (cg::launch_offsets(len, off, partials, d, stream) != cudaSuccess) return CG_ERR_CUDA;
    if (cg::launch_v3_unpack(side, side_bytes, d, mt, rec, status, stream) != cudaSuccess) return CG_ERR_CUDA;
    return launched(cg::launch_decode_pipe(packed, packed_bytes, off, len, nullptr, rec, max1, d, mt,
                                           out_dtype == CG_OUT_F16 ? 2 : 1, out_k, out_v, out_layer_stride, status,
                                           stream));
}

}  // extern "C"
