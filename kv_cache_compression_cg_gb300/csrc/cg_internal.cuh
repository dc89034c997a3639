// cg_internal.cuh - shared device-side definitions of the sm_103a codec.
//
// Layouts follow the codec specification in include/cachegen.h.
// Citation key: [CG] = web page "CacheGen 技术详解：KV Cache 的高效压缩与流式传输".
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/cachegen.h"

namespace cg {

// NVTX range over one ABI call, named after the entry point: a profiler or
// tracer attached to the process shows each call's launches under its name;
// with no tool attached the push and pop return at once.
struct TraceRange {
    explicit TraceRange(const char *name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};
#define CG_TRACE_RANGE() ::cg::TraceRange cg_trace_range_(__func__)

// SMs of the current device, looked up once per device (per translation unit).
inline int device_sm_count() {
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (counts[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

// Per-call geometry, passed by value to every kernel.
struct Dims {
    int L, T, C, Tc;       // layers, tokens, channels, tokens per chunk
    int nch;               // number of chunks
    int A[2];              // alphabet width of K and V
    long long layer_stride;  // elements between layers of the fp16 input
    long long nstreams;      // 2*L*T
    long long stage_bytes;   // per-stream staging bytes in the workspace
    int G;                   // token-locality delta group (1: none) [CG §1.2(1)]
};

// MAX = bins / 2 - 1 per (kv, layer) [CG §2.3(1)], in kernel parameter space.
struct MaxTab {
    unsigned char v[2][CG_MAX_LAYERS];
};

__host__ __device__ inline int chunk_tokens(const Dims &d, int k) {
    int rest = d.T - k * d.Tc;
    return rest < d.Tc ? rest : d.Tc;
}

// First stream id of chunk k; stream (k, kv, l, tl) = base + (kv*L + l)*Tc_k + tl.
__host__ __device__ inline long long chunk_stream_base(const Dims &d, int k) {
    return 2LL * d.L * d.Tc * k;
}

// First CDF entry of (k, kv, l); row c follows at + c*A[kv].
__host__ __device__ inline long long cdf_slice_offset(const Dims &d, int k, int kv, int l) {
    long long per_chunk = (long long)d.L * d.C * (d.A[0] + d.A[1]);
    long long tensor = kv ? (long long)d.L * d.C * d.A[0] : 0;
    return per_chunk * k + tensor + (long long)l * d.C * d.A[kv];
}

// Format 2: byte offset of the count records of slice (k, kv, l). Records of
// a chunk are K layer 0 [C][A_0], layer 1 [C][A_1], ..., then V, with
// A_j = 2 * MAX_j + 1. Every thread of the CTA calls this (block reduction
// over the layers; two barriers); every thread gets the offset. red is
// shared scratch of 3 * (warps) words, free again when this returns.
__device__ __forceinline__ long long record_slice_offset(const Dims &d, const MaxTab &mt, int k, int kv, int l,
                                                         unsigned long long *red) {
    unsigned long long tk = 0, tv = 0, pre = 0;
    for (int j = threadIdx.x; j < d.L; j += blockDim.x) {
        const unsigned long long ak = 2ull * mt.v[0][j] + 1, av = 2ull * mt.v[1][j] + 1;
        tk += ak;
        tv += av;
        if (j < l) pre += kv ? av : ak;
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        tk += __shfl_xor_sync(0xFFFFFFFFu, tk, o);
        tv += __shfl_xor_sync(0xFFFFFFFFu, tv, o);
        pre += __shfl_xor_sync(0xFFFFFFFFu, pre, o);
    }
    const int warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    if ((threadIdx.x & 31) == 0) {
        red[3 * warp] = tk;
        red[3 * warp + 1] = tv;
        red[3 * warp + 2] = pre;
    }
    __syncthreads();
    tk = tv = pre = 0;
    for (int w = 0; w < nw; w++) {
        tk += red[3 * w];
        tv += red[3 * w + 1];
        pre += red[3 * w + 2];
    }
    __syncthreads();
    return (long long)d.C * ((long long)k * (long long)(tk + tv) + (kv ? (long long)tk : 0LL) + (long long)pre);
}

__device__ __forceinline__ long long record_slice_offset(const Dims &d, const MaxTab &mt, int k, int kv, int l) {
    __shared__ unsigned long long red[3 * 32];
    return record_slice_offset(d, mt, k, kv, l, red);
}

// Symbols [2][L][T][C] and max1 [2][L][T].
__host__ __device__ inline long long group_index(const Dims &d, int kv, int l, long long t) {
    return ((long long)kv * d.L + l) * d.T + t;
}

// Work unit of the coders: one (chunk, kv, layer) slice of Tc_k streams.
__host__ __device__ inline void slice_coords(const Dims &d, long long b, int &k, int &kv, int &l) {
    l = (int)(b % d.L);
    long long r = b / d.L;
    kv = (int)(r % 2);
    k = (int)(r / 2);
}

// Per-stream staging area: kStagePrefix bytes of slack, then the stream's
// words (the encoder parks a placeholder word in the slack before the first
// real one, which keeps its store path free of a branch).
constexpr int kStagePrefix = 16;

__host__ __device__ inline uint8_t *stage_stream(uint8_t *stage, long long sid, const Dims &d) {
    return stage + sid * d.stage_bytes + kStagePrefix;
}

// Scan helper sizes.
constexpr int kScanBlock = 1024;      // threads per scan block
constexpr int kScanItems = 2;         // items per thread
constexpr int kScanTile = kScanBlock * kScanItems;

__host__ __device__ inline long long scan_tiles(long long n) {
    return (n + kScanTile - 1) / kScanTile;
}

// ---- launchers (each returns cudaGetLastError()) --------------------------
cudaError_t launch_quantize(const uint16_t *k, const uint16_t *v, const Dims &d,
                            const MaxTab &mt, uint8_t *sym, uint16_t *max1,
                            int32_t *status, cudaStream_t s);

// mode: 0 = count + build CDF only (cdf_out), 1 = encode with cdf_in,
//       2 = count + build CDF (cdf_out) + encode. rec != nullptr: format 2
//       (per-layer alphabets from mt, count records to rec instead of cdf_out).
cudaError_t launch_code_slices(const uint8_t *sym, const uint16_t *cdf_in,
                               uint16_t *cdf_out, uint8_t *stage, uint32_t *len,
                               const Dims &d, int mode, int32_t *status,
                               cudaStream_t s, const MaxTab *mt = nullptr,
                               uint8_t *rec = nullptr);

cudaError_t launch_scan_and_pack(const uint32_t *len, uint64_t *off,
                                 const uint8_t *stage, uint8_t *packed,
                                 uint64_t capacity, unsigned long long *partials,
                                 const Dims &d, int32_t *status, cudaStream_t s);

// off = exclusive scan of len (off[nstreams] = total); partials as for
// launch_scan_and_pack.
cudaError_t launch_offsets(const uint32_t *len, uint64_t *off, unsigned long long *partials, const Dims &d,
                           cudaStream_t s);

// Format 3 side buffer <-> format 2 count records (layout in include/cachegen.h).
// pack: totals holds nslices + 1 uint64 of scratch; side must hold the
// largest format 3 size. unpack: nbytes of side are readable; a buffer the
// encoder cannot produce sets CG_FLAG_CORRUPT (records stay in bounds).
cudaError_t launch_v3_pack(const uint8_t *rec, const Dims &d, const MaxTab &mt, uint8_t *side,
                           unsigned long long *totals, cudaStream_t s);
cudaError_t launch_v3_unpack(const uint8_t *side, unsigned long long nbytes, const Dims &d, const MaxTab &mt,
                             uint8_t *rec, int32_t *status, cudaStream_t s);
// Byte offsets of the format 3 parts: M at offM, B at offB, V at offV.
__host__ __device__ inline void v3_layout(const Dims &d, long long &offM, long long &offB, long long &offV) {
    const long long ns = 2LL * d.L * d.nch, nrec = ns * d.C;
    offM = 8 * (ns + 1);
    offB = (offM + nrec + 3) / 4 * 4;
    offV = offB + 4 * nrec;
}

// Fused quantise + CDF + encode straight from fp16 (chunks <= 256 tokens,
// A <= 64, C % 8 == 0, 16-byte aligned rows); compress_fused_applies says when.
bool compress_fused_applies(const Dims &d, const uint16_t *k, const uint16_t *v);
// Writes max1, cdf, len, off (incl. off[nstreams]) and packed; `state` holds
// 2 + 2 * nslices uint64 words (two tickets, a look-back slot and a byte total
// per slice), set up by the launch itself.
// cdf != nullptr: format 1 (CDF entries out); otherwise rec gets format 2's
// count records.
cudaError_t launch_compress_fused(const uint16_t *k, const uint16_t *v, const Dims &d,
                                  const MaxTab &mt, uint16_t *max1, uint16_t *cdf, uint8_t *rec,
                                  uint8_t *stage, uint32_t *len, uint64_t *off,
                                  uint8_t *packed, uint64_t capacity,
                                  unsigned long long *state, int32_t *status,
                                  cudaStream_t s);

// mode: 0 = symbols out (sym), 1 = dequantised binary32 out (out_k, out_v).
cudaError_t launch_decode(const uint8_t *packed, uint64_t packed_bytes,
                          const uint64_t *off, const uint32_t *len,
                          const uint16_t *cdf, const uint16_t *max1,
                          const Dims &d, const MaxTab &mt, int mode, uint8_t *sym,
                          float *out_k, float *out_v, int32_t *status,
                          cudaStream_t s);

// Chunks of up to 256 tokens; rec != nullptr selects format 2 (CDF rows from
// the count records, cdf unused). out_dtype 1: binary32, 2: binary16 (rounded
// to nearest-even); outputs [L][T][C] with layers `ols` elements apart.
cudaError_t launch_decode_pipe(const uint8_t *packed, uint64_t packed_bytes,
                               const uint64_t *off, const uint32_t *len,
                               const uint16_t *cdf, const uint8_t *rec,
                               const uint16_t *max1, const Dims &d, const MaxTab &mt,
                               int out_dtype, void *out_k, void *out_v, long long ols,
                               int32_t *status, cudaStream_t s);

// launch_decode_pipe for d.G > 1 (the token-locality delta).
cudaError_t launch_decode_pipe_delta(const uint8_t *packed, uint64_t packed_bytes,
                                     const uint64_t *off, const uint32_t *len,
                                     const uint16_t *cdf, const uint8_t *rec,
                                     const uint16_t *max1, const Dims &d, const MaxTab &mt,
                                     int out_dtype, void *out_k, void *out_v, long long ols,
                                     int32_t *status, cudaStream_t s);

// Any chunk size up to CG_MAX_CHUNK_TOKENS (used by launch_decode beyond 256).
cudaError_t launch_decode_generic(const uint8_t *packed, uint64_t packed_bytes,
                                  const uint64_t *off, const uint32_t *len,
                                  const uint16_t *cdf, const uint16_t *max1,
                                  const Dims &d, const MaxTab &mt, int mode,
                                  uint8_t *sym, float *out_k, float *out_v,
                                  int32_t *status, cudaStream_t s);

cudaError_t launch_dequantize(const uint8_t *sym, const uint16_t *max1,
                              const Dims &d, const MaxTab &mt, float *out_k,
                              float *out_v, cudaStream_t s);

// Token-locality delta (d.G > 1): anchors quantised as above, the other rows
// of each group as deltas from the anchor's reconstruction; dequantisation
// adds the reconstruction back. Binary32 output [L][T][C].
cudaError_t launch_quantize_delta(const uint16_t *k, const uint16_t *v, const Dims &d,
                                  const MaxTab &mt, uint8_t *sym, uint16_t *max1,
                                  int32_t *status, cudaStream_t s);
cudaError_t launch_dequantize_delta(const uint8_t *sym, const uint16_t *max1,
                                    const Dims &d, const MaxTab &mt, float *out_k,
                                    float *out_v, cudaStream_t s);

// Token groups of the delta: chunk-local, G tokens from each chunk's first.
__host__ __device__ inline long long delta_groups_per_chunk(const Dims &d) {
    return (d.Tc + d.G - 1) / d.G;
}
// Work unit `task` -> (kv, l), the anchor's token t_a and the group's rows n
// (n <= 0: past the end of a short last chunk).
__host__ __device__ inline void delta_task(const Dims &d, long long task, int &kv, int &l, long long &t_a, int &n) {
    const long long gpc = delta_groups_per_chunk(d);
    const int g = (int)(task % gpc);
    long long r = task / gpc;
    const int k = (int)(r % d.nch);
    r /= d.nch;
    l = (int)(r % d.L);
    kv = (int)(r / d.L);
    const int Tk = chunk_tokens(d, k);
    t_a = (long long)k * d.Tc + (long long)g * d.G;
    n = min(d.G, Tk - g * d.G);
}

}  // namespace cg
