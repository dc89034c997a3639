// noalloc.cu - cg_compress_chunk_noalloc: the fused compress with its scratch
// in a static device array owned by the library instead of a caller workspace.
//
// Meant for callers that cannot allocate device memory at all: code running
// under a host framework whose memory pool owns every device byte and hands
// the codec only the tensors it works on, or a latency-critical path that must
// not take cudaMalloc's implicit device synchronisation. They pass inputs and
// outputs as usual; the scratch comes from g_noalloc_workspace below.
#include <mutex>

#include "cg_internal.cuh"

namespace {

// The library's own compress scratch. Every GPU that loads the library holds
// it until the process exits; every call on that GPU shares it.
static __device__ __align__(256) unsigned char g_noalloc_workspace[CG_NOALLOC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the static array on the current device, looked up once per
// device (with that device current) and cached. Host code cannot pass the
// array's name to a kernel: on the host that name is a stand-in, not a device
// address.
cg_status noalloc_workspace(void **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess || p == nullptr)
            return CG_ERR_CUDA;
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return CG_OK;
}

}  // namespace

extern "C" cg_status cg_compress_chunk_noalloc(const uint16_t *k, const uint16_t *v,
                                               const cg_shape *shape, const int32_t *bins_k,
                                               const int32_t *bins_v, uint16_t *max1,
                                               uint16_t *cdf, uint8_t *packed, uint64_t capacity,
                                               uint32_t *len, uint64_t *off, int32_t *status,
                                               cudaStream_t stream) {
    CG_TRACE_RANGE();
    const uint64_t need = cg_compress_workspace_bytes(shape);
    if (need == 0) return CG_ERR_INVALID_ARG;
    if (need > CG_NOALLOC_WORKSPACE_BYTES) return CG_ERR_WORKSPACE;
    void *ws = nullptr;
    const cg_status st = noalloc_workspace(&ws);
    if (st != CG_OK) return st;
    return cg_compress_chunk(k, v, shape, bins_k, bins_v, max1, cdf, packed, capacity, len, off, ws,
                             CG_NOALLOC_WORKSPACE_BYTES, status, stream);
}
