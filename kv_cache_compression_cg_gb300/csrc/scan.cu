// scan.cu - stream-length scan and packing (format P: streams back to back
// in stream-id order, uint64 exclusive offsets) on sm_103a.
//
// Three launches, no inter-CTA waiting: tile totals, one CTA scanning the
// tile totals, then each tile rescans its lengths, writes off[] and copies its
// streams from the per-stream staging area into the packed buffer (only
// destination bytes below the capacity are written).
#include "cg_internal.cuh"

namespace cg {
namespace {

__device__ __forceinline__ unsigned long long block_inclusive_scan(unsigned long long v,
                                                                   unsigned long long *warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        const int nw = blockDim.x >> 5;
        unsigned long long w = lane < nw ? warp_sums[lane] : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o) w += n;
        }
        if (lane < nw) warp_sums[lane] = w;
    }
    __syncthreads();
    const unsigned long long before = warp > 0 ? warp_sums[warp - 1] : 0ull;
    __syncthreads();
    return v + before;
}

// Sum of each tile of kScanTile lengths.
__global__ void __launch_bounds__(kScanBlock) k_tile_sums(const uint32_t *__restrict__ len, long long n,
                                                         unsigned long long *__restrict__ partials) {
    __shared__ unsigned long long ws[32];
    const long long base = (long long)blockIdx.x * kScanTile + (long long)threadIdx.x * kScanItems;
    unsigned long long s = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; i++)
        if (base + i < n) s += len[base + i];
    const unsigned long long incl = block_inclusive_scan(s, ws);
    if (threadIdx.x == blockDim.x - 1) partials[blockIdx.x] = incl;
}

// Exclusive scan of the tile totals in place (one CTA); partials[ntiles] = total.
__global__ void __launch_bounds__(kScanBlock) k_scan_partials(unsigned long long *partials, long long ntiles) {
    __shared__ unsigned long long ws[32];
    __shared__ unsigned long long last;
    unsigned long long carry = 0;
    for (long long b = 0; b < ntiles; b += blockDim.x) {
        const long long i = b + threadIdx.x;
        const unsigned long long v = i < ntiles ? partials[i] : 0ull;
        const unsigned long long incl = block_inclusive_scan(v, ws);
        if (i < ntiles) partials[i] = carry + incl - v;
        if (threadIdx.x == blockDim.x - 1) last = incl;
        __syncthreads();
        carry += last;
        __syncthreads();
    }
    if (threadIdx.x == 0) partials[ntiles] = carry;
}

// Offsets of one tile plus the copy of its streams into the packed buffer.
__global__ void __launch_bounds__(kScanBlock) k_offsets_and_pack(
    const uint32_t *__restrict__ len, long long n, const unsigned long long *__restrict__ partials,
    long long ntiles, uint64_t *__restrict__ off, const uint8_t *__restrict__ stage,
    long long stage_bytes, uint8_t *__restrict__ packed, unsigned long long capacity,
    int32_t *status) {
    __shared__ unsigned long long ws[32];
    __shared__ unsigned long long offs[kScanTile];
    __shared__ uint32_t lens[kScanTile];
    const long long tile0 = (long long)blockIdx.x * kScanTile;
    const long long base = tile0 + (long long)threadIdx.x * kScanItems;
    uint32_t v[kScanItems];
    unsigned long long s = 0;
#pragma unroll
    for (int i = 0; i < kScanItems; i++) {
        v[i] = (base + i < n) ? len[base + i] : 0u;
        s += v[i];
    }
    const unsigned long long incl = block_inclusive_scan(s, ws);
    unsigned long long o = partials[blockIdx.x] + incl - s;
#pragma unroll
    for (int i = 0; i < kScanItems; i++) {
        const int li = threadIdx.x * kScanItems + i;
        offs[li] = o;
        lens[li] = v[i];
        if (base + i < n) off[base + i] = o;
        o += v[i];
    }
    const unsigned long long total = partials[ntiles];
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        off[n] = total;
        if (total > capacity && status) atomicOr(status, CG_FLAG_CAPACITY);
    }
    if (stage == nullptr) return;  // offsets only
    __syncthreads();
    // copy: one warp per stream, 4 bytes per lane per step from the aligned stage
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long nt = min((long long)kScanTile, n - tile0);
    for (long long li = warp; li < nt; li += blockDim.x >> 5) {
        const unsigned long long dst = offs[li];
        const uint32_t L = lens[li];
        const uint8_t *src = stage + (tile0 + li) * stage_bytes + kStagePrefix;
        for (uint32_t b = 4u * lane; b < L; b += 128u) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(src + b);
            const uint32_t nb = min(4u, L - b);
#pragma unroll
            for (uint32_t j = 0; j < 4; j++) {
                const unsigned long long p = dst + b + j;
                if (j < nb && p < capacity) packed[p] = (uint8_t)(w >> (8 * j));
            }
        }
    }
}

}  // namespace

cudaError_t launch_scan_and_pack(const uint32_t *len, uint64_t *off, const uint8_t *stage,
                                 uint8_t *packed, uint64_t capacity, unsigned long long *partials,
                                 const Dims &d, int32_t *status, cudaStream_t s) {
    const long long n = d.nstreams;
    const long long ntiles = scan_tiles(n);
    k_tile_sums<<<(unsigned)ntiles, kScanBlock, 0, s>>>(len, n, partials);
    k_scan_partials<<<1, kScanBlock, 0, s>>>(partials, ntiles);
    k_offsets_and_pack<<<(unsigned)ntiles, kScanBlock, 0, s>>>(len, n, partials, ntiles, off, stage,
                                                               d.stage_bytes, packed, capacity, status);
    return cudaGetLastError();
}

cudaError_t launch_offsets(const uint32_t *len, uint64_t *off, unsigned long long *partials, const Dims &d,
                           cudaStream_t s) {
    return launch_scan_and_pack(len, off, nullptr, nullptr, 0, partials, d, nullptr, s);
}

}  // namespace cg
