// records3.cu - format 3 side information: format 2's count records
// [CG §2.3(2)] without their zero bytes, and back. Per record a mode byte and
// a 32-bit presence mask of the other symbols with a nonzero count; the
// counts themselves, one byte each, back to back per slice, located by
// per-slice offsets (layout in include/cachegen.h). Small kernels next to the
// coders: a few bytes per record in and out.
#include "cg_internal.cuh"

namespace cg {
namespace {

constexpr int kB = 256;

// Exclusive block scan of one value per thread (kB threads); the block total
// comes back in `total`.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t &total) {
    __shared__ uint32_t warp_sums[kB / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kB / 32; w++) {
        before += w < warp ? warp_sums[w] : 0u;
        total += warp_sums[w];
    }
    __syncthreads();
    return before + incl - v;
}

// A tile of records (nb bytes at src, contiguous) into shared memory, 32-bit
// loads when src is 4-byte aligned.
__device__ __forceinline__ void load_tile(uint8_t *dst, const uint8_t *src, int nb) {
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        // 16-byte loads, several in flight per thread
#pragma unroll 4
        for (int i = threadIdx.x; i < nb / 16; i += kB)
            reinterpret_cast<uint4 *>(dst)[i] = __ldg(reinterpret_cast<const uint4 *>(src) + i);
        for (int i = (nb & ~15) + threadIdx.x; i < nb; i += kB) dst[i] = src[i];
    } else if ((reinterpret_cast<uintptr_t>(src) & 3) == 0) {
#pragma unroll 8
        for (int i = threadIdx.x; i < nb / 4; i += kB)
            reinterpret_cast<uint32_t *>(dst)[i] = __ldg(reinterpret_cast<const uint32_t *>(src) + i);
        for (int i = (nb & ~3) + threadIdx.x; i < nb; i += kB) dst[i] = src[i];
    } else {
#pragma unroll 8
        for (int i = threadIdx.x; i < nb; i += kB) dst[i] = src[i];
    }
}

// A record's byte 1 + i counts the i-th symbol other than the mode.
__device__ __forceinline__ int other_symbol(int i, int mode) { return i < mode ? i : i + 1; }

// Per slice: the number of nonzero count bytes in its records.
__global__ void __launch_bounds__(kB) k_v3_totals(const uint8_t *__restrict__ rec, Dims d, MaxTab mt,
                                                  unsigned long long *__restrict__ totals) {
    int k, kv, l;
    slice_coords(d, blockIdx.x, k, kv, l);
    const int A = 2 * mt.v[kv][l] + 1;
    const uint8_t *r = rec + record_slice_offset(d, mt, k, kv, l);
    const long long nb = (long long)d.C * A;
    uint32_t n = 0;
    // count the nonzero bytes, less those in a record's first byte (the mode)
    if ((reinterpret_cast<uintptr_t>(r) & 15) == 0) {
#pragma unroll 4
        for (long long i = threadIdx.x; i < nb / 16; i += kB) {
            const uint4 q = __ldg(reinterpret_cast<const uint4 *>(r) + i);
            // nonzero bytes: __vcmpne4 gives 0xFF per differing byte
            n += (uint32_t)(__popc(__vcmpne4(q.x, 0u)) + __popc(__vcmpne4(q.y, 0u)) + __popc(__vcmpne4(q.z, 0u)) +
                            __popc(__vcmpne4(q.w, 0u))) / 8u;
        }
        for (long long i = (nb & ~15LL) + threadIdx.x; i < nb; i += kB) n += r[i] != 0 ? 1u : 0u;
    } else {
#pragma unroll 8
        for (long long i = threadIdx.x; i < nb; i += kB) n += r[i] != 0 ? 1u : 0u;
    }
#pragma unroll 4
    for (int c = threadIdx.x; c < d.C; c += kB) n -= r[(long long)c * A] != 0 ? 1u : 0u;
    uint32_t total;
    block_excl_scan(n, total);
    if (threadIdx.x == 0) totals[blockIdx.x] = total;
}

// O[s] = exclusive scan of the slice totals, O[nslice] = the sum (one CTA).
__global__ void __launch_bounds__(kB) k_v3_offsets(const unsigned long long *__restrict__ totals, long long ns,
                                                   unsigned long long *__restrict__ O) {
    __shared__ unsigned long long warp_sums[kB / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long carry = 0;
    for (long long b = 0; b < ns; b += kB) {
        const long long i = b + threadIdx.x;
        const unsigned long long v = i < ns ? totals[i] : 0ull;
        unsigned long long incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        unsigned long long before = 0, sum = 0;
#pragma unroll
        for (int w = 0; w < kB / 32; w++) {
            before += w < warp ? warp_sums[w] : 0ull;
            sum += warp_sums[w];
        }
        if (i < ns) O[i] = carry + before + incl - v;
        carry += sum;
        __syncthreads();
    }
    if (threadIdx.x == 0) O[ns] = carry;
}

// Per slice: modes, presence masks and the nonzero counts at O[s].
__global__ void __launch_bounds__(kB) k_v3_pack(const uint8_t *__restrict__ rec, Dims d, MaxTab mt,
                                                uint8_t *__restrict__ side) {
    __shared__ __align__(16) uint8_t s_rec[kB * 32];  // a tile's records (A <= 32)
    int k, kv, l;
    slice_coords(d, blockIdx.x, k, kv, l);
    const int A = 2 * mt.v[kv][l] + 1;
    const uint8_t *r0 = rec + record_slice_offset(d, mt, k, kv, l);
    long long offM, offB, offV;
    v3_layout(d, offM, offB, offV);
    const long long s = blockIdx.x;
    uint8_t *V = side + offV + reinterpret_cast<const unsigned long long *>(side)[s];
    uint32_t run = 0;  // count bytes of the slice's earlier channels
    for (int c0 = 0; c0 < d.C; c0 += kB) {
        const int c = c0 + threadIdx.x;
        uint32_t bits = 0, n = 0;
        int mode = 0;
        load_tile(s_rec, r0 + (long long)c0 * A, min(kB, d.C - c0) * A);
        __syncthreads();
        const uint8_t *r = s_rec + threadIdx.x * A;
        if (c < d.C) {
            mode = r[0];
            for (int i = 0; i < A - 1; i++) bits |= (r[1 + i] != 0 ? 1u : 0u) << other_symbol(i, mode);
            n = (uint32_t)__popc(bits);
        }
        uint32_t total;
        const uint32_t at = run + block_excl_scan(n, total);
        if (c < d.C) {
            const long long g = s * d.C + c;
            side[offM + g] = (uint8_t)mode;
            reinterpret_cast<uint32_t *>(side + offB)[g] = bits;
            uint32_t j = at;
            for (uint32_t b = bits; b; b &= b - 1) {  // the set bits, in increasing symbol order
                const int t = __ffs(b) - 1;
                V[j++] = r[1 + (t < mode ? t : t - 1)];
            }
        }
        __syncthreads();  // the tile buffer is refilled next
        run += total;
    }
}

// Per slice: the format 2 records back from the side buffer, checking what
// the encoder guarantees; reads stay inside the buffer's nbytes. The slice's
// counts come into shared memory first (one coalesced pass, when they fit),
// each tile's masks are loaded a tile ahead, and each tile of records is
// assembled in shared memory and leaves in 32-bit stores (the records of
// consecutive channels are contiguous).
constexpr int kVStage = 16384;  // count bytes of a slice staged in shared memory

__global__ void __launch_bounds__(kB) k_v3_unpack(const uint8_t *__restrict__ side, unsigned long long nbytes,
                                                  Dims d, MaxTab mt, uint8_t *__restrict__ rec,
                                                  int32_t *status) {
    __shared__ __align__(16) uint8_t s_rec[kB * 32];  // a tile's records (A <= 32)
    __shared__ __align__(16) uint8_t s_v[kVStage];    // the slice's counts
    int k, kv, l;
    slice_coords(d, blockIdx.x, k, kv, l);
    const int A = 2 * mt.v[kv][l] + 1;
    uint8_t *r0 = rec + record_slice_offset(d, mt, k, kv, l);
    long long offM, offB, offV;
    v3_layout(d, offM, offB, offV);
    const long long s = blockIdx.x, ns = 2LL * d.L * d.nch;
    const unsigned long long *O = reinterpret_cast<const unsigned long long *>(side);
    const unsigned long long vbytes = nbytes - (unsigned long long)offV;  // nbytes >= offV (checked on the host)
    const unsigned long long vtotal = O[ns];
    unsigned long long beg = O[s], end = O[s + 1];
    bool bad = O[0] != 0 || vtotal > vbytes || beg > end || end > vtotal;
    if (bad) beg = end = 0;  // decode from empty counts
    const uint8_t *V = side + offV;
    const unsigned long long nv = end - beg;
    const bool staged = nv <= (unsigned long long)kVStage;
    if (staged) {
#pragma unroll 8
        for (unsigned long long i = threadIdx.x; i < nv; i += kB) s_v[i] = V[beg + i];
    }
    const uint8_t *M = side + offM + s * d.C;
    const uint32_t *Bm = reinterpret_cast<const uint32_t *>(side + offB) + s * d.C;
    int mode_n = threadIdx.x < d.C ? M[threadIdx.x] : 0;  // the next tile's mask, loaded ahead
    uint32_t bits_n = threadIdx.x < d.C ? Bm[threadIdx.x] : 0u;
    uint32_t run = 0;
    for (int c0 = 0; c0 < d.C; c0 += kB) {
        const int c = c0 + threadIdx.x;
        int mode = mode_n;
        uint32_t bits = bits_n;
        if (c + kB < d.C) {
            mode_n = M[c + kB];
            bits_n = Bm[c + kB];
        }
        if (c < d.C) {
            const uint32_t legal = (A < 32 ? (1u << A) - 1u : 0xFFFFFFFFu) & ~(mode < 32 ? 1u << mode : 0u);
            if (mode >= A || (bits & ~legal)) {
                bad = true;
                mode = mode < A ? mode : 0;
                bits &= legal;
            }
        } else {
            mode = 0;
            bits = 0;
        }
        for (int i = threadIdx.x; i < kB * 32 / 16; i += kB) reinterpret_cast<uint4 *>(s_rec)[i] = make_uint4(0, 0, 0, 0);
        uint32_t total;
        const uint32_t at = run + block_excl_scan((uint32_t)__popc(bits), total);  // within the slice (a barrier)
        if (c < d.C) {
            uint8_t *r = s_rec + threadIdx.x * A;
            r[0] = (uint8_t)mode;
            unsigned long long j = at;
            for (uint32_t b = bits; b; b &= b - 1) {  // the set bits, in increasing symbol order
                const int t = __ffs(b) - 1;
                uint8_t n = 0;
                if (j < nv) {
                    n = staged ? s_v[j] : V[beg + j];
                    bad |= n == 0;
                } else {
                    bad = true;
                }
                r[1 + (t < mode ? t : t - 1)] = n;
                j++;
            }
        }
        __syncthreads();
        // the tile's records out: [c0 * A, (c0 + nc) * A) of the slice
        const int nb = (min(kB, d.C - c0)) * A;
        uint8_t *dst = r0 + (long long)c0 * A;
        if ((reinterpret_cast<uintptr_t>(dst) & 3) == 0) {
            for (int i = threadIdx.x; i < nb / 4; i += kB)
                reinterpret_cast<uint32_t *>(dst)[i] = reinterpret_cast<const uint32_t *>(s_rec)[i];
            for (int i = (nb & ~3) + threadIdx.x; i < nb; i += kB) dst[i] = s_rec[i];
        } else {
            for (int i = threadIdx.x; i < nb; i += kB) dst[i] = s_rec[i];
        }
        __syncthreads();
        run += total;
    }
    if (run != nv) bad = true;
    if (bad && status) atomicOr(status, CG_FLAG_CORRUPT);
}

}  // namespace

cudaError_t launch_v3_pack(const uint8_t *rec, const Dims &d, const MaxTab &mt, uint8_t *side,
                           unsigned long long *totals, cudaStream_t s) {
    const long long ns = 2LL * d.L * d.nch;
    k_v3_totals<<<(unsigned)ns, kB, 0, s>>>(rec, d, mt, totals);
    k_v3_offsets<<<1, kB, 0, s>>>(totals, ns, reinterpret_cast<unsigned long long *>(side));
    k_v3_pack<<<(unsigned)ns, kB, 0, s>>>(rec, d, mt, side);
    return cudaGetLastError();
}

cudaError_t launch_v3_unpack(const uint8_t *side, unsigned long long nbytes, const Dims &d, const MaxTab &mt,
                             uint8_t *rec, int32_t *status, cudaStream_t s) {
    const long long ns = 2LL * d.L * d.nch;
    k_v3_unpack<<<(unsigned)ns, kB, 0, s>>>(side, nbytes, d, mt, rec, status);
    return cudaGetLastError();
}

}  // namespace cg
