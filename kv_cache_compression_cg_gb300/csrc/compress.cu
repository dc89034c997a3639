// compress.cu - the fused compress kernel: adaptive quantisation
// [CG §2.3(1)], per-channel CDF [CG §2.3(2)], range encoding [CG §1.2(3)] and
// packing of one (chunk, kv, layer) slice per CTA, straight from fp16.
//
// Used for chunks of up to 256 tokens, alphabets up to 64 and C % 8 == 0 with
// 16-byte aligned rows (other shapes take the quantise + slice-coder + scan
// kernels). One thread per token stream. Per CTA:
//   0. take a slice ticket (so every slice a CTA waits on below belongs to a
//      CTA that is already running); max1 of every token row (warp per row,
//      128-bit loads, max of the fp16 magnitude bits) and factor = MAX / max1
//      (0 for an all-zero row: every value then maps to MAX);
//   then per window of W channels:
//   1. load the [Tc_k x W] fp16 tile with 128-bit loads, quantise it on the
//      way into a shared symbol tile, and count each symbol with a shared
//      atomic add into a per-window [symbol][channel] table of 16-bit counters
//      (padded rows: the eight channels of one vector land in distinct banks);
//   2. four threads per channel normalise its counts into a CDF row (two
//      passes over their quarter of the alphabet, combined with shuffles),
//      written as packed (lo | f << 16) entries and as the uint16 CDF output;
//   3. every thread codes its token's W symbols;
//   after the last window:
//   4. a block scan of the stream lengths gives offsets inside the slice, a
//      decoupled look-back over the preceding slices' totals gives the slice's
//      offset in the packed buffer (spins are bounded; on timeout the
//      CG_FLAG_TIMEOUT bit is set and the CTA carries on), and the CTA copies
//      its streams from the staging area (L2-resident, just written) into
//      place, clipped at the capacity.
#include <cuda_fp16.h>

#include "cg_internal.cuh"
#include "coder.cuh"

namespace cg {
namespace {

constexpr int kNT = 256;  // threads = max tokens per chunk on this path
constexpr int kNW = kNT / 32;
constexpr uint32_t kTotal = 65536u;
constexpr unsigned long long kFlagAggregate = 1ull << 62;
constexpr unsigned long long kFlagPrefix = 2ull << 62;
constexpr unsigned long long kValueMask = (1ull << 62) - 1;
constexpr int kSpinLimit = 1 << 22;

struct FusedSmem {
    size_t tile, cnt, cdfw, ftab, fac, m1, scan, bytes;
    int cnt_stride;  // 32-bit words per counter row (one row per symbol)
};

template <int W>
__host__ __device__ inline FusedSmem fused_layout(int A) {
    FusedSmem s;
    s.cnt_stride = W / 2 + 1;
    size_t o = 0;
    s.tile = o;
    o += (size_t)kNT * (W + 4);
    o = (o + 15) & ~(size_t)15;
    s.cnt = o;  // [symbol][channel] uint16 counters, rows padded by one word
    o += (size_t)A * s.cnt_stride * 4;
    s.cdfw = o;  // [channel][A + 1] uint32
    o += (size_t)W * (A + 1) * 4;
    s.ftab = o;  // f(n), n = 0..kNT, uint16
    o += (size_t)(kNT + 1) * 2;
    o = (o + 3) & ~(size_t)3;
    s.fac = o;  // float per token
    o += (size_t)kNT * 4;
    s.m1 = o;  // max1 bits per token
    o += (size_t)kNT * 2;
    o = (o + 7) & ~(size_t)7;
    s.scan = o;  // kNW + 4 uint64 for the block scan and the slice base
    o += (size_t)(kNW + 4) * 8;
    s.bytes = (o + 15) & ~(size_t)15;
    return s;
}

// Quantise two halves packed in w to two symbols (specification Q); factor 0
// encodes an all-zero row. The unsigned min keeps non-finite input in range.
__device__ __forceinline__ uint32_t quant2(uint32_t w, float factor, float fmax, uint32_t qmax) {
    const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&w));
    const uint32_t q0 = min((uint32_t)__float2int_rn(__fadd_rn(__fmul_rn(x.x, factor), fmax)), qmax);
    const uint32_t q1 = min((uint32_t)__float2int_rn(__fadd_rn(__fmul_rn(x.y, factor), fmax)), qmax);
    return q0 | (q1 << 8);
}

// Count symbol q of channel c (in the window) in the [q][c] uint16 table.
__device__ __forceinline__ void count_symbol(uint32_t *cnt, int stride, uint32_t q, int c) {
    atomicAdd(cnt + q * stride + (c >> 1), 1u << (16 * (c & 1)));
}

__device__ __forceinline__ uint32_t count_of(const uint32_t *cnt, int stride, int s, int c) {
    return (cnt[s * stride + (c >> 1)] >> (16 * (c & 1))) & 0xFFFFu;
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__global__ void k_compress_init(unsigned long long *state, long long nslices) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i <= nslices;
         i += (long long)gridDim.x * blockDim.x)
        state[i] = 0ull;  // state[0] is the ticket counter, state[1 + s] slice s
}

template <int W>
__global__ void __launch_bounds__(kNT, 4) k_compress_fused(
    const uint16_t *__restrict__ kin, const uint16_t *__restrict__ vin, Dims d, MaxTab mt,
    uint16_t *__restrict__ max1_out, uint16_t *__restrict__ cdf_out, uint8_t *__restrict__ stage,
    uint32_t *__restrict__ len, uint64_t *__restrict__ off, uint8_t *__restrict__ packed,
    unsigned long long capacity, unsigned long long *state, int32_t *status) {
    constexpr int TS = W + 4;
    constexpr int VPR = W / 8;  // 8-half vectors per tile row
    constexpr int TPC = kNT / W;  // threads per channel in the CDF step
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_ticket;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_ticket = (int)atomicAdd(state, 1ull);
    __syncthreads();
    const int ticket = s_ticket;
    int k, kv, l;
    slice_coords(d, ticket, k, kv, l);
    const int A = d.A[kv];
    const int Tk = chunk_tokens(d, k);
    const int MAX = mt.v[kv][l];
    const float fmax = (float)MAX;
    const uint32_t qmax = 2u * (uint32_t)MAX;
    const FusedSmem lay = fused_layout<W>(A);
    const int cs = lay.cnt_stride;
    uint8_t *tile = smem + lay.tile;
    uint32_t *cnt = reinterpret_cast<uint32_t *>(smem + lay.cnt);
    uint32_t *cdfw = reinterpret_cast<uint32_t *>(smem + lay.cdfw);
    uint16_t *ftab = reinterpret_cast<uint16_t *>(smem + lay.ftab);
    float *fac = reinterpret_cast<float *>(smem + lay.fac);
    uint16_t *m1 = reinterpret_cast<uint16_t *>(smem + lay.m1);
    unsigned long long *scan = reinterpret_cast<unsigned long long *>(smem + lay.scan);

    const long long t0 = (long long)k * d.Tc;
    const uint16_t *x = (kv ? vin : kin) + (long long)l * d.layer_stride + t0 * d.C;
    const long long cdf_base = cdf_slice_offset(d, k, kv, l);
    const long long sid0 = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk;
    const long long sid = sid0 + tid;
    uint8_t *stream = stage_stream(stage, tid < Tk ? sid : sid0, d);

    // 0. max1 per token row, the per-row factor and the f(n) table
    const int nvec = d.C >> 3;
    bool nonfinite = false;
    for (int r = warp; r < Tk; r += kNW) {
        const uint4 *row = reinterpret_cast<const uint4 *>(x + (long long)r * d.C);
        unsigned m = 0;
        for (int v0 = lane; v0 < nvec; v0 += 128) {
            uint4 q[4];
#pragma unroll
            for (int u = 0; u < 4; u++)
                q[u] = (v0 + 32 * u < nvec) ? __ldg(row + v0 + 32 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int u = 0; u < 4; u++) {
                m = __vmaxu2(m, q[u].x & 0x7FFF7FFFu);
                m = __vmaxu2(m, q[u].y & 0x7FFF7FFFu);
                m = __vmaxu2(m, q[u].z & 0x7FFF7FFFu);
                m = __vmaxu2(m, q[u].w & 0x7FFF7FFFu);
            }
        }
        m = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
        if (lane == 0) {
            m1[r] = (uint16_t)m;
            max1_out[group_index(d, kv, l, t0 + r)] = (uint16_t)m;
            nonfinite |= (m >= 0x7C00u);
        }
    }
    for (int n = tid; n <= Tk; n += kNT)
        ftab[n] = (uint16_t)(1u + ((uint32_t)n * (kTotal - (uint32_t)A)) / (uint32_t)Tk);
    for (int i = tid; i < A * cs; i += kNT) cnt[i] = 0;
    __syncthreads();
    if (tid < Tk) {
        const unsigned mb = m1[tid];
        fac[tid] = mb ? __fdiv_rn(fmax, __half2float(__ushort_as_half((unsigned short)mb))) : 0.0f;
    }
    __syncthreads();

    Enc e;
    enc_init(e);
    for (int c0 = 0; c0 < d.C; c0 += W) {
        const int Wc = min(W, d.C - c0);  // a multiple of 8
        // 1. fp16 tile -> symbol tile, counting every symbol
        for (int i = tid; i < Tk * VPR; i += kNT) {
            const int r = i / VPR, j = i % VPR;
            if (8 * j < Wc) {
                const uint4 h = __ldg(reinterpret_cast<const uint4 *>(x + (long long)r * d.C + c0) + j);
                const float f = fac[r];
                const uint32_t s01 = quant2(h.x, f, fmax, qmax), s23 = quant2(h.y, f, fmax, qmax);
                const uint32_t s45 = quant2(h.z, f, fmax, qmax), s67 = quant2(h.w, f, fmax, qmax);
                uint32_t *dst = reinterpret_cast<uint32_t *>(tile + r * TS + 8 * j);
                dst[0] = s01 | (s23 << 16);
                dst[1] = s45 | (s67 << 16);
                const int cb = 8 * j;
                count_symbol(cnt, cs, s01 & 0xFF, cb);
                count_symbol(cnt, cs, s01 >> 8, cb + 1);
                count_symbol(cnt, cs, s23 & 0xFF, cb + 2);
                count_symbol(cnt, cs, s23 >> 8, cb + 3);
                count_symbol(cnt, cs, s45 & 0xFF, cb + 4);
                count_symbol(cnt, cs, s45 >> 8, cb + 5);
                count_symbol(cnt, cs, s67 & 0xFF, cb + 6);
                count_symbol(cnt, cs, s67 >> 8, cb + 7);
            }
        }
        __syncthreads();
        // 2. CDF rows: thread (channel c, part p) owns symbols p, p + TPC, ...
        {
            const int c = tid / TPC, p = tid % TPC;
            // a warp covers 32 / TPC channels and Wc is a multiple of 8, so a
            // warp is entirely inside or entirely outside the window
            if (c < Wc) {
                uint32_t sum = 0, key = 0;
                for (int s = p; s < A; s += TPC) {
                    const uint32_t n = count_of(cnt, cs, s, c);
                    sum += ftab[n];
                    key = max(key, (n << 8) | (255u - (uint32_t)s));  // largest n, then smallest s
                }
#pragma unroll
                for (int o = 1; o < TPC; o <<= 1) {
                    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
                    key = max(key, __shfl_xor_sync(0xFFFFFFFFu, key, o));
                }
                const uint32_t best = 255u - (key & 255u);
                const uint32_t extra = kTotal - sum;
                // cumulative walk over the symbols in order: each part walks the
                // whole row's prefix of its own symbols through shuffles
                uint32_t *row = cdfw + c * (A + 1);
                uint16_t *g = cdf_out + cdf_base + (long long)(c0 + c) * A;
                uint32_t lo = 0;
                for (int s0 = 0; s0 < A; s0 += TPC) {
                    const int s = s0 + p;
                    uint32_t f = 0;
                    if (s < A) f = (uint32_t)ftab[count_of(cnt, cs, s, c)] + ((uint32_t)s == best ? extra : 0u);
                    uint32_t incl = f;
#pragma unroll
                    for (int o = 1; o < TPC; o <<= 1) {
                        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o, TPC);
                        if (p >= o) incl += v;
                    }
                    if (s < A) {
                        const uint32_t mylo = lo + incl - f;
                        row[s] = mylo | (f << 16);
                        g[s] = (uint16_t)mylo;
                    }
                    lo += __shfl_sync(0xFFFFFFFFu, incl, TPC - 1, TPC);
                }
            }
        }
        __syncthreads();
        // the counters are free again: clear them for the next window
        for (int i = tid; i < A * cs; i += kNT) cnt[i] = 0;
        // 3. code my token's symbols of this window
        if (tid < Tk) {
            const uint8_t *my = tile + tid * TS;
            const uint32_t *row = cdfw;
            const int rs = A + 1;
            if (Wc == W) {
#pragma unroll 4
                for (int c = 0; c < W; c += 4) {
                    const uint32_t q4 = *reinterpret_cast<const uint32_t *>(my + c);
                    if (e.nbits >= 32) enc_flush_word(e, stream);
                    enc_symbol(e, row[q4 & 0xFF]);
                    enc_symbol(e, row[rs + ((q4 >> 8) & 0xFF)]);
                    if (e.nbits >= 32) enc_flush_word(e, stream);
                    enc_symbol(e, row[2 * rs + ((q4 >> 16) & 0xFF)]);
                    enc_symbol(e, row[3 * rs + (q4 >> 24)]);
                    row += 4 * rs;
                }
            } else {
                for (int c = 0; c < Wc; c++) {
                    if (e.nbits >= 32) enc_flush_word(e, stream);
                    enc_symbol(e, row[c * rs + my[c]]);
                }
            }
        }
        __syncthreads();
    }

    // 4. lengths, offsets inside the slice, the slice's place, the copy
    const uint32_t mylen = tid < Tk ? enc_finish(e, stream) : 0u;
    unsigned long long incl = mylen;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scan[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        unsigned long long run = 0;
        for (int w = 0; w < kNW; w++) {
            const unsigned long long t = scan[w];
            scan[w] = run;
            run += t;
        }
        // decoupled look-back over the previous slices (ticket order = stream order)
        unsigned long long *mine = state + 1 + ticket;
        unsigned long long base = 0;
        bool timed_out = false;
        if (ticket == 0) {
            st_release(mine, kFlagPrefix | run);
        } else {
            st_release(mine, kFlagAggregate | run);
            long long j = ticket - 1;
            while (j >= 0) {
                unsigned long long v = ld_acquire(state + 1 + j);
                int spins = 0;
                while ((v >> 62) == 0 && spins < kSpinLimit) {
                    __nanosleep(64);
                    v = ld_acquire(state + 1 + j);
                    spins++;
                }
                if ((v >> 62) == 0) {
                    timed_out = true;
                    break;
                }
                base += v & kValueMask;
                if ((v >> 62) == 2) break;
                j--;
            }
            st_release(mine, kFlagPrefix | ((base + run) & kValueMask));
        }
        scan[kNW] = base;
        scan[kNW + 1] = run;
        if (timed_out && status) atomicOr(status, CG_FLAG_TIMEOUT);
        if (ticket == 2LL * d.L * d.nch - 1) {
            off[d.nstreams] = base + run;
            if (base + run > capacity && status) atomicOr(status, CG_FLAG_CAPACITY);
        }
    }
    __syncthreads();
    const unsigned long long base = scan[kNW];
    const unsigned long long myoff = base + scan[warp] + incl - mylen;
    if (tid < Tk) {
        len[sid] = mylen;
        off[sid] = myoff;
    }
    // copy: every stream's (offset, length) goes through shared memory, then a
    // warp at a time copies one stream in consecutive 4-byte words
    unsigned long long *info = reinterpret_cast<unsigned long long *>(tile);  // reuse: 2 x kNT uint64
    if (tid < Tk) {
        info[2 * tid] = myoff;
        info[2 * tid + 1] = mylen;
    }
    __syncthreads();
    for (int t = warp; t < Tk; t += kNW) {
        const unsigned long long dst = info[2 * t];
        const uint32_t n = (uint32_t)info[2 * t + 1];
        const uint8_t *src = stage_stream(stage, sid0 + t, d);
        for (uint32_t b = 4u * lane; b < n; b += 128u) {
            const uint32_t wv = *reinterpret_cast<const uint32_t *>(src + b);
            const uint32_t nb = min(4u, n - b);
#pragma unroll
            for (uint32_t q = 0; q < 4; q++) {
                const unsigned long long pos = dst + b + q;
                if (q < nb && pos < capacity) packed[pos] = (uint8_t)(wv >> (8 * q));
            }
        }
    }
    if (nonfinite && status) atomicOr(status, CG_FLAG_NONFINITE);
}

template <int W>
cudaError_t launch_w(const uint16_t *k, const uint16_t *v, const Dims &d, const MaxTab &mt,
                     uint16_t *max1, uint16_t *cdf, uint8_t *stage, uint32_t *len, uint64_t *off,
                     uint8_t *packed, uint64_t capacity, unsigned long long *state, int32_t *status,
                     cudaStream_t s) {
    const size_t s0 = fused_layout<W>(d.A[0]).bytes, s1 = fused_layout<W>(d.A[1]).bytes;
    const size_t smem = s0 > s1 ? s0 : s1;
    cudaError_t err = cudaFuncSetAttribute(k_compress_fused<W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    const long long nslices = 2LL * d.L * d.nch;
    k_compress_init<<<(unsigned)((nslices + 1 + 255) / 256), 256, 0, s>>>(state, nslices);
    k_compress_fused<W><<<(unsigned)nslices, kNT, smem, s>>>(k, v, d, mt, max1, cdf, stage, len, off, packed,
                                                              capacity, state, status);
    return cudaGetLastError();
}

}  // namespace

bool compress_fused_applies(const Dims &d, const uint16_t *k, const uint16_t *v) {
    const int tmax = d.Tc < d.T ? d.Tc : d.T;
    const int A = d.A[0] > d.A[1] ? d.A[0] : d.A[1];
    const bool aligned = ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0 &&
                         d.layer_stride % 8 == 0;
    return tmax <= kNT && A <= 64 && d.C % 8 == 0 && aligned;
}

cudaError_t launch_compress_fused(const uint16_t *k, const uint16_t *v, const Dims &d, const MaxTab &mt,
                                  uint16_t *max1, uint16_t *cdf, uint8_t *stage, uint32_t *len,
                                  uint64_t *off, uint8_t *packed, uint64_t capacity,
                                  unsigned long long *state, int32_t *status, cudaStream_t s) {
    const int A = d.A[0] > d.A[1] ? d.A[0] : d.A[1];
    if (A <= 32)
        return launch_w<64>(k, v, d, mt, max1, cdf, stage, len, off, packed, capacity, state, status, s);
    return launch_w<32>(k, v, d, mt, max1, cdf, stage, len, off, packed, capacity, state, status, s);
}

}  // namespace cg
