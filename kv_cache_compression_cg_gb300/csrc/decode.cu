// decode.cu - range decoding [CG §2.4(1)] fused with dequantisation
// [CG §2.4(2)] for chunks of up to 256 tokens, specialised at compile time on
// the CDF width P (the alphabet rounded up to a power of two).
//
// CTA per (chunk, kv, layer) slice, thread per token stream. For each window of
// W channels the CTA stages the window's cumulative counts and frequencies in
// shared memory (entries at or past A hold 65536 / 0, so an unrolled binary
// search of log2(P) steps never leaves a valid stream's row); every thread
// decodes its W symbols into a shared symbol tile, four per 32-bit store; the
// tile then leaves as coalesced rows: dequantised binary32 through a per-layer
// table of (q - MAX) / MAX, or raw symbols.
#include <cuda_fp16.h>

#include "cg_internal.cuh"

namespace cg {
namespace {

constexpr uint32_t kM = 65536u;
constexpr int kThreads = 256;

template <int P>
struct DecodeCfg {
    static constexpr int W = P <= 32 ? 64 : (P == 64 ? 32 : 16);  // channels per window
    static constexpr int TS = W + 4;                                 // symbol tile row stride
};

struct Stream {
    uint32_t code, range;
    uint64_t bb;     // bit buffer, next bits at the top
    int nb;          // valid bits in bb
    uint32_t next;   // prefetched big-endian word at byte offset wa
    long long wa;    // offset of `next`; bytes [start, wa) are in bb or consumed
    long long start; // first byte of the stream
    long long end;   // one past the last readable byte of the stream
};

// Big-endian word at aligned byte offset wa, bytes outside [start, end) read
// as 0; taken only for a stream's first and last words.
__device__ __noinline__ uint32_t word_at_edge(const uint8_t *packed, long long wa, long long start,
                                              long long end) {
    uint32_t w = 0;
    for (int i = 0; i < 4; i++) {
        const long long p = wa + i;
        w = (w << 8) | ((p >= start && p < end) ? (uint32_t)__ldg(packed + p) : 0u);
    }
    return w;
}

__device__ __forceinline__ uint32_t word_at(const uint8_t *packed, long long wa, long long start,
                                            long long end) {
    if (wa >= start && wa + 4 <= end)
        return __byte_perm(__ldg(reinterpret_cast<const uint32_t *>(packed + wa)), 0, 0x0123);
    return word_at_edge(packed, wa, start, end);
}

// Next word of the stream (wa >= start always holds once initialised).
__device__ __forceinline__ uint32_t load_word(const uint8_t *packed, long long wa, long long start,
                                              long long end) {
    if (wa + 4 <= end)
        return __byte_perm(__ldg(reinterpret_cast<const uint32_t *>(packed + wa)), 0, 0x0123);
    return word_at_edge(packed, wa, start, end);
}

// Move the prefetched word into the bit buffer (needs nb <= 32) and start the
// load of the following one, which has the next ~32 bits of decoding to land.
__device__ __forceinline__ void refill(Stream &s, const uint8_t *packed) {
    s.bb |= (uint64_t)s.next << (32 - s.nb);
    s.nb += 32;
    s.wa += 4;
    s.next = load_word(packed, s.wa, s.start, s.end);
}

__device__ __forceinline__ void stream_init(Stream &s, const uint8_t *packed, long long start,
                                            long long end) {
    s.start = start;
    s.end = end;
    const int a = (int)(start & 3);
    const long long w0 = start - a;
    const uint32_t w = word_at(packed, w0, start, end);
    s.bb = ((uint64_t)w << 32) << (8 * a);
    s.nb = 32 - 8 * a;
    s.wa = w0 + 4;
    s.next = load_word(packed, s.wa, start, end);
    refill(s, packed);
    s.code = (uint32_t)(s.bb >> 32);
    s.bb <<= 32;
    s.nb -= 32;
    s.range = 0xFFFFFFFFu;
    refill(s, packed);
}

// One binary-search step over a uint16 CDF row at shared address `addr`:
// move addr forward by STEP entries when r * row[STEP] <= code.
template <int STEP>
__device__ __forceinline__ void search_step(uint32_t &addr, uint32_t r, uint32_t code) {
    asm("{\n\t.reg .pred p;\n\t.reg .u32 v;\n\t"
        "ld.shared.u16 v, [%0 + %3];\n\t"
        "mul.lo.u32 v, %1, v;\n\t"
        "setp.le.u32 p, v, %2;\n\t"
        "@p add.u32 %0, %0, %3;\n\t}"
        : "+r"(addr)
        : "r"(r), "r"(code), "n"(2 * STEP));
}

template <int STEP>
__device__ __forceinline__ void search_from(uint32_t &addr, uint32_t r, uint32_t code) {
    search_step<STEP>(addr, r, code);
    if constexpr (STEP > 1) search_from<STEP / 2>(addr, r, code);
}

// One symbol from the row of its channel: `cum` is the shared address of the
// uint16 cumulative row, its frequencies sit frq_off bytes further; needs
// nb >= 16. Entries at or past A hold cum = 65535: a valid stream's code never
// reaches them (its symbol's upper bound is at most 65535), and the clamp to
// A - 1 gives a corrupt stream the decoder rule's answer (largest s < A with
// r*cum[s] <= code).
template <int P>
__device__ __forceinline__ uint32_t decode_symbol(Stream &s, uint32_t cum, uint32_t frq_off,
                                                  uint32_t amax) {
    const uint32_t r = s.range >> 16;
    uint32_t addr = cum;
    search_from<P / 2>(addr, r, s.code);
    addr = min(addr, cum + 2 * amax);
    uint32_t lo, f;
    asm("ld.shared.u16 %0, [%1];" : "=r"(lo) : "r"(addr));
    asm("ld.shared.u16 %0, [%1];" : "=r"(f) : "r"(addr + frq_off));
    s.code -= r * lo;
    s.range = r * f;
    const uint32_t sh = __clz(s.range) & 24;
    s.code = __funnelshift_l((uint32_t)(s.bb >> 32), s.code, sh);
    s.bb <<= sh;
    s.nb -= (int)sh;
    s.range <<= sh;
    return (addr - cum) >> 1;
}

constexpr int kHelpers = 32;  // one helper warp per CTA

template <int P>
struct PipeSmem {
    static constexpr int W = DecodeCfg<P>::W;
    static constexpr int TS = DecodeCfg<P>::TS;
    static constexpr size_t cum = 0;                                   // [2][W][P] uint16
    static constexpr size_t frq = cum + 2ull * W * P * 2;              // [2][W][P] uint16
    static constexpr size_t tile = (frq + 2ull * W * P * 2 + 15) & ~15ull;  // [2][kThreads*TS]
    static constexpr size_t unit = tile + 2ull * kThreads * TS;        // float[256]
    static constexpr size_t m1 = unit + 256 * 4;                       // float[kThreads]
    static constexpr size_t bytes = m1 + kThreads * 4;
};

// Stage the CDF rows of window [c0, c0 + Wc) (helper warp): cum[c][j] =
// cdf[c][j] (65535 for j >= A), frq[c][j] = cdf[c][j+1] - cdf[c][j] (0 for
// j >= A, with cdf[c][A] = 65536). When A == P and the rows are 16-byte
// aligned the window's Wc*A entries are one contiguous run and move as
// independent 128-bit loads.
template <int P>
__device__ __forceinline__ void stage_rows(uint16_t *cum, uint16_t *frq, const uint16_t *src, int A,
                                           int Wc, int lane, bool vec) {
    if (vec && A == P) {
        const int nvec = Wc * P / 8;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        uint4 *d4 = reinterpret_cast<uint4 *>(cum);
        constexpr int U = 4;
        for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
            uint4 t[U];
#pragma unroll
            for (int u = 0; u < U; u++)
                if (v0 + 32 * u < nvec) t[u] = __ldg(s4 + v0 + 32 * u);
#pragma unroll
            for (int u = 0; u < U; u++)
                if (v0 + 32 * u < nvec) d4[v0 + 32 * u] = t[u];
        }
        __syncwarp();
        for (int i = lane; i < Wc * P; i += 32) {
            const int j = i % P;
            const uint32_t hi = j + 1 < P ? (uint32_t)cum[i + 1] : kM;
            frq[i] = (uint16_t)(hi - cum[i]);
        }
        return;
    }
    for (int i = lane; i < Wc * P; i += 32) {
        const int c = i / P, j = i % P;
        uint32_t lo = 65535u, f = 0;
        if (j < A) {
            lo = src[c * A + j];
            const uint32_t hi = j + 1 < A ? (uint32_t)src[c * A + j + 1] : kM;
            f = hi - lo;
        }
        cum[i] = (uint16_t)lo;
        frq[i] = (uint16_t)f;
    }
}

// Write the decoded window in `tile` out as rows: dequantised binary32
// (MODE 1) or symbols (MODE 0). Executed by `nthr` threads with index `id`.
template <int P, int MODE>
__device__ __forceinline__ void write_window(const uint8_t *tile, const float *unit, const float *m1s,
                                             const Dims &d, int kv, int l, long long t0, int Tk, int c0,
                                             int Wc, uint8_t *sym, float *out_k, float *out_v, int id,
                                             int nthr) {
    constexpr int W = DecodeCfg<P>::W;
    constexpr int TS = DecodeCfg<P>::TS;
    if (MODE == 0) {
        uint8_t *dst = sym + group_index(d, kv, l, t0) * d.C + c0;
        for (int i = id; i < Tk * W; i += nthr) {
            const int r = i / W, j = i % W;
            if (j < Wc) dst[(long long)r * d.C + j] = tile[r * TS + j];
        }
        return;
    }
    float *out = (kv ? out_v : out_k) + ((long long)l * d.T + t0) * d.C + c0;
    if (Wc == W && (d.C & 3) == 0) {
        constexpr int PR = W / 4;  // float4 per row
        for (int i = id; i < Tk * PR; i += nthr) {
            const int r = i / PR, j = i % PR;
            const uint32_t q4 = *reinterpret_cast<const uint32_t *>(tile + r * TS + 4 * j);
            const float m = m1s[r];
            float4 o;
            o.x = __fmul_rn(unit[q4 & 0xFF], m);
            o.y = __fmul_rn(unit[(q4 >> 8) & 0xFF], m);
            o.z = __fmul_rn(unit[(q4 >> 16) & 0xFF], m);
            o.w = __fmul_rn(unit[q4 >> 24], m);
            reinterpret_cast<float4 *>(out + (long long)r * d.C)[j] = o;
        }
    } else {
        for (int i = id; i < Tk * W; i += nthr) {
            const int r = i / W, j = i % W;
            if (j < Wc) out[(long long)r * d.C + j] = __fmul_rn(unit[tile[r * TS + j]], m1s[r]);
        }
    }
}

// CTA = kThreads decoder threads (one per token stream) + one helper warp.
// Iteration i: decoders decode window i with rows[i & 1] into tile[i & 1]
// while the helper stages rows[(i + 1) & 1] and writes out tile[(i + 1) & 1]
// (window i - 1); one barrier per window.
template <int P, int MODE>
__global__ void __launch_bounds__(kThreads + kHelpers, 4) k_decode_pipe(
    const uint8_t *__restrict__ packed, long long packed_bytes, const uint64_t *__restrict__ off,
    const uint32_t *__restrict__ len, const uint16_t *__restrict__ cdf,
    const uint16_t *__restrict__ max1, Dims d, MaxTab mt, uint8_t *__restrict__ sym,
    float *__restrict__ out_k, float *__restrict__ out_v, int32_t *status) {
    using L = PipeSmem<P>;
    constexpr int W = L::W;
    constexpr int TS = L::TS;
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t *cum = reinterpret_cast<uint16_t *>(smem + L::cum);
    uint16_t *frq = reinterpret_cast<uint16_t *>(smem + L::frq);
    uint8_t *tile = smem + L::tile;
    float *unit = reinterpret_cast<float *>(smem + L::unit);
    float *m1s = reinterpret_cast<float *>(smem + L::m1);

    int k, kv, l;
    slice_coords(d, blockIdx.x, k, kv, l);
    const int A = d.A[kv];
    const uint32_t amax = (uint32_t)A - 1;
    const int Tk = chunk_tokens(d, k);
    const int tid = threadIdx.x;
    const bool helper = tid >= kThreads;
    const int hl = tid - kThreads;  // helper lane
    const long long t0 = (long long)k * d.Tc;
    const long long cdf_base = cdf_slice_offset(d, k, kv, l);
    const long long sid = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk + tid;
    const int nwin = (d.C + W - 1) / W;

    if (MODE == 1 && !helper) {
        const int MAX = mt.v[kv][l];
        unit[tid] = __fdiv_rn((float)(tid - MAX), (float)MAX);
        if (tid < Tk) m1s[tid] = __half2float(__ushort_as_half(max1[group_index(d, kv, l, t0 + tid)]));
    }
    Stream s;
    bool corrupt = false;
    if (!helper && tid < Tk) {
        long long start = (long long)off[sid];
        long long end = start + (long long)len[sid];
        if (start > packed_bytes || end > packed_bytes) {
            corrupt = true;
            start = min(start, packed_bytes);
            end = min(end, packed_bytes);
        }
        stream_init(s, packed, start, end);
    }
    // 128-bit row loads need 16-byte aligned windows: cdf itself, and every
    // slice offset a multiple of 8 entries (both alphabets multiples of 8)
    const bool vec = ((reinterpret_cast<uintptr_t>(cdf) & 15) == 0) && (d.A[0] % 8 == 0) &&
                     (d.A[1] % 8 == 0);
    if (helper) stage_rows<P>(cum, frq, cdf + cdf_base, A, min(W, d.C), hl, vec);
    __syncthreads();

    for (int i = 0; i < nwin; i++) {
        const int b = i & 1;
        const int c0 = i * W;
        const int Wc = min(W, d.C - c0);
        if (!helper) {
            if (tid < Tk) {
                // shared addresses of this buffer's rows; frequencies follow at a fixed offset
                const uint32_t cb = (uint32_t)__cvta_generic_to_shared(cum + b * W * P);
                const uint32_t fo = (uint32_t)(L::frq - L::cum);
                uint8_t *my = tile + b * kThreads * TS + tid * TS;
                if (Wc == W) {
#pragma unroll 4
                    for (int c = 0; c < W; c += 4) {
                        const uint32_t rc = cb + 2 * P * c;
                        if (s.nb < 32) refill(s, packed);
                        const uint32_t q0 = decode_symbol<P>(s, rc, fo, amax);
                        const uint32_t q1 = decode_symbol<P>(s, rc + 2 * P, fo, amax);
                        if (s.nb < 32) refill(s, packed);
                        const uint32_t q2 = decode_symbol<P>(s, rc + 4 * P, fo, amax);
                        const uint32_t q3 = decode_symbol<P>(s, rc + 6 * P, fo, amax);
                        *reinterpret_cast<uint32_t *>(my + c) = q0 | (q1 << 8) | (q2 << 16) | (q3 << 24);
                    }
                } else {
                    for (int c = 0; c < Wc; c++) {
                        if (s.nb < 32) refill(s, packed);
                        my[c] = (uint8_t)decode_symbol<P>(s, cb + 2 * P * c, fo, amax);
                    }
                }
            }
        } else {
            if (i + 1 < nwin)
                stage_rows<P>(cum + (b ^ 1) * W * P, frq + (b ^ 1) * W * P,
                              cdf + cdf_base + (long long)(c0 + W) * A, A, min(W, d.C - c0 - W), hl, vec);
            if (i >= 1)
                write_window<P, MODE>(tile + (b ^ 1) * kThreads * TS, unit, m1s, d, kv, l, t0, Tk, c0 - W, W,
                                      sym, out_k, out_v, hl, kHelpers);
        }
        __syncthreads();
    }
    // the last window, written by the whole CTA
    {
        const int i = nwin - 1;
        write_window<P, MODE>(tile + (i & 1) * kThreads * TS, unit, m1s, d, kv, l, t0, Tk, i * W,
                              min(W, d.C - i * W), sym, out_k, out_v, tid, kThreads + kHelpers);
    }
    if (!helper && tid < Tk) {
        const long long consumed = (s.wa - s.start) - s.nb / 8;
        if ((corrupt || consumed != (long long)len[sid] + 3) && status) atomicOr(status, CG_FLAG_CORRUPT);
    }
}

template <int P>
cudaError_t launch_p(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                     const uint32_t *len, const uint16_t *cdf, const uint16_t *max1, const Dims &d,
                     const MaxTab &mt, int mode, uint8_t *sym, float *out_k, float *out_v,
                     int32_t *status, cudaStream_t s) {
    const unsigned nslices = (unsigned)(2LL * d.L * d.nch);
    const int smem = (int)PipeSmem<P>::bytes;
    cudaError_t err;
    if (mode == 1) {
        err = cudaFuncSetAttribute(k_decode_pipe<P, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        k_decode_pipe<P, 1><<<nslices, kThreads + kHelpers, smem, s>>>(
            packed, (long long)packed_bytes, off, len, cdf, max1, d, mt, sym, out_k, out_v, status);
    } else {
        err = cudaFuncSetAttribute(k_decode_pipe<P, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        k_decode_pipe<P, 0><<<nslices, kThreads + kHelpers, smem, s>>>(
            packed, (long long)packed_bytes, off, len, cdf, max1, d, mt, sym, out_k, out_v, status);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                          const uint32_t *len, const uint16_t *cdf, const uint16_t *max1,
                          const Dims &d, const MaxTab &mt, int mode, uint8_t *sym, float *out_k,
                          float *out_v, int32_t *status, cudaStream_t s) {
    const int tmax = d.Tc < d.T ? d.Tc : d.T;
    const int A = d.A[0] > d.A[1] ? d.A[0] : d.A[1];
    if (tmax > kThreads)
        return launch_decode_generic(packed, packed_bytes, off, len, cdf, max1, d, mt, mode, sym, out_k,
                                     out_v, status, s);
    if (A <= 8) return launch_p<8>(packed, packed_bytes, off, len, cdf, max1, d, mt, mode, sym, out_k, out_v, status, s);
    if (A <= 16) return launch_p<16>(packed, packed_bytes, off, len, cdf, max1, d, mt, mode, sym, out_k, out_v, status, s);
    if (A <= 32) return launch_p<32>(packed, packed_bytes, off, len, cdf, max1, d, mt, mode, sym, out_k, out_v, status, s);
    if (A <= 64) return launch_p<64>(packed, packed_bytes, off, len, cdf, max1, d, mt, mode, sym, out_k, out_v, status, s);
    if (A <= 128) return launch_p<128>(packed, packed_bytes, off, len, cdf, max1, d, mt, mode, sym, out_k, out_v, status, s);
    return launch_p<256>(packed, packed_bytes, off, len, cdf, max1, d, mt, mode, sym, out_k, out_v, status, s);
}

}  // namespace cg
