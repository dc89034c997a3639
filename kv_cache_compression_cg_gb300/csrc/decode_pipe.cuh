// decode_pipe.cuh - range decoding [CG §2.4(1)] fused with dequantisation
// [CG §2.4(2)] for chunks of up to 256 tokens: the kernel template, over the
// CDF width P (the alphabet rounded up to a power of two), the output type,
// the side-information format and the token-locality delta [CG §1.2(1)].
// Translation units that launch an instantiation include it (each gets its
// own copy, in an anonymous namespace).
//
// CTA per (chunk, kv, layer) slice: 256 decoder threads (one per token stream)
// and one helper warp. While the decoders work on window i the helper stages
// window i + 1's cumulative counts and frequencies in shared memory (entries at
// or past A hold 65535 / 0, so an unrolled binary search of log2(P) steps never
// leaves a row). Every decoder thread decodes its W symbols into its row of a
// shared tile, four per 32-bit store; then each warp writes its own 32 rows out
// as coalesced row segments, dequantised through a per-layer table of
// (q - MAX) / MAX. One barrier per window (for the row buffers); the tile
// rows are warp-private, except with the delta, where a row's anchor may
// belong to another warp and the decoder threads meet at a second barrier
// before the writes. Launches of at most one slice per SM take k_decode_lm
// further down instead (decoding threads fed by support threads, and a slice
// split over two SMs where the launch leaves room).
//
// Stream state is 32-bit: code, range, a 64-bit bit buffer held as two words,
// and a prefetched word whose load has the next ~32 coded bits to land. Bytes
// past a stream's end read as zero; the masked load runs only for a stream's
// last words.
#pragma once

#include <cuda_fp16.h>

#include "cg_internal.cuh"

namespace cg {
namespace {

constexpr uint32_t kM = 65536u;
constexpr int kThreads = 256;
constexpr int kHelpers = 32;  // one helper warp per CTA

template <int P>
struct DecodeCfg {
    static constexpr int W = P <= 32 ? 64 : (P == 64 ? 32 : 16);  // channels per window
    static constexpr int TS = W + 4;                                 // symbol tile row stride
    // tile bytes hold 4s (a byte offset into the dequantisation table) while
    // that fits a byte, else s
    static constexpr int SYM_SHIFT = P <= 64 ? 2 : 0;
};

struct Stream {
    uint32_t code, range;
    uint32_t bhi, blo;    // bit buffer, next bits at the top of bhi
    int nb;               // valid bits in (bhi, blo)
    uint32_t raw;         // the loaded next word, as in memory (not yet byte-swapped or masked)
    int rem;              // stream bytes from raw's word onwards (<= 0 once past the end)
    const uint32_t *wp;   // raw's word; stays on the stream's last word once rem <= 4
};

// Bytes [0, n) of the 4 at p in memory order (the others read as zero); for a
// stream's first word and, in warps holding a stream that ends in the
// buffer's last partial word, for every word.
__device__ __noinline__ uint32_t bytes_masked(const uint8_t *p, int n) {
    uint32_t w = 0;
    for (int i = 0; i < 4; i++)
        if (i < n) w |= (uint32_t)__ldg(p + i) << (8 * i);
    return w;
}

// Append the prefetched word below the nb valid bits when nb < 32, then load
// the following word (TAIL: byte by byte, within the stream only). The
// appended word is raw byte-swapped with the bytes past the stream's end
// cleared; the loaded word is first used by the next refill, so its latency
// hides behind about 32 decoded bits. Past the end the load repeats the
// stream's last word, so it never leaves the stream's words.
template <bool TAIL>
__device__ __forceinline__ void refill(Stream &s) {
    if (!TAIL) {
        if (s.nb < 32) {
            uint32_t v = __byte_perm(s.raw, 0, 0x0123);
            if (s.rem < 4) {  // the stream ends inside (or before) this word
                const int t = max(32 - 8 * s.rem, 0);  // bits past the stream's end
                v &= t >= 32 ? 0u : (0xFFFFFFFFu << t);
            }
            s.bhi |= v >> s.nb;
            s.blo |= __funnelshift_r(0u, v, (uint32_t)s.nb);  // v << (32 - nb), 0 for nb = 0
            s.nb += 32;
            if (s.rem > 4) s.wp++;
            s.rem -= 4;
            s.raw = __ldg(s.wp);
        }
    } else if (s.nb < 32) {
        uint32_t v = __byte_perm(s.raw, 0, 0x0123);
        v = s.rem >= 4 ? v : (s.rem <= 0 ? 0u : v & (0xFFFFFFFFu << (32 - 8 * s.rem)));
        s.bhi |= v >> s.nb;
        s.blo |= s.nb ? v << (32 - s.nb) : 0u;
        s.nb += 32;
        if (s.rem > 4) s.wp++;
        s.rem -= 4;
        s.raw = s.rem > 0 ? bytes_masked(reinterpret_cast<const uint8_t *>(s.wp), s.rem) : 0u;
    }
}

// refill<false> without a branch, for the latency-mode decoder, where each
// stream's dependent chain sets the time: the append is a select, and the next
// word's load runs every time (at the same address when nothing was appended,
// so it stays inside the stream's words). The throughput decoder keeps the
// branch (there every unconditional instruction costs issue slots).
__device__ __forceinline__ void refill_sel(Stream &s) {
    const bool need = s.nb < 32;
    uint32_t v = __byte_perm(s.raw, 0, 0x0123);
    const int t = max(32 - 8 * s.rem, 0);  // bits past the stream's end
    v &= s.rem >= 4 ? 0xFFFFFFFFu : (t >= 32 ? 0u : (0xFFFFFFFFu << t));
    v = need ? v : 0u;
    const uint32_t nbs = need ? (uint32_t)s.nb : 0u;
    s.bhi |= v >> nbs;
    s.blo |= __funnelshift_r(0u, v, nbs);  // v << (32 - nb), 0 for nb = 0
    s.nb += need ? 32 : 0;
    s.wp += (need && s.rem > 4) ? 1 : 0;
    s.rem -= need ? 4 : 0;
    s.raw = __ldg(s.wp);
}

// Stream over bytes [start, end) of the packed buffer (4-byte aligned); the
// first words come byte by byte.
__device__ __forceinline__ void stream_init(Stream &s, const uint8_t *packed, long long start, long long end) {
    const int a = (int)(start & 3);
    const long long w0 = start - a;
    // first word: bytes [a, min(4, end - w0)) belong to the stream; the bytes
    // before `a` leave with the shift
    const int n0 = (int)min(4LL, end - w0);
    s.bhi = __byte_perm(bytes_masked(packed + w0, n0), 0, 0x0123) << (8 * a);
    s.blo = 0;
    s.nb = 32 - 8 * a;
    s.rem = (int)(end - (w0 + 4));
    s.wp = reinterpret_cast<const uint32_t *>(packed + w0) + (s.rem > 0 ? 1 : 0);
    s.raw = s.rem > 0 ? bytes_masked(packed + w0 + 4, s.rem) : 0u;
    if (a == 0) {  // the first word alone fills code
        s.code = s.bhi;
        s.bhi = 0;
        s.nb = 0;
    } else {
        refill<true>(s);
        s.code = s.bhi;
        s.bhi = s.blo;
        s.blo = 0;
        s.nb -= 32;
    }
    s.range = 0xFFFFFFFFu;
    refill<true>(s);
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

// The same search over SPAN entries four ways per level: the entries at
// SPAN / 4, SPAN / 2 and 3 SPAN / 4 are loaded and compared at once, which
// halves the dependent loads of the search (a shorter chain per symbol, for
// more instructions: the decoder of launches whose time is set by that chain).
template <int SPAN>
__device__ __forceinline__ void search4(uint32_t &addr, uint32_t r, uint32_t code) {
    if constexpr (SPAN >= 4) {
        constexpr int Q = SPAN / 4;
        uint32_t c1, c2, c3;
        asm("ld.shared.u16 %0, [%1 + %2];" : "=r"(c1) : "r"(addr), "n"(2 * Q));
        asm("ld.shared.u16 %0, [%1 + %2];" : "=r"(c2) : "r"(addr), "n"(4 * Q));
        asm("ld.shared.u16 %0, [%1 + %2];" : "=r"(c3) : "r"(addr), "n"(6 * Q));
        const uint32_t n = (r * c1 <= code ? 1u : 0u) + (r * c2 <= code ? 1u : 0u) + (r * c3 <= code ? 1u : 0u);
        addr += 2u * Q * n;
        search4<Q>(addr, r, code);
    } else if constexpr (SPAN == 2) {
        search_step<1>(addr, r, code);
    }
}

// One symbol from the row of its channel: `cum` is the shared address of the
// uint16 cumulative row, its frequencies sit frq_off bytes further; needs
// nb >= 16. Searches the first PS entries of the row (PS >= A). Returns the
// entry's byte offset in the row (2s). Entries at or
// past A hold cum = 65535: a valid stream's code never passes symbol A - 1's
// upper bound, and with CLAMP (A < P) the clamp to A - 1 gives both a valid
// stream whose code reaches r * 65535 and a corrupt stream the decoder rule's
// answer (largest s < A with r*cum[s] <= code). With A == P no entry is
// padding and the search cannot pass A - 1.
template <int PS, bool CLAMP, bool WIDE = false>
__device__ __forceinline__ uint32_t decode_symbol(Stream &s, uint32_t cum, uint32_t frq_off, uint32_t amax2) {
    const uint32_t r = s.range >> 16;
    uint32_t addr = cum;
    if (WIDE)
        search4<PS>(addr, r, s.code);
    else
        search_from<PS / 2>(addr, r, s.code);
    if (CLAMP) addr = min(addr, cum + amax2);
    uint32_t lo, f;
    asm("ld.shared.u16 %0, [%1];" : "=r"(lo) : "r"(addr));
    asm("ld.shared.u16 %0, [%1];" : "=r"(f) : "r"(addr + frq_off));
    s.code -= r * lo;
    s.range = r * f;
    // bits to shift out, 0, 8 or 16 (range >= 2^8 here): by compares on the
    // latency path (no count-leading-zeros in the chain), else by clz
    const uint32_t sh = WIDE ? (s.range < 0x10000u ? 16u : (s.range < 0x1000000u ? 8u : 0u)) : (__clz(s.range) & 24);
    s.code = __funnelshift_l(s.bhi, s.code, sh);
    s.bhi = __funnelshift_l(s.blo, s.bhi, sh);
    s.blo <<= sh;
    s.nb -= (int)sh;
    s.range <<= sh;
    return addr - cum;
}

template <int P>
struct PipeSmem {
    static constexpr int W = DecodeCfg<P>::W;
    static constexpr int TS = DecodeCfg<P>::TS;
    static constexpr size_t cum = 0;                                        // [2][W][P] uint16
    static constexpr size_t frq = cum + 2ull * W * P * 2;                   // [2][W][P] uint16
    static constexpr size_t tile = (frq + 2ull * W * P * 2 + 15) & ~15ull;  // [kThreads*TS]
    static constexpr size_t m1 = tile + 1ull * kThreads * TS;               // float[kThreads]
    static constexpr size_t recs = m1 + kThreads * 4;                       // format 2: [2][W*P] records
    static constexpr size_t bytes = recs + 2ull * W * P;
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

// Format 2, step 1 (helper warp): the count records of one window (nb
// contiguous bytes) into shared memory with coalesced loads.
__device__ __forceinline__ void copy_records(uint8_t *srec, const uint8_t *recw, int nb, int lane) {
    if ((reinterpret_cast<uintptr_t>(recw) & 3) == 0) {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(recw);
        uint32_t *sw = reinterpret_cast<uint32_t *>(srec);
        for (int i = lane; i < nb / 4; i += 32) sw[i] = __ldg(w + i);
        for (int i = (nb & ~3) + lane; i < nb; i += 32) srec[i] = __ldg(recw + i);
    } else {
        for (int i = lane; i < nb; i += 32) srec[i] = __ldg(recw + i);
    }
}

// Format 2, step 2 (the 256 decoder threads): the window's CDF rows rebuilt
// from its records in shared memory. TPC = 256 / W threads share a channel
// (four for P <= 32, eight for P = 64, sixteen for wider rows), each owning
// P / TPC consecutive symbols: counts -> f(n) through the slice's table,
// TPC-lane sums of the counts, a TPC-lane scan of f, the remainder to the
// record's mode (which shifts the running sum of the symbols after it);
// entries at or past A hold 65535 / 0. A record whose mode byte is outside
// the alphabet or whose counts exceed Tk is corrupt: its channel gets every
// token on the mode (symbol 0 when the mode byte is invalid) and the function
// returns true. Channels at or past Wc (a partial last window) are built from
// unused bytes into rows no window reads, and not checked.
template <int P>
__device__ __forceinline__ bool build_rows_v2(uint16_t *cum, uint16_t *frq, const uint8_t *srec, int A, uint32_t Tk,
                                              int W, int Wc, int t, const uint16_t *ftab) {
    constexpr int TPC = kThreads / DecodeCfg<P>::W;  // threads per channel
    constexpr int SP = P / TPC;                       // symbols per thread
    const int c = t / TPC, p = t % TPC;
    if (c >= W) return false;  // whole TPC-lane groups
    const int j0 = p * SP;
    const uint8_t *r = srec + c * A;
    int mode = r[0];
    auto count_at = [&](int j) -> uint32_t {  // stored count of symbol j != mode
        return (j < A && j != mode) ? (uint32_t)r[j < mode ? j + 1 : j] : 0u;
    };
    if constexpr (SP <= 8) {
        // counts and frequencies in registers; entries leave two per 32-bit store
        uint32_t n[SP], fv[SP];
        uint32_t others = 0;
#pragma unroll
        for (int jj = 0; jj < SP; jj++) {
            n[jj] = count_at(j0 + jj);
            others += n[jj];
        }
#pragma unroll
        for (int o = 1; o < TPC; o <<= 1) others += __shfl_xor_sync(0xFFFFFFFFu, others, o);
        const bool ok = mode < A && others <= Tk;
        if (!ok) mode = mode < A ? mode : 0;
        const uint32_t nmode = ok ? Tk - others : Tk;
        uint32_t fl = 0;  // this thread's sum of f (without the remainder)
#pragma unroll
        for (int jj = 0; jj < SP; jj++) {
            const int j = j0 + jj;
            fv[jj] = j < A ? (uint32_t)ftab[j == mode ? nmode : (ok ? n[jj] : 0u)] : 0u;
            fl += fv[jj];
        }
        uint32_t incl = fl;
#pragma unroll
        for (int o = 1; o < TPC; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o, TPC);
            if (p >= o) incl += v;
        }
        const uint32_t rem = kM - __shfl_sync(0xFFFFFFFFu, incl, TPC - 1, TPC);
        uint32_t acc = incl - fl;
        uint32_t *cr = reinterpret_cast<uint32_t *>(cum + c * P + j0);  // j0 and SP even: 4-byte aligned
        uint32_t *fr = reinterpret_cast<uint32_t *>(frq + c * P + j0);
#pragma unroll
        for (int jj = 0; jj < SP; jj += 2) {
            uint32_t cv[2], fw[2];
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const int j = j0 + jj + h;
                cv[h] = j < A ? acc + (j > mode ? rem : 0u) : 65535u;
                fw[h] = j < A ? fv[jj + h] + (j == mode ? rem : 0u) : 0u;
                acc += fv[jj + h];
            }
            cr[jj / 2] = (cv[0] & 0xFFFFu) | (cv[1] << 16);
            fr[jj / 2] = (fw[0] & 0xFFFFu) | (fw[1] << 16);
        }
        return !ok && c < Wc;
    } else {
        uint32_t others = 0;
#pragma unroll 1
        for (int jj = 0; jj < SP; jj++) others += count_at(j0 + jj);
#pragma unroll
        for (int o = 1; o < TPC; o <<= 1) others += __shfl_xor_sync(0xFFFFFFFFu, others, o);
        const bool ok = mode < A && others <= Tk;
        if (!ok) mode = mode < A ? mode : 0;
        const uint32_t nmode = ok ? Tk - others : Tk;
        auto f_at = [&](int jj) -> uint32_t {
            const int j = j0 + jj;
            if (j >= A) return 0u;
            return ftab[j == mode ? nmode : (ok ? count_at(j) : 0u)];
        };
        uint32_t fl = 0;
#pragma unroll 1
        for (int jj = 0; jj < SP; jj++) fl += f_at(jj);
        uint32_t incl = fl;
#pragma unroll
        for (int o = 1; o < TPC; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o, TPC);
            if (p >= o) incl += v;
        }
        const uint32_t rem = kM - __shfl_sync(0xFFFFFFFFu, incl, TPC - 1, TPC);
        uint32_t acc = incl - fl;
        uint16_t *cr = cum + c * P;
        uint16_t *fr = frq + c * P;
#pragma unroll 1
        for (int jj = 0; jj < SP; jj++) {
            const int j = j0 + jj;
            const uint32_t f = f_at(jj);
            if (j < A) {
                cr[j] = (uint16_t)(acc + (j > mode ? rem : 0u));
                fr[j] = (uint16_t)(f + (j == mode ? rem : 0u));
            } else {
                cr[j] = 65535u;
                fr[j] = 0;
            }
            acc += f;
        }
        return !ok && c < Wc;
    }
}

__device__ __forceinline__ uint32_t lds_u32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

// Write the decoded window in `tile` out as rows of the dequantised values
// unit[s] * max1 (unit[s] = (s - MAX) / MAX), binary32 (MODE 1) or rounded to
// nearest-even binary16 (MODE 2), into [L][T][C] with layers `ols` elements
// apart. NTHR threads with index `id` share the work. With 4s in the tile
// bytes and the table 256-byte aligned, one byte permute makes each entry's
// shared address (table base with the low byte replaced). `vec` says the
// output rows allow 16-byte (binary32) or 8-byte (binary16) stores.
template <int P, int MODE, int NTHR>
__device__ __forceinline__ void write_window(const uint8_t *tile, const float *unit, const float *m1s,
                                             const Dims &d, int kv, int l, long long t0, int Tk, int c0, int Wc,
                                             void *out_k, void *out_v, long long ols, bool vec, int id) {
    constexpr int W = DecodeCfg<P>::W;
    constexpr int TS = DecodeCfg<P>::TS;
    constexpr int SH = DecodeCfg<P>::SYM_SHIFT;
    constexpr int ES = MODE == 2 ? 2 : 4;  // output element bytes
    char *out = static_cast<char *>(kv ? out_v : out_k) + ((long long)l * ols + t0 * d.C + c0) * ES;
    if (SH == 2 && Wc == W && vec && NTHR % (W / 4) == 0) {
        constexpr int PR = W / 4;        // four-value groups per row
        constexpr int RPI = NTHR / PR;   // rows per pass
        const int j = id % PR;
        int r = id / PR;
        const uint32_t us = (uint32_t)__cvta_generic_to_shared(unit);
        uint32_t ts = (uint32_t)__cvta_generic_to_shared(tile) + r * TS + 4 * j;
        uint32_t ms = (uint32_t)__cvta_generic_to_shared(m1s) + 4 * r;
        char *o = out + ((long long)r * d.C + 4 * j) * ES;
        const long long ostep = (long long)RPI * d.C * ES;
#pragma unroll 1
        for (; r < Tk; r += RPI, ts += RPI * TS, ms += 4 * RPI, o += ostep) {
            const uint32_t q4 = lds_u32(ts) & 0xFCFCFCFCu;  // 4s: keeps every table load aligned
            const float m = lds_f32(ms);
            const float u0 = lds_f32(__byte_perm(q4, us, 0x7650));
            const float u1 = lds_f32(__byte_perm(q4, us, 0x7651));
            const float u2 = lds_f32(__byte_perm(q4, us, 0x7652));
            const float u3 = lds_f32(__byte_perm(q4, us, 0x7653));
            const float x0 = __fmul_rn(u0, m), x1 = __fmul_rn(u1, m), x2 = __fmul_rn(u2, m), x3 = __fmul_rn(u3, m);
            if (MODE == 2) {
                const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
                *reinterpret_cast<uint2 *>(o) = make_uint2(*reinterpret_cast<const uint32_t *>(&h01),
                                                           *reinterpret_cast<const uint32_t *>(&h23));
            } else {
                *reinterpret_cast<float4 *>(o) = make_float4(x0, x1, x2, x3);
            }
        }
    } else {
        for (int i = id; i < Tk * W; i += NTHR) {
            const int r = i / W, j = i % W;
            if (j < Wc) {
                const float x = __fmul_rn(unit[tile[r * TS + j] >> SH], m1s[r]);
                char *e = out + ((long long)r * d.C + j) * ES;
                if (MODE == 2)
                    *reinterpret_cast<__half *>(e) = __float2half_rn(x);
                else
                    *reinterpret_cast<float *>(e) = x;
            }
        }
    }
}

// The delta's writer [CG §1.2(1)]: x^ = a^ + D(q), a^ = D(q_a) of the row's
// anchor (in any warp's rows, hence the barrier before it); an anchor row
// takes itself as its anchor with max1 0 (a^ = +-0 of D's own sign, so the sum
// is D(q) exactly). Warp `rbase / 32` writes its rows [rbase, rbase + rows).
template <int P, int MODE>
__device__ __forceinline__ void write_window_delta(const uint8_t *tile, const float *unit, const float *m1s,
                                                   const float *m1a, const uint8_t *anchor, const Dims &d, int kv,
                                                   int l, long long t0, int rbase, int rows, int c0, int Wc,
                                                   void *out_k, void *out_v, long long ols, bool vec, int lane) {
    constexpr int W = DecodeCfg<P>::W;
    constexpr int TS = DecodeCfg<P>::TS;
    constexpr int SH = DecodeCfg<P>::SYM_SHIFT;
    constexpr int ES = MODE == 2 ? 2 : 4;
    char *out = static_cast<char *>(kv ? out_v : out_k) + ((long long)l * ols + (t0 + rbase) * d.C + c0) * ES;
    if (SH == 2 && Wc == W && vec && 32 % (W / 4) == 0) {
        constexpr int PR = W / 4;
        constexpr int RPI = 32 / PR;
        const int j = lane % PR;
        const uint32_t us = (uint32_t)__cvta_generic_to_shared(unit);
        const uint32_t tb = (uint32_t)__cvta_generic_to_shared(tile) + 4 * j;
#pragma unroll 1
        for (int r = lane / PR; r < rows; r += RPI) {
            const int rr = rbase + r;
            const uint32_t q4 = lds_u32(tb + rr * TS) & 0xFCFCFCFCu;
            const uint32_t a4 = lds_u32(tb + anchor[rr] * TS) & 0xFCFCFCFCu;
            const float m = m1s[rr], ma = m1a[rr];
            const float x0 = __fadd_rn(__fmul_rn(lds_f32(__byte_perm(a4, us, 0x7650)), ma),
                                       __fmul_rn(lds_f32(__byte_perm(q4, us, 0x7650)), m));
            const float x1 = __fadd_rn(__fmul_rn(lds_f32(__byte_perm(a4, us, 0x7651)), ma),
                                       __fmul_rn(lds_f32(__byte_perm(q4, us, 0x7651)), m));
            const float x2 = __fadd_rn(__fmul_rn(lds_f32(__byte_perm(a4, us, 0x7652)), ma),
                                       __fmul_rn(lds_f32(__byte_perm(q4, us, 0x7652)), m));
            const float x3 = __fadd_rn(__fmul_rn(lds_f32(__byte_perm(a4, us, 0x7653)), ma),
                                       __fmul_rn(lds_f32(__byte_perm(q4, us, 0x7653)), m));
            char *o = out + ((long long)r * d.C + 4 * j) * ES;
            if (MODE == 2) {
                const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
                *reinterpret_cast<uint2 *>(o) = make_uint2(*reinterpret_cast<const uint32_t *>(&h01),
                                                           *reinterpret_cast<const uint32_t *>(&h23));
            } else {
                *reinterpret_cast<float4 *>(o) = make_float4(x0, x1, x2, x3);
            }
        }
    } else {
        for (int i = lane; i < rows * W; i += 32) {
            const int r = i / W, j = i % W;
            if (j < Wc) {
                const int rr = rbase + r;
                const float x = __fadd_rn(__fmul_rn(unit[tile[anchor[rr] * TS + j] >> SH], m1a[rr]),
                                          __fmul_rn(unit[tile[rr * TS + j] >> SH], m1s[rr]));
                char *e = out + ((long long)r * d.C + j) * ES;
                if (MODE == 2)
                    *reinterpret_cast<__half *>(e) = __float2half_rn(x);
                else
                    *reinterpret_cast<float *>(e) = x;
            }
        }
    }
}

// Decode this thread's Wc symbols of one window into its tile row: rows are P
// entries apart, the search covers the first PS (the alphabet fits in PS).
template <int P, int PS, bool CLAMP, bool TAIL, bool WIDE = false>
__device__ __forceinline__ void decode_window(Stream &s, uint32_t cb, uint32_t fo, uint32_t amax2, uint8_t *my,
                                              int Wc) {
    constexpr int W = DecodeCfg<P>::W;
    constexpr int SH = DecodeCfg<P>::SYM_SHIFT;
    if (Wc == W && !TAIL) {
#pragma unroll 4
        for (int c = 0; c < W; c += 4) {
            const uint32_t rc = cb + 2 * P * c;
            if (WIDE) refill_sel(s); else refill<TAIL>(s);
            const uint32_t e0 = decode_symbol<PS, CLAMP, WIDE>(s, rc, fo, amax2);
            const uint32_t e1 = decode_symbol<PS, CLAMP, WIDE>(s, rc + 2 * P, fo, amax2);
            if (WIDE) refill_sel(s); else refill<TAIL>(s);
            const uint32_t e2 = decode_symbol<PS, CLAMP, WIDE>(s, rc + 4 * P, fo, amax2);
            const uint32_t e3 = decode_symbol<PS, CLAMP, WIDE>(s, rc + 6 * P, fo, amax2);
            // e = 2s: store 4s (SH == 2) or s
            const uint32_t w = SH == 2 ? 2u * (e0 | (e1 << 8) | (e2 << 16) | (e3 << 24))
                                       : (e0 >> 1) | ((e1 >> 1) << 8) | ((e2 >> 1) << 16) | ((e3 >> 1) << 24);
            *reinterpret_cast<uint32_t *>(my + c) = w;
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < Wc; c++) {
            refill<TAIL>(s);
            const uint32_t e = decode_symbol<PS, CLAMP, WIDE>(s, cb + 2 * P * c, fo, amax2);
            my[c] = (uint8_t)(SH == 2 ? 2u * e : e >> 1);
        }
    }
}

// The order in which the decoder's CTAs take the (kv, layer) pairs: by
// decreasing MAX (a wider alphabet costs a longer search and more coded bits
// per symbol), ties in (kv, layer) order; each pair's chunks consecutively.
// Slices of one wave finish together less often than they start, so the
// launch's last, partial wave is cheapest when it holds the lightest slices.
struct SliceOrder {
    uint16_t pair[2 * CG_MAX_LAYERS];  // kv * L + l
};

inline SliceOrder make_slice_order(const Dims &d, const MaxTab &mt) {
    SliceOrder o;
    int start[257] = {0};  // counting sort on 255 - MAX: stable, descending MAX
    for (int kv = 0; kv < 2; kv++)
        for (int l = 0; l < d.L; l++) start[256 - mt.v[kv][l]]++;
    for (int key = 1; key <= 256; key++) start[key] += start[key - 1];
    for (int kv = 0; kv < 2; kv++)
        for (int l = 0; l < d.L; l++) o.pair[start[255 - mt.v[kv][l]]++] = (uint16_t)(kv * d.L + l);
    return o;
}

// CTA = kThreads decoder threads (one per token stream) + one helper warp.
// Iteration i: decoders decode window i with rows[i & 1] and write it out
// while the helper stages rows[(i + 1) & 1]; one barrier per window.
template <int P, int MODE, bool V2, bool DELTA>
__global__ void __launch_bounds__(kThreads + kHelpers, 4) k_decode_pipe(
    const uint8_t *__restrict__ packed, long long packed_bytes, const uint64_t *__restrict__ off,
    const uint32_t *__restrict__ len, const uint16_t *__restrict__ cdf, const uint8_t *__restrict__ rec,
    const uint16_t *__restrict__ max1, Dims d, MaxTab mt, SliceOrder ord, void *__restrict__ out_k,
    void *__restrict__ out_v, long long ols, int32_t *status) {
    using L = PipeSmem<P>;
    constexpr int W = L::W;
    constexpr int TS = L::TS;
    __shared__ __align__(256) float s_unit[256];  // (s - MAX) / MAX
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t *cum = reinterpret_cast<uint16_t *>(smem + L::cum);
    uint16_t *frq = reinterpret_cast<uint16_t *>(smem + L::frq);
    uint8_t *tile = smem + L::tile;
    float *m1s = reinterpret_cast<float *>(smem + L::m1);
    uint8_t *srec = smem + L::recs;

    // CTA b takes chunk b mod nch of the (b / nch)-th (kv, layer) pair in
    // decreasing-alphabet order: the costliest slices start first
    const int pair = ord.pair[blockIdx.x / d.nch];
    const int k = (int)(blockIdx.x % d.nch);
    const int kv = pair >= d.L ? 1 : 0;
    const int l = pair - kv * d.L;
    constexpr bool v2 = V2;  // format 2: CDF rows from count records
    const int A = v2 ? 2 * mt.v[kv][l] + 1 : d.A[kv];
    const uint32_t amax2 = 2u * ((uint32_t)A - 1);
    const int Tk = chunk_tokens(d, k);
    const int tid = threadIdx.x;
    const bool helper = tid >= kThreads;
    const int hl = tid - kThreads;  // helper lane
    const long long t0 = (long long)k * d.Tc;
    const long long side_base = v2 ? record_slice_offset(d, mt, k, kv, l) : cdf_slice_offset(d, k, kv, l);
    const long long sid = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk + tid;
    const int nwin = (d.C + W - 1) / W;

    __shared__ uint16_t s_ftab[kThreads + 2];  // format 2: f(n) = 1 + n (65536 - A) / Tk
    if (v2)
        for (int n = tid; n <= Tk; n += kThreads + kHelpers)
            s_ftab[n] = (uint16_t)(1u + ((uint32_t)n * (kM - (uint32_t)A)) / (uint32_t)Tk);
    // the delta: each row's anchor row and the anchor's max1 (0 for an anchor)
    __shared__ float s_m1a[DELTA ? kThreads : 1];
    __shared__ uint8_t s_anchor[DELTA ? kThreads : 1];
    if (!helper) {
        const int MAX = mt.v[kv][l];
        s_unit[tid] = __fdiv_rn((float)(tid - MAX), (float)MAX);
        if (tid < Tk) m1s[tid] = __half2float(__ushort_as_half(max1[group_index(d, kv, l, t0 + tid)]));
        if (DELTA) {
            const int ra = tid - tid % d.G;
            s_anchor[tid] = (uint8_t)ra;
            s_m1a[tid] = (tid < Tk && ra != tid)
                             ? __half2float(__ushort_as_half(max1[group_index(d, kv, l, t0 + ra)]))
                             : 0.0f;
        }
    }
    Stream s;
    bool corrupt = false, tail = false;
    if (!helper && tid < Tk) {
        long long start = (long long)off[sid];
        long long end = start + (long long)len[sid];
        if (start > packed_bytes || end > packed_bytes) {
            corrupt = true;
            start = min(start, packed_bytes);
            end = min(end, packed_bytes);
        }
        stream_init(s, packed, start, end);
        // whole-word loads stay inside the stream's first and last words; in
        // the buffer's last, partial word they would cross its end
        const long long p4 = packed_bytes & ~3LL;
        tail = end > p4 || (start & ~3LL) >= p4;
    }
    if (!helper) tail = __any_sync(0xFFFFFFFFu, tail);  // warp-uniform refill path
    // 128-bit row loads need 16-byte aligned windows: cdf itself, and every
    // slice offset a multiple of 8 entries (both alphabets multiples of 8)
    const bool vec = ((reinterpret_cast<uintptr_t>(cdf) & 15) == 0) && (d.A[0] % 8 == 0) &&
                     (d.A[1] % 8 == 0);
    bool bad_rec = false;
    if (v2) {
        // records of windows 0 and 1 in, rows of window 0 built; later windows:
        // the helper copies window i + 2's records while the decoder threads
        // build window i + 1's rows and decode window i
        if (helper) {
            copy_records(srec, rec + side_base, min(W, d.C) * A, hl);
            if (nwin > 1) copy_records(srec + W * P, rec + side_base + (long long)W * A, min(W, d.C - W) * A, hl);
        }
        __syncthreads();  // s_ftab and the records
        if (!helper) bad_rec |= build_rows_v2<P>(cum, frq, srec, A, (uint32_t)Tk, W, min(W, d.C), tid, s_ftab);
    } else if (helper) {
        stage_rows<P>(cum, frq, cdf + side_base, A, min(W, d.C), hl, vec);
    }
    __syncthreads();

    const uint32_t fo = (uint32_t)(L::frq - L::cum);
    // whole four-value groups per store: rows, layers and both outputs aligned to the group
    const uintptr_t galign = MODE == 2 ? 8 : 16;
    const bool ovec = (d.C & 3) == 0 && (ols & 3) == 0 &&
                      ((reinterpret_cast<uintptr_t>(out_k) | reinterpret_cast<uintptr_t>(out_v)) & (galign - 1)) == 0;
    const int warp = tid >> 5, lane = tid & 31;
    const int wrows = min(32, Tk - 32 * warp);  // rows of this decoder warp
    uint8_t *wtile = tile + warp * 32 * TS;
    for (int i = 0; i < nwin; i++) {
        const int b = i & 1;
        const int c0 = i * W;
        const int Wc = min(W, d.C - c0);
        if (!helper) {
            if (V2 && i + 1 < nwin)  // window i + 1's rows into the other buffer
                bad_rec |= build_rows_v2<P>(cum + (b ^ 1) * W * P, frq + (b ^ 1) * W * P, srec + (b ^ 1) * W * P, A,
                                            (uint32_t)Tk, W, min(W, d.C - c0 - W), tid, s_ftab);
            if (tid < Tk) {
                // shared address of this buffer's rows; frequencies follow at a fixed offset
                const uint32_t cb = (uint32_t)__cvta_generic_to_shared(cum + b * W * P);
                uint8_t *my = tile + tid * TS;
                constexpr int PH = P > 4 ? P / 2 : P;
                if (!V2 && A == P) {  // format 2's alphabets are odd: never equal to P
                    if (tail)
                        decode_window<P, P, false, true>(s, cb, fo, amax2, my, Wc);
                    else
                        decode_window<P, P, false, false>(s, cb, fo, amax2, my, Wc);
                } else if (A <= PH) {  // the alphabet fits in half the row: one search step less
                    if (tail)
                        decode_window<P, PH, true, true>(s, cb, fo, amax2, my, Wc);
                    else
                        decode_window<P, PH, true, false>(s, cb, fo, amax2, my, Wc);
                } else {
                    if (tail)
                        decode_window<P, P, true, true>(s, cb, fo, amax2, my, Wc);
                    else
                        decode_window<P, P, true, false>(s, cb, fo, amax2, my, Wc);
                }
            }
            if (DELTA) {
                // anchors may sit in other warps' rows: all decoder threads meet
                // (the helper warp does not take part)
                asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory");
                if (wrows > 0)
                    write_window_delta<P, MODE>(tile, s_unit, m1s, s_m1a, s_anchor, d, kv, l, t0, 32 * warp, wrows,
                                                c0, Wc, out_k, out_v, ols, ovec, lane);
            } else {
                __syncwarp();
                if (wrows > 0)
                    write_window<P, MODE, 32>(wtile, s_unit, m1s + 32 * warp, d, kv, l, t0 + 32 * warp, wrows, c0,
                                              Wc, out_k, out_v, ols, ovec, lane);
            }
            __syncwarp();  // the rows are read before the next window overwrites them
        } else if (V2) {
            if (i + 2 < nwin)  // records of window i + 2 replace window i's (its rows were built last round)
                copy_records(srec + b * W * P, rec + side_base + (long long)(c0 + 2 * W) * A,
                             min(W, d.C - c0 - 2 * W) * A, hl);
        } else if (i + 1 < nwin) {
            stage_rows<P>(cum + (b ^ 1) * W * P, frq + (b ^ 1) * W * P, cdf + side_base + (long long)(c0 + W) * A, A,
                          min(W, d.C - c0 - W), hl, vec);
        }
        __syncthreads();
    }
    if (!helper && tid < Tk) {
        // bytes taken from the stream: up to the loaded word (which starts rem
        // bytes before the end), less the whole bytes still in the bit buffer
        const long long consumed = (long long)len[sid] - s.rem - s.nb / 8;
        if ((corrupt || consumed != (long long)len[sid] + 3) && status) atomicOr(status, CG_FLAG_CORRUPT);
    }
    if (bad_rec && status) atomicOr(status, CG_FLAG_CORRUPT);
}

// Latency mode: launches of at most one slice per SM, where a slice's time is
// set by the serial chain of each token stream. A CTA of DEC + 256 threads
// splits the work by warp: the first DEC threads only decode (thread t decodes
// token R0 + t, searching four ways per level: fewer dependent loads per
// symbol), the other 256 build window i + 1's CDF rows and write window i - 1's
// dequantised rows out while window i is decoded, from double-buffered rows
// and symbol tiles; one named barrier of all threads per window hands them
// over.
// DEC = 256: a CTA per slice (at most one slice per SM). DEC = 128 (at most
// one slice per two SMs, no delta): two CTAs per slice, each decoding half of
// its token streams (rows [R0, R0 + h), h = ceil(Tc_k / 2)) with its own copy
// of the CDF rows, which halves the instructions each SM issues per symbol.
template <int P, int DEC>
struct LmDecSmem {
    static constexpr int W = DecodeCfg<P>::W;
    static constexpr int TS = DecodeCfg<P>::TS;
    static constexpr size_t cum = 0;                                        // [2][W][P] uint16
    static constexpr size_t frq = cum + 2ull * W * P * 2;                   // [2][W][P] uint16
    static constexpr size_t tile = (frq + 2ull * W * P * 2 + 15) & ~15ull;  // [2][DEC * TS]
    static constexpr size_t m1 = tile + 2ull * DEC * TS;                    // float[DEC]
    static constexpr size_t recs = m1 + DEC * 4;                            // format 2: [W * P] records
    static constexpr size_t bytes = recs + 1ull * W * P;
};

template <int P, int MODE, bool V2, bool DELTA, int DEC>
__global__ void __launch_bounds__(DEC + kThreads, 1) k_decode_lm(
    const uint8_t *__restrict__ packed, long long packed_bytes, const uint64_t *__restrict__ off,
    const uint32_t *__restrict__ len, const uint16_t *__restrict__ cdf, const uint8_t *__restrict__ rec,
    const uint16_t *__restrict__ max1, Dims d, MaxTab mt, void *__restrict__ out_k, void *__restrict__ out_v,
    long long ols, int32_t *status) {
    using L = LmDecSmem<P, DEC>;
    constexpr int W = L::W;
    constexpr int TS = L::TS;
    constexpr int SUP = kThreads;          // support threads
    constexpr int NT = DEC + SUP;          // threads
    constexpr int NP = kThreads / DEC;     // CTAs per slice
    static_assert(!DELTA || NP == 1, "a token's anchor row must be in the same CTA");
    __shared__ __align__(256) float s_unit[256];  // (s - MAX) / MAX
    __shared__ uint16_t s_ftab[kThreads + 2];
    __shared__ float s_m1a[DELTA ? kThreads : 1];
    __shared__ uint8_t s_anchor[DELTA ? kThreads : 1];
    extern __shared__ __align__(16) unsigned char smem[];
    uint16_t *cum = reinterpret_cast<uint16_t *>(smem + L::cum);
    uint16_t *frq = reinterpret_cast<uint16_t *>(smem + L::frq);
    uint8_t *tile = smem + L::tile;
    float *m1s = reinterpret_cast<float *>(smem + L::m1);
    uint8_t *srec = smem + L::recs;

    int k, kv, l;
    slice_coords(d, blockIdx.x / NP, k, kv, l);
    const int A = V2 ? 2 * mt.v[kv][l] + 1 : d.A[kv];
    const uint32_t amax2 = 2u * ((uint32_t)A - 1);
    const int Tk = chunk_tokens(d, k);
    const int hrows = (Tk + NP - 1) / NP;
    const int R0 = (int)(blockIdx.x % NP) * hrows;
    const int nr = min(hrows, Tk - R0);  // this CTA's rows of the slice
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool dec = tid < DEC;
    const int st = tid - DEC;  // support thread 0 .. SUP - 1
    const long long t0 = (long long)k * d.Tc + R0;  // first row of this CTA
    const long long side_base = V2 ? record_slice_offset(d, mt, k, kv, l) : cdf_slice_offset(d, k, kv, l);
    const long long sid = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk + R0 + tid;
    const int nwin = (d.C + W - 1) / W;

    for (int n = tid; n <= Tk; n += NT)
        if (V2) s_ftab[n] = (uint16_t)(1u + ((uint32_t)n * (kM - (uint32_t)A)) / (uint32_t)Tk);
    for (int q = tid; q < 256; q += NT) {
        const int MAX = mt.v[kv][l];
        s_unit[q] = __fdiv_rn((float)(q - MAX), (float)MAX);
    }
    if (dec) {
        if (tid < nr) m1s[tid] = __half2float(__ushort_as_half(max1[group_index(d, kv, l, t0 + tid)]));
        if (DELTA) {
            const int ra = tid - tid % d.G;
            s_anchor[tid] = (uint8_t)ra;
            s_m1a[tid] = (tid < Tk && ra != tid)
                             ? __half2float(__ushort_as_half(max1[group_index(d, kv, l, t0 + ra)]))
                             : 0.0f;
        }
    }
    Stream s;
    bool corrupt = false, tail = false;
    if (dec && tid < nr) {
        long long start = (long long)off[sid];
        long long end = start + (long long)len[sid];
        if (start > packed_bytes || end > packed_bytes) {
            corrupt = true;
            start = min(start, packed_bytes);
            end = min(end, packed_bytes);
        }
        stream_init(s, packed, start, end);
        const long long p4 = packed_bytes & ~3LL;
        tail = end > p4 || (start & ~3LL) >= p4;
    }
    if (dec) tail = __any_sync(0xFFFFFFFFu, tail);
    const bool vec = ((reinterpret_cast<uintptr_t>(cdf) & 15) == 0) && (d.A[0] % 8 == 0) && (d.A[1] % 8 == 0);
    const uintptr_t galign = MODE == 2 ? 8 : 16;
    const bool ovec = (d.C & 3) == 0 && (ols & 3) == 0 &&
                      ((reinterpret_cast<uintptr_t>(out_k) | reinterpret_cast<uintptr_t>(out_v)) & (galign - 1)) == 0;
    bool bad_rec = false;
    __syncthreads();  // tables and max1

    // support: the rows of window j into buffer j & 1
    auto build = [&](int j) {
        const int c0 = j * W, Wc = min(W, d.C - c0);
        uint16_t *cb = cum + (j & 1) * W * P, *fb = frq + (j & 1) * W * P;
        if (V2) {
            // the window's records (contiguous) into shared memory, all support threads at once
            const uint8_t *rw = rec + side_base + (long long)c0 * A;
            const int nb = Wc * A;
            const int lead = (int)((16 - (reinterpret_cast<uintptr_t>(rw) & 15)) & 15);  // bytes before a 16-byte boundary
            const int head = min(lead, nb), nvec = (nb - head) >> 4;
            for (int i = st; i < head; i += SUP) srec[i] = __ldg(rw + i);
            for (int i = st; i < nvec; i += SUP) {
                const uint4 q = __ldg(reinterpret_cast<const uint4 *>(rw + head) + i);
                uint8_t *dst = srec + head + 16 * i;
#pragma unroll
                for (int b = 0; b < 4; b++) {
                    const uint32_t w = b == 0 ? q.x : b == 1 ? q.y : b == 2 ? q.z : q.w;
#pragma unroll
                    for (int y = 0; y < 4; y++) dst[4 * b + y] = (uint8_t)(w >> (8 * y));
                }
            }
            for (int i = head + 16 * nvec + st; i < nb; i += SUP) srec[i] = __ldg(rw + i);
            asm volatile("bar.sync 1, %0;" ::"n"(SUP) : "memory");  // the records are in
            bad_rec |= build_rows_v2<P>(cb, fb, srec, A, (uint32_t)Tk, W, Wc, st, s_ftab);
        } else if (warp == DEC / 32) {
            stage_rows<P>(cb, fb, cdf + side_base + (long long)c0 * A, A, Wc, lane, vec);
        }
    };
    // support: window j's decoded tile out
    auto write = [&](int j) {
        const int c0 = j * W, Wc = min(W, d.C - c0);
        const uint8_t *tb = tile + (j & 1) * DEC * TS;
        if (DELTA) {
            const int sw = warp - DEC / 32;
            const int rows = min(32, nr - 32 * sw);
            if (rows > 0)
                write_window_delta<P, MODE>(tb, s_unit, m1s, s_m1a, s_anchor, d, kv, l, t0, 32 * sw, rows, c0, Wc,
                                            out_k, out_v, ols, ovec, lane);
        } else {
            write_window<P, MODE, SUP>(tb, s_unit, m1s, d, kv, l, t0, nr, c0, Wc, out_k, out_v, ols, ovec, st);
        }
    };
    if (!dec) build(0);
    asm volatile("bar.sync 2, %0;" ::"n"(NT) : "memory");  // window 0's rows
    const uint32_t fo = (uint32_t)(L::frq - L::cum);
    for (int i = 0; i < nwin; i++) {
        const int b = i & 1;
        const int Wc = min(W, d.C - i * W);
        if (dec) {
            if (tid < nr) {
                const uint32_t cb = (uint32_t)__cvta_generic_to_shared(cum + b * W * P);
                uint8_t *my = tile + b * DEC * TS + tid * TS;
                constexpr int PH = P > 4 ? P / 2 : P;
                if (!V2 && A == P) {
                    if (tail)
                        decode_window<P, P, false, true, true>(s, cb, fo, amax2, my, Wc);
                    else
                        decode_window<P, P, false, false, true>(s, cb, fo, amax2, my, Wc);
                } else if (A <= PH) {
                    if (tail)
                        decode_window<P, PH, true, true, true>(s, cb, fo, amax2, my, Wc);
                    else
                        decode_window<P, PH, true, false, true>(s, cb, fo, amax2, my, Wc);
                } else {
                    if (tail)
                        decode_window<P, P, true, true, true>(s, cb, fo, amax2, my, Wc);
                    else
                        decode_window<P, P, true, false, true>(s, cb, fo, amax2, my, Wc);
                }
            }
        } else {
            if (i + 1 < nwin) build(i + 1);
            if (i >= 1) write(i - 1);
        }
        asm volatile("bar.sync 2, %0;" ::"n"(NT) : "memory");  // window i handed over
    }
    if (!dec) write(nwin - 1);
    if (dec && tid < nr) {
        const long long consumed = (long long)len[sid] - s.rem - s.nb / 8;
        if ((corrupt || consumed != (long long)len[sid] + 3) && status) atomicOr(status, CG_FLAG_CORRUPT);
    }
    if (bad_rec && status) atomicOr(status, CG_FLAG_CORRUPT);
}

template <int P, int MODE, bool V2, bool DELTA>
cudaError_t launch_pm(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off, const uint32_t *len,
                      const uint16_t *cdf, const uint8_t *rec, const uint16_t *max1, const Dims &d, const MaxTab &mt,
                      void *out_k, void *out_v, long long ols, int32_t *status, cudaStream_t s) {
    const unsigned nslices = (unsigned)(2LL * d.L * d.nch);
    const int sms = device_sm_count();
    if constexpr (!DELTA) {
        if (sms > 0 && 2 * nslices <= (unsigned)sms) {  // latency mode: a slice per two SMs
            const int lsmem = (int)LmDecSmem<P, 128>::bytes;
            cudaError_t err = cudaFuncSetAttribute(k_decode_lm<P, MODE, V2, false, 128>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, lsmem);
            if (err != cudaSuccess) return err;
            k_decode_lm<P, MODE, V2, false, 128><<<2 * nslices, 128 + kThreads, lsmem, s>>>(
                packed, (long long)packed_bytes, off, len, cdf, rec, max1, d, mt, out_k, out_v, ols, status);
            return cudaGetLastError();
        }
    }
    if (sms > 0 && nslices <= (unsigned)sms) {  // latency mode: a slice per SM
        const int lsmem = (int)LmDecSmem<P, 256>::bytes;
        cudaError_t err = cudaFuncSetAttribute(k_decode_lm<P, MODE, V2, DELTA, 256>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, lsmem);
        if (err != cudaSuccess) return err;
        k_decode_lm<P, MODE, V2, DELTA, 256><<<nslices, 512, lsmem, s>>>(
            packed, (long long)packed_bytes, off, len, cdf, rec, max1, d, mt, out_k, out_v, ols, status);
        return cudaGetLastError();
    }
    const int smem = (int)PipeSmem<P>::bytes;
    cudaError_t err = cudaFuncSetAttribute(k_decode_pipe<P, MODE, V2, DELTA>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    k_decode_pipe<P, MODE, V2, DELTA><<<nslices, kThreads + kHelpers, smem, s>>>(
        packed, (long long)packed_bytes, off, len, cdf, rec, max1, d, mt, make_slice_order(d, mt), out_k, out_v,
        ols, status);
    return cudaGetLastError();
}

template <int P, bool DELTA>
cudaError_t launch_p(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off, const uint32_t *len,
                     const uint16_t *cdf, const uint8_t *rec, const uint16_t *max1, const Dims &d, const MaxTab &mt,
                     int out_dtype, void *out_k, void *out_v, long long ols, int32_t *status, cudaStream_t s) {
    if (rec) {
        if (out_dtype == 2)
            return launch_pm<P, 2, true, DELTA>(packed, packed_bytes, off, len, cdf, rec, max1, d, mt, out_k, out_v,
                                                ols, status, s);
        return launch_pm<P, 1, true, DELTA>(packed, packed_bytes, off, len, cdf, rec, max1, d, mt, out_k, out_v, ols,
                                            status, s);
    }
    if (out_dtype == 2)
        return launch_pm<P, 2, false, DELTA>(packed, packed_bytes, off, len, cdf, rec, max1, d, mt, out_k, out_v, ols,
                                             status, s);
    return launch_pm<P, 1, false, DELTA>(packed, packed_bytes, off, len, cdf, rec, max1, d, mt, out_k, out_v, ols,
                                         status, s);
}

// The CDF width for the call's largest alphabet (format 2: 2 * MAX + 1), then
// the instantiation.
template <bool DELTA>
cudaError_t launch_pipe_any(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off, const uint32_t *len,
                            const uint16_t *cdf, const uint8_t *rec, const uint16_t *max1, const Dims &d,
                            const MaxTab &mt, int out_dtype, void *out_k, void *out_v, long long ols,
                            int32_t *status, cudaStream_t s) {
    int A = d.A[0] > d.A[1] ? d.A[0] : d.A[1];
    if (rec) {
        A = 0;
        for (int kv = 0; kv < 2; kv++)
            for (int l = 0; l < d.L; l++) A = 2 * mt.v[kv][l] + 1 > A ? 2 * mt.v[kv][l] + 1 : A;
    }
#define CG_LAUNCH_P(PP)                                                                                       \
    return launch_p<PP, DELTA>(packed, packed_bytes, off, len, cdf, rec, max1, d, mt, out_dtype, out_k, out_v, \
                               ols, status, s)
    if (A <= 8) CG_LAUNCH_P(8);
    if (A <= 16) CG_LAUNCH_P(16);
    if (A <= 32) CG_LAUNCH_P(32);
    if (A <= 64) CG_LAUNCH_P(64);
    if (A <= 128) CG_LAUNCH_P(128);
    CG_LAUNCH_P(256);
#undef CG_LAUNCH_P
}

}  // namespace
}  // namespace cg
