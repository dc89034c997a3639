// compress.cu - the fused compress kernel: adaptive quantisation
// [CG §2.3(1)], per-channel CDF [CG §2.3(2)], range encoding [CG §1.2(3)] and
// packing of one (chunk, kv, layer) slice per CTA, straight from fp16.
//
// Used for chunks of up to 256 tokens, alphabets up to 64 (a 32-symbol and a
// 64-symbol form of the kernel), C % 8 == 0 and 16-byte aligned rows (other
// shapes take the quantise + slice-coder + scan kernels). One thread per
// token stream, 256 threads, three CTAs per SM (two for the 64-symbol form
// with the delta). Launches of at most one slice per SM take the latency-mode
// kernels further down instead.
//
// The fp16 slice [Tc_k][C] arrives in [rows][64-channel] boxes by TMA
// (cp.async.bulk.tensor, completion on an mbarrier; every wait is bounded and
// sets CG_FLAG_TIMEOUT when it runs out). Per CTA:
//   0. take a slice ticket (slices start in stream order);
//   1. max1 pass: the slice's boxes stream through two buffers; each lane
//      keeps the running max of the fp16 magnitude bits of its rows, then a
//      half-warp reduction gives max1 per token and factor = MAX / max1
//      (0 for an all-zero row: every value then maps to MAX);
//   then per window of 64 channels (the next window's box is in flight while
//   this one is coded):
//   2. quantise the box, four channels per lane, two rows per warp
//      instruction, each warp on the rows it codes later (so only a warp-level
//      sync separates its coding of one window from its writes of the next).
//      y = RN(RN(x * factor) + MAX) in binary32 (the adds two at a time as
//      f32x2); adding 1.5 * 2^23 rounds y to the nearest integer, ties to even, into
//      the low bits. Symbols go to a shared tile as 8q (4q for 64 symbols: a
//      byte offset into a CDF row), counts to a [symbol][channel] table of
//      16-bit counters;
//   3. four threads per channel turn its counts into a CDF row in one pass
//      (own eight (sixteen) symbols, then a four-lane scan), zeroing the
//      counters they read, and write the row's entries to shared memory and
//      lo (format 1) or the count record (format 2) to the output;
//   4. every thread codes its token's 64 symbols;
//   after the last window:
//   5. each stream's length and the slice's byte total go out; no CTA of this
//      kernel waits on another.
// k_pack then places the slices: it publishes every slice total at once, so
// its decoupled look-back over the preceding slices only waits for CTAs that
// have just started (spins are bounded), and copies the streams from the
// staging area (just written, mostly L2-resident) into the packed buffer,
// clipped at the capacity.
#include <cuda.h>  // CUtensorMap and its enums; the encoder is fetched through the runtime
#include <cuda_fp16.h>

#include <mutex>

#include "cg_internal.cuh"
#include "coder.cuh"

namespace cg {
namespace {

constexpr int kNT = 256;  // threads = max tokens per chunk on this path
constexpr int kNW = kNT / 32;
constexpr int kW = 64;        // channels per window = fp16 box width (128-byte rows)
constexpr int kAmax = 32;     // largest alphabet on this path
constexpr int kAS = kAmax + 1;  // (lo, f) entries per CDF row in shared memory
constexpr int kSP = 8;        // symbols per CDF thread (four threads per channel)
constexpr int kCntRow = kW + 2;  // 16-bit counters per symbol row (one spare word)
constexpr int kSymRow = kW + 4;  // bytes per symbol-tile row (spreads rows over banks)
constexpr uint32_t kTotal = 65536u;
constexpr uint32_t kMagic = 0x4B400000u;  // bits of 1.5 * 2^23
constexpr unsigned long long kFlagAggregate = 1ull << 62;
constexpr unsigned long long kValueMask = (1ull << 62) - 1;
constexpr int kSpinLimit = 1 << 22;
constexpr int kWaitLimit = 1 << 22;

// The union region: CDF rows, counters and symbol tile while coding; the
// second fp16 box buffer during the max1 pass.
constexpr int kCdfwBytes = kW * kAS * 8;
constexpr int kCntBytes = kAmax * kCntRow * 2;
constexpr int kSymBytes = kNT * kSymRow;
constexpr int kBoxBytesMax = kNT * kW * 2;
constexpr int kCodeBytes = kCdfwBytes + kCntBytes + kSymBytes;
constexpr int kUnionBytes = kCodeBytes > kBoxBytesMax ? kCodeBytes : kBoxBytesMax;

// Sizes of the throughput kernel for alphabets up to AM symbols (32, or 64 for
// layers of up to 64 bins, format 1, or 65, format 2): rows of AM + 1 CDF
// entries, AM / 4 symbols per CDF thread, an AM-row counter table. An entry is
// (lo, f) as two words for 32 symbols, one word lo | (f - 1) << 16 for 64 (so
// that three CTAs fit an SM). Tile bytes hold q << SH, the byte offset of the
// entry in its row (8q for q < 32, 4q for q < 64).
template <int AM>
struct Alpha {
    static constexpr int AS = AM + 1;
    static constexpr int SP = AM / 4;
    static constexpr int SH = AM <= 32 ? 3 : 2;
    static constexpr int EB = 1 << SH;  // bytes per CDF entry
    static constexpr int cdfw_bytes = kW * AS * EB;
    static constexpr int cnt_bytes = AM * kCntRow * 2;
    static constexpr int code_bytes = cdfw_bytes + cnt_bytes + kSymBytes;
    static constexpr int union_bytes = code_bytes > kBoxBytesMax ? code_bytes : kBoxBytesMax;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bounded wait for the phase with the given parity; false if it ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < kWaitLimit; i++) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

// Box (x = channel, y = token, z = layer) of the tensor map into shared memory.
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap *map, int x, int y, int z,
                                         uint32_t bar, uint32_t bytes) {
    mbar_expect_tx(bar, bytes);
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Pull a box into L2 ahead of its TMA load.
__device__ __forceinline__ void tma_prefetch_l2(const CUtensorMap *map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void red_add(uint32_t addr, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Thread-block cluster helpers (two CTAs sharing a slice in latency mode).
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared address `addr` of this CTA, as the same location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ uint32_t ld_peer_u16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared::cluster.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_peer_u64(uint32_t addr) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

// Every thread of both CTAs of the cluster arrives, then waits.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive (release, cluster scope) on the mbarrier at shared::cluster address `remote`.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// Bounded wait (acquire, cluster scope) for the phase with the given parity.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < kWaitLimit; i++) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ unsigned long long pair(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}

// y + 1.5 * 2^23 for two values, y = RN(RN(x * factor) + MAX) (specification
// Q); the low byte of each result is rint(y) for y in [-0.5, 255]. The
// products stay scalar: ptxas fuses a packed mul.rn.f32x2 feeding a packed
// add.rn.f32x2 into one rounding (a fused multiply-add), which moves rare
// near-ties to the next level; the two adds are packed.
__device__ __forceinline__ void quant_pair(uint32_t h2, float f, unsigned long long fm, unsigned long long mg,
                                           uint32_t &b0, uint32_t &b1) {
    const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
    const float p0 = __fmul_rn(x.x, f), p1 = __fmul_rn(x.y, f);
    asm("{\n\t.reg .b64 t;\n\t"
        "mov.b64 t, {%2, %3};\n\t"
        "add.rn.f32x2 t, t, %4;\n\t"
        "add.rn.f32x2 t, t, %5;\n\t"
        "mov.b64 {%0, %1}, t;\n\t}"
        : "=r"(b0), "=r"(b1)
        : "f"(p0), "f"(p1), "l"(fm), "l"(mg));
}

// quant_pair for two binary32 values (the delta's d).
__device__ __forceinline__ void quant_pair_f(float d0, float d1, float f, unsigned long long fm,
                                             unsigned long long mg, uint32_t &b0, uint32_t &b1) {
    const float p0 = __fmul_rn(d0, f), p1 = __fmul_rn(d1, f);
    asm("{\n\t.reg .b64 t;\n\t"
        "mov.b64 t, {%2, %3};\n\t"
        "add.rn.f32x2 t, t, %4;\n\t"
        "add.rn.f32x2 t, t, %5;\n\t"
        "mov.b64 {%0, %1}, t;\n\t}"
        : "=r"(b0), "=r"(b1)
        : "f"(p0), "f"(p1), "l"(fm), "l"(mg));
}

__device__ __forceinline__ float lds_f32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}

// Smallest binary16 >= m (m >= 0), as bits; 65504's bits above it or for NaN.
__device__ __forceinline__ uint32_t half_up_bits(float m) {
    const uint32_t h = __half_as_ushort(__float2half_ru(m));
    return h >= 0x7C00u ? 0x7BFFu : h;
}

// The delta [CG §1.2(1)] on one quad of row r, given the anchor row's quad xa:
// a^ = D(Q(xa)) (the anchor's q recomputed with its factor fa, its table
// entry times ma; ma = 0 makes an anchor its own zero reference), d = x - a^.
__device__ __forceinline__ void delta_quad(uint2 x, uint2 xa, float fa, float ma, uint32_t us, uint32_t qmax,
                                           unsigned long long fm, unsigned long long mg, float (&dv)[4]) {
    uint32_t c0, c1, c2, c3;
    quant_pair(xa.x, fa, fm, mg, c0, c1);
    quant_pair(xa.y, fa, fm, mg, c2, c3);
    // table index clamped to [0, 2 MAX]: in bounds whatever the box holds
    const float a0 = __fmul_rn(lds_f32(us + 4u * min(c0 - kMagic, qmax)), ma);
    const float a1 = __fmul_rn(lds_f32(us + 4u * min(c1 - kMagic, qmax)), ma);
    const float a2 = __fmul_rn(lds_f32(us + 4u * min(c2 - kMagic, qmax)), ma);
    const float a3 = __fmul_rn(lds_f32(us + 4u * min(c3 - kMagic, qmax)), ma);
    const float2 x01 = __half22float2(*reinterpret_cast<const __half2 *>(&x.x));
    const float2 x23 = __half22float2(*reinterpret_cast<const __half2 *>(&x.y));
    dv[0] = __fsub_rn(x01.x, a0);
    dv[1] = __fsub_rn(x01.y, a1);
    dv[2] = __fsub_rn(x23.x, a2);
    dv[3] = __fsub_rn(x23.y, a3);
}

__device__ __forceinline__ unsigned long long ld_acquire(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned long long *p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// state: [0] compress ticket, [1] pack ticket, [2 + s] look-back slot of
// slice s, [2 + nslices + s] byte total of slice s (written by the compress
// kernel). The tickets and slots start at zero.
__global__ void k_compress_init(unsigned long long *state, long long nslices) {
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < 2 + nslices;
         i += (long long)gridDim.x * blockDim.x)
        state[i] = 0ull;
}

// Step 2 for one window: quantise this lane's quads of its rows, store 8q to
// the symbol tile and count q. SAFE (a slice with a non-finite max1, or a box
// whose wait ran out) clamps q to [0, 2 MAX] before using it; finite input
// under its own max1 needs no clamp.
// fac[r * FS] is row r's factor (FS = 17: the factors sit in the symbol tile's
// row padding).
template <bool SAFE, int SH = 3, int FS = 1>
__device__ __forceinline__ void quantise_window(const unsigned char *box, const float *fac, uint8_t *sym,
                                                uint32_t cnt_lane, int rbase, int kq, int Tk,
                                                unsigned long long fm, unsigned long long mg, uint32_t qmax) {
#pragma unroll 4
    for (int i = 0; i < kNT / 32 * 2; i++) {
        const int r = rbase + 2 * i;
        if (r >= Tk) break;
        const uint2 x = *reinterpret_cast<const uint2 *>(box + r * (kW * 2) + 8 * kq);
        const float f = fac[r * FS];
        uint32_t b0, b1, b2, b3;
        quant_pair(x.x, f, fm, mg, b0, b1);
        quant_pair(x.y, f, fm, mg, b2, b3);
        if (SAFE) {
            b0 = min(b0 - kMagic, qmax) + kMagic;
            b1 = min(b1 - kMagic, qmax) + kMagic;
            b2 = min(b2 - kMagic, qmax) + kMagic;
            b3 = min(b3 - kMagic, qmax) + kMagic;
        }
        const uint32_t lo2 = __byte_perm(b0, b1, 0x0040), hi2 = __byte_perm(b2, b3, 0x0040);
        *reinterpret_cast<uint32_t *>(sym + r * kSymRow + 4 * kq) = __byte_perm(lo2, hi2, 0x5410) << SH;
        // counter word of (q, channel pair) = cnt_lane + 132 q (+4 for the second pair)
        red_add(b0 * (kCntRow * 2) + cnt_lane, 1u);
        red_add(b1 * (kCntRow * 2) + cnt_lane, 1u << 16);
        red_add(b2 * (kCntRow * 2) + cnt_lane + 4, 1u);
        red_add(b3 * (kCntRow * 2) + cnt_lane + 4, 1u << 16);
    }
}

// Step 3 for one window: CDF thread ct (channel ct >> 2, part ct & 3) turns
// the counts of its eight symbols into (lo, f) entries of the channel's row,
// clearing the counters it read, and writes the side output (CDF entries, or
// the format 2 count record).
// NC == 2 (two CTAs per slice): the counts are this CTA's table `tb` (in
// elements) plus the same table of the peer CTA (rank ^ 1), read through
// distributed shared memory; the other table (the last window's, which both
// CTAs have read) is cleared instead; only rank 0 writes the side output.
template <bool V2, int NC = 1, int AM = kAmax>
__device__ __forceinline__ void build_cdf_window(int ct, uint16_t *cnt16, const uint16_t *ftab, void *cdfw,
                                                 void *side_out, long long side_base, int c0, int Wc, int A,
                                                 int tb = 0, uint32_t rank = 0) {
    constexpr int kSP = Alpha<AM>::SP;
    constexpr int kAS = Alpha<AM>::AS;
    constexpr int kCntBytes = Alpha<AM>::cnt_bytes;
    const int c = ct >> 2, p = ct & 3;
    // a warp covers eight channels and Wc is a multiple of 8, so a warp
    // is entirely inside or entirely outside the window
    if (c >= Wc) return;
    uint32_t fj[kSP], pre[kSP];
    uint32_t sum = 0, key = 0;
    uint32_t nb[(kSP + 3) / 4] = {};  // counts, one byte each (capped)
#pragma unroll
    for (int j = 0; j < kSP; j++) {
        const int s = kSP * p + j;
        uint32_t fv = 0;
        if (s < A) {
            uint16_t *cp = cnt16 + s * kCntRow + c;
            uint32_t n;
            if constexpr (NC == 2) {
                n = (uint32_t)cp[tb] + ld_peer_u16(peer_addr(smem_u32(cp + tb), rank ^ 1u));
                cp[(kCntBytes / 2) - tb] = 0;
            } else {
                n = *cp;
                *cp = 0;
            }
            fv = ftab[n];
            key = max(key, (n << 8) | (255u - (uint32_t)s));  // largest n, then smallest s
            if (V2) nb[j / 4] |= min(n, 255u) << (8 * (j % 4));
        }
        pre[j] = sum;
        sum += fv;
        fj[j] = fv;
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o, 4);
        if (p >= o) incl += v;
        key = max(key, __shfl_xor_sync(0xFFFFFFFFu, key, o));
    }
    const uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 3, 4);
    const uint32_t base = incl - sum;
    const uint32_t best = 255u - (key & 255u);
    const uint32_t extra = kTotal - total;
    unsigned char *row = static_cast<unsigned char *>(cdfw) + c * kAS * Alpha<AM>::EB;
    const bool out = NC == 1 || rank == 0;
    auto put = [&](uint32_t s, uint32_t lo, uint32_t f) {
        if constexpr (Alpha<AM>::EB == 8)
            reinterpret_cast<uint2 *>(row)[s] = make_uint2(lo, f);
        else
            reinterpret_cast<uint32_t *>(row)[s] = lo | ((f - 1u) << 16);
    };
    if (V2) {
        // count record: the mode, then the other symbols' counts
        uint8_t *g = static_cast<uint8_t *>(side_out) + side_base + (long long)(c0 + c) * A;
        if (p == 0 && out) g[0] = (uint8_t)best;
#pragma unroll
        for (int j = 0; j < kSP; j++) {
            const uint32_t s = (uint32_t)(kSP * p + j);
            if ((int)s < A) {
                const uint32_t lo = base + pre[j] + (s > best ? extra : 0u);
                const uint32_t f = fj[j] + (s == best ? extra : 0u);
                put(s, lo, f);
                if (s != best && out) g[s + (s < best ? 1u : 0u)] = (uint8_t)((nb[j / 4] >> (8 * (j % 4))) & 0xFFu);
            }
        }
    } else {
        uint16_t *g = static_cast<uint16_t *>(side_out) + side_base + (long long)(c0 + c) * A;
        // rows of a multiple of 8 entries (C % 8 == 0, so every row and every
        // thread's part of one starts 16-byte aligned): the part leaves as
        // 16-byte stores instead of one store per entry
        const bool vec = (A & 7) == 0 && (reinterpret_cast<uintptr_t>(side_out) & 15) == 0;
        uint32_t pk[kSP / 2];
#pragma unroll
        for (int j = 0; j < kSP; j++) {
            const uint32_t s = (uint32_t)(kSP * p + j);
            uint32_t lo = 0;
            if ((int)s < A) {
                lo = base + pre[j] + (s > best ? extra : 0u);
                const uint32_t f = fj[j] + (s == best ? extra : 0u);
                put(s, lo, f);
                if (out && !vec) g[s] = (uint16_t)lo;
            }
            if (j & 1)
                pk[j / 2] |= lo << 16;
            else
                pk[j / 2] = lo & 0xFFFFu;
        }
        if (out && vec) {
            // eight entries a store; A is a multiple of 8, so each store is
            // wholly inside the row or wholly past it
            uint4 *gv = reinterpret_cast<uint4 *>(g + kSP * p);
#pragma unroll
            for (int q = 0; q < kSP / 8; q++)
                if (kSP * p + 8 * q < A) gv[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
    }
}

// Step 4 for one window: code this thread's row of the symbol tile (bytes
// q << SH) with the window's CDF rows: two-word (lo, f) entries for 32 symbols,
// one-word lo | (f - 1) << 16 entries for 64.
template <int AM>
__device__ __forceinline__ uint2 ld_entry(const unsigned char *at) {
    if constexpr (Alpha<AM>::EB == 8)
        return *reinterpret_cast<const uint2 *>(at);
    else
        return make_uint2(*reinterpret_cast<const uint32_t *>(at), 0u);
}

template <int AM>
__device__ __forceinline__ void enc_entry(Enc &e, uint2 en) {
    if constexpr (Alpha<AM>::EB == 8)
        enc_symbol_lf(e, en.x, en.y);
    else
        enc_symbol_m1(e, en.x);
}

// SEL: the flush without a branch (enc_flush_sel), for the latency-mode coders.
template <int AM = kAmax, bool SEL = false>
__device__ __forceinline__ void encode_window(Enc &e, uint8_t *stream, const uint8_t *symrow, const void *cdfw,
                                              int Wc) {
    constexpr int kRow = Alpha<AM>::AS * Alpha<AM>::EB;  // bytes per CDF row
    const unsigned char *rows = static_cast<const unsigned char *>(cdfw);
    if (Wc == kW) {
#pragma unroll
        for (int g = 0; g < kW / 4; g++) {
            // every tile byte is q << SH (written by the quantiser), the aligned
            // offset of q's entry in its row: byte loads, no unpacking
            const unsigned char *m4 = symrow + 4 * g;
            const unsigned char *r0 = rows + (4 * g) * kRow;
            // (the four entries are loaded ahead of the flush's stores)
            const uint2 e0 = ld_entry<AM>(r0 + m4[0]);
            const uint2 e1 = ld_entry<AM>(r0 + kRow + m4[1]);
            const uint2 e2 = ld_entry<AM>(r0 + 2 * kRow + m4[2]);
            const uint2 e3 = ld_entry<AM>(r0 + 3 * kRow + m4[3]);
            if (SEL)
                enc_flush_sel(e, stream);
            else if (e.nbits >= 32)
                enc_flush_word(e, stream);
            enc_entry<AM>(e, e0);
            enc_entry<AM>(e, e1);
            if (SEL)
                enc_flush_sel(e, stream);
            else if (e.nbits >= 32)
                enc_flush_word(e, stream);
            enc_entry<AM>(e, e2);
            enc_entry<AM>(e, e3);
        }
    } else {
        for (int c = 0; c < Wc; c++) {
            const uint2 en = ld_entry<AM>(rows + c * kRow + (symrow[c] & (0xFFu << Alpha<AM>::SH)));
            if (e.nbits >= 32) enc_flush_word(e, stream);
            enc_entry<AM>(e, en);
        }
    }
}

// The reference max1 of row r with anchor row ra: the anchor's, or 0 for an
// anchor itself.
__device__ __forceinline__ float anchor_m1(const uint16_t *m1, int ra, int r) {
    return ra == r ? 0.0f : __half2float(__ushort_as_half(m1[ra]));
}

// Step 2 with the delta: every row as d = x - a^ (anchors against +-0), q
// clamped to [0, 2 MAX] (max1 rounded to 65504 can sit below max |d|).
template <int SH = 3>
__device__ __forceinline__ void quantise_window_delta(const unsigned char *box, const float *fac,
                                                      const uint8_t *anchor, const uint16_t *m1, uint32_t us,
                                                      uint8_t *sym, uint32_t cnt_lane, int rbase, int kq, int Tk,
                                                      unsigned long long fm, unsigned long long mg, uint32_t qmax) {
#pragma unroll 2
    for (int i = 0; i < kNT / 32 * 2; i++) {
        const int r = rbase + 2 * i;
        if (r >= Tk) break;
        const int ra = anchor[r];
        const uint2 x = *reinterpret_cast<const uint2 *>(box + r * (kW * 2) + 8 * kq);
        const uint2 xa = *reinterpret_cast<const uint2 *>(box + ra * (kW * 2) + 8 * kq);
        float dv[4];
        delta_quad(x, xa, fac[ra], anchor_m1(m1, ra, r), us, qmax, fm, mg, dv);
        const float f = fac[r];
        uint32_t b0, b1, b2, b3;
        quant_pair_f(dv[0], dv[1], f, fm, mg, b0, b1);
        quant_pair_f(dv[2], dv[3], f, fm, mg, b2, b3);
        b0 = (uint32_t)min(max((int)(b0 - kMagic), 0), (int)qmax) + kMagic;
        b1 = (uint32_t)min(max((int)(b1 - kMagic), 0), (int)qmax) + kMagic;
        b2 = (uint32_t)min(max((int)(b2 - kMagic), 0), (int)qmax) + kMagic;
        b3 = (uint32_t)min(max((int)(b3 - kMagic), 0), (int)qmax) + kMagic;
        const uint32_t lo2 = __byte_perm(b0, b1, 0x0040), hi2 = __byte_perm(b2, b3, 0x0040);
        *reinterpret_cast<uint32_t *>(sym + r * kSymRow + 4 * kq) = __byte_perm(lo2, hi2, 0x5410) << SH;
        red_add(b0 * (kCntRow * 2) + cnt_lane, 1u);
        red_add(b1 * (kCntRow * 2) + cnt_lane, 1u << 16);
        red_add(b2 * (kCntRow * 2) + cnt_lane + 4, 1u);
        red_add(b3 * (kCntRow * 2) + cnt_lane + 4, 1u << 16);
    }
}

// V2 (format 2): the alphabet is the layer's 2*MAX + 1 symbols and the side
// output is the count records (uint8) instead of the CDF entries (uint16).
// DELTA: the token-locality delta [CG §1.2(1)] with groups of d.G tokens; the
// anchors' max1 comes from a pre-pass over the anchor rows (plain loads of
// kin / vin), then pass 1 takes max |x - a^| per row and step 2 quantises d.
template <bool V2, bool DELTA, int AM>
__global__ void __launch_bounds__(kNT, AM <= 32 || !DELTA ? 3 : 2) k_compress_tma(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, const uint16_t *kin,
    const uint16_t *vin, Dims d, MaxTab mt, int box_rows, uint16_t *__restrict__ max1_out,
    void *__restrict__ side_out, uint8_t *__restrict__ stage, uint32_t *__restrict__ len,
    unsigned long long *state, int32_t *status) {
    using AL = Alpha<AM>;
    // 64 symbols without the delta: the row factors sit in the symbol tile's
    // row padding and max1 in the CDF rows until the coding starts, so that
    // three CTAs fit an SM
    constexpr bool kLean = AM > 32 && !DELTA;
    constexpr int FS = kLean ? kSymRow / 4 : 1;  // float stride of the row factors
    __shared__ unsigned long long s_scan[kNW + 4];
    __shared__ unsigned long long s_bar[2];
    __shared__ uint16_t s_ftab[kNT + 2];
    __shared__ int s_ticket;
    // the delta: each row's anchor row and the table (q - MAX) / MAX (an
    // anchor row keeps its max1 in s_m1 from the pre-pass on)
    __shared__ uint8_t s_anchor[DELTA ? kNT : 1];
    __shared__ uint8_t s_aidx[DELTA ? kNT : 1];  // the delta: each row's anchor index (row / G)
    __shared__ float s_unitc[DELTA ? 64 : 1];
    extern __shared__ __align__(128) unsigned char dsm[];

    // the union: static for 32-symbol alphabets (its addresses are constants);
    // for 64 it follows the box buffer in dynamic shared memory
    unsigned char *s_union;
    if constexpr (AM <= 32) {
        __shared__ __align__(1024) unsigned char s_union_st[AL::union_bytes];
        s_union = s_union_st;
    } else {
        const uint32_t dy = smem_u32(dsm);
        s_union = dsm + (((dy + 127u) & ~127u) + (uint32_t)box_rows * (kW * 2)) - dy;
    }
    unsigned char *cdfw = s_union;
    uint16_t *cnt16 = reinterpret_cast<uint16_t *>(s_union + AL::cdfw_bytes);
    uint32_t *cnt32 = reinterpret_cast<uint32_t *>(s_union + AL::cdfw_bytes);
    uint8_t *sym = s_union + AL::cdfw_bytes + AL::cnt_bytes;
    float *s_fac;
    uint16_t *s_m1;
    if constexpr (kLean) {
        s_fac = reinterpret_cast<float *>(sym + kW);
        s_m1 = reinterpret_cast<uint16_t *>(s_union);
    } else {
        __shared__ float s_fac_st[kNT];
        __shared__ uint16_t s_m1_st[kNT];
        s_fac = s_fac_st;
        s_m1 = s_m1_st;
    }
    const uint32_t dyn = smem_u32(dsm);
    const uint32_t buf0 = (dyn + 127u) & ~127u;  // box buffer 0 (dynamic, 128-byte aligned)
    const uint32_t buf1 = smem_u32(s_union);     // box buffer 1 (max1 pass only)
    const unsigned char *box0 = dsm + (buf0 - dyn);
    const uint32_t bar0 = smem_u32(&s_bar[0]), bar1 = smem_u32(&s_bar[1]);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s_ticket = (int)atomicAdd(state, 1ull);
        mbar_init(bar0);
        mbar_init(bar1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    const int ticket = s_ticket;
    int k, kv, l;
    slice_coords(d, ticket, k, kv, l);
    const int Tk = chunk_tokens(d, k);
    const int MAX = mt.v[kv][l];
    const int A = V2 ? 2 * MAX + 1 : d.A[kv];
    const CUtensorMap *tm = kv ? &tmv : &tmk;
    const int t0 = k * d.Tc;
    const int nwin = (d.C + kW - 1) / kW;
    const uint32_t box_bytes = (uint32_t)box_rows * (kW * 2);
    // (the union is free until the first boxes are asked for)
    const long long side_base = V2 ? record_slice_offset(d, mt, k, kv, l, reinterpret_cast<unsigned long long *>(s_union))
                                   : cdf_slice_offset(d, k, kv, l);
    const long long sid0 = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk;
    const long long sid = sid0 + tid;
    uint8_t *stream = stage_stream(stage, tid < Tk ? sid : sid0, d);
    // this lane's rows (rbase + 2i) and quad (channels 4 kq .. 4 kq + 3 of a window)
    const int kq = lane & 15;
    const int rbase = 32 * warp + (lane >> 4);
    bool timed_out = false;

    if (tid == 0) {
        tma_load(buf0, tm, 0, t0, l, bar0, box_bytes);
        if (nwin > 1) tma_load(buf1, tm, kW, t0, l, bar1, box_bytes);
        for (int m = 2; m < 4 && m < nwin; m++) tma_prefetch_l2(tm, m * kW, t0, l);
    }

    const float fmax = (float)MAX;
    const unsigned long long fm = pair(fmax, fmax);
    const unsigned long long mg = pair(12582912.0f, 12582912.0f);
    const uint32_t qmax = 2u * (uint32_t)MAX;
    const uint32_t us = smem_u32(s_unitc);
    if (DELTA) {
        // 0. anchors' max1 (rows 0, G, 2G, ... of the chunk), one warp per anchor row
        const uint16_t *xb = (kv ? vin : kin) + (long long)l * d.layer_stride + (long long)t0 * d.C;
        const int na = (Tk + d.G - 1) / d.G;
        const int nv = d.C >> 3;
        for (int j = warp; j < na; j += kNW) {
            const uint4 *row = reinterpret_cast<const uint4 *>(xb + (long long)j * d.G * d.C);
            uint32_t m = 0;
            for (int c = lane; c < nv; c += 32) {
                const uint4 q = __ldg(row + c);
                m = __vmaxu2(m, q.x & 0x7FFF7FFFu);
                m = __vmaxu2(m, q.y & 0x7FFF7FFFu);
                m = __vmaxu2(m, q.z & 0x7FFF7FFFu);
                m = __vmaxu2(m, q.w & 0x7FFF7FFFu);
            }
            m = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
            if (lane == 0) s_m1[j * d.G] = (uint16_t)m;
        }
        __syncthreads();
        const int ra = tid - tid % d.G;
        s_anchor[tid] = (uint8_t)ra;
        s_aidx[tid] = (uint8_t)(tid / d.G);
        if (tid < Tk && ra == tid) {
            const unsigned mb = s_m1[tid];
            s_fac[tid] = mb ? __fdiv_rn(fmax, __half2float(__ushort_as_half((unsigned short)mb))) : 0.0f;
        }
        if (tid < 64) s_unitc[tid] = __fdiv_rn((float)(tid - MAX), fmax);
        __syncthreads();
    }

    // 1. max1 pass over the slice's boxes (buffers alternate); with the delta,
    // max |x - a^| as binary32 bits (non-negative floats order like their bits).
    // When the anchor rows' reconstructions of a box (binary32, 256 bytes per
    // anchor row) fit in the shared union beside the second box buffer (groups
    // of 10 or more for 256-token chunks), each is computed once per box and
    // read back by the rows of its group; otherwise each row recomputes its
    // anchor's quad.
    const int na = DELTA ? (Tk + d.G - 1) / d.G : 0;
    const bool ahat_shared = DELTA && na * (kW * 4) <= AL::union_bytes - (int)box_bytes;
    float4 *ahat = reinterpret_cast<float4 *>(s_union + box_bytes);
    uint32_t ph0 = 0, ph1 = 0;
    uint32_t mx[16];
#pragma unroll
    for (int i = 0; i < 16; i++) mx[i] = 0;
    for (int m = 0; m < nwin; m++) {
        const bool odd = (m & 1) != 0;
        if (!mbar_wait(odd ? bar1 : bar0, odd ? ph1 : ph0)) timed_out = true;
        if (odd)
            ph1 ^= 1u;
        else
            ph0 ^= 1u;
        const unsigned char *box = odd ? s_union : box0;
        if (DELTA && ahat_shared) {
            for (int idx = tid; idx < na * 16; idx += kNT) {
                const int ra = (idx >> 4) * d.G, q = idx & 15;
                const uint2 xa = *reinterpret_cast<const uint2 *>(box + ra * (kW * 2) + 8 * q);
                const float fa = s_fac[ra], ma = __half2float(__ushort_as_half(s_m1[ra]));
                uint32_t c0, c1, c2, c3;
                quant_pair(xa.x, fa, fm, mg, c0, c1);
                quant_pair(xa.y, fa, fm, mg, c2, c3);
                ahat[idx] = make_float4(__fmul_rn(lds_f32(us + 4u * min(c0 - kMagic, qmax)), ma),
                                        __fmul_rn(lds_f32(us + 4u * min(c1 - kMagic, qmax)), ma),
                                        __fmul_rn(lds_f32(us + 4u * min(c2 - kMagic, qmax)), ma),
                                        __fmul_rn(lds_f32(us + 4u * min(c3 - kMagic, qmax)), ma));
            }
            __syncthreads();  // the box's anchor reconstructions are in
#pragma unroll
            for (int i = 0; i < 16; i++) {
                const int r = rbase + 2 * i;
                if (r < Tk) {
                    const uint2 x = *reinterpret_cast<const uint2 *>(box + r * (kW * 2) + 8 * kq);
                    // an anchor is its own zero reference: |x - (+-0)| = |x|
                    const float4 a4 = s_anchor[r] == r ? make_float4(0.f, 0.f, 0.f, 0.f) : ahat[16 * s_aidx[r] + kq];
                    const float2 x01 = __half22float2(*reinterpret_cast<const __half2 *>(&x.x));
                    const float2 x23 = __half22float2(*reinterpret_cast<const __half2 *>(&x.y));
                    const uint32_t m01 = max(__float_as_uint(__fsub_rn(x01.x, a4.x)) & 0x7FFFFFFFu,
                                             __float_as_uint(__fsub_rn(x01.y, a4.y)) & 0x7FFFFFFFu);
                    const uint32_t m23 = max(__float_as_uint(__fsub_rn(x23.x, a4.z)) & 0x7FFFFFFFu,
                                             __float_as_uint(__fsub_rn(x23.y, a4.w)) & 0x7FFFFFFFu);
                    mx[i] = max(mx[i], max(m01, m23));
                }
            }
        } else {
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const int r = rbase + 2 * i;
            if (r < Tk) {
                const uint2 x = *reinterpret_cast<const uint2 *>(box + r * (kW * 2) + 8 * kq);
                if (DELTA) {
                    const int ra = s_anchor[r];
                    const uint2 xa = *reinterpret_cast<const uint2 *>(box + ra * (kW * 2) + 8 * kq);
                    float dv[4];
                    delta_quad(x, xa, s_fac[ra], anchor_m1(s_m1, ra, r), us, qmax, fm, mg, dv);
                    const uint32_t m01 = max(__float_as_uint(dv[0]) & 0x7FFFFFFFu, __float_as_uint(dv[1]) & 0x7FFFFFFFu);
                    const uint32_t m23 = max(__float_as_uint(dv[2]) & 0x7FFFFFFFu, __float_as_uint(dv[3]) & 0x7FFFFFFFu);
                    mx[i] = max(mx[i], max(m01, m23));
                } else {
                    mx[i] = __vmaxu2(mx[i], x.x & 0x7FFF7FFFu);
                    mx[i] = __vmaxu2(mx[i], x.y & 0x7FFF7FFFu);
                }
            }
        }
        }
        __syncthreads();  // the buffer is free again
        if (tid == 0) {
            if (m + 4 < nwin) tma_prefetch_l2(tm, (m + 4) * kW, t0, l);
            if (m + 2 < nwin)
                tma_load(odd ? buf1 : buf0, tm, (m + 2) * kW, t0, l, odd ? bar1 : bar0, box_bytes);
            else if (!odd)
                tma_load(buf0, tm, 0, t0, l, bar0, box_bytes);  // first window of the coding loop
        }
    }
    bool nonfinite = false;
    {
        uint32_t mine = 0;
#pragma unroll
        for (int i = 0; i < 16; i++) {
            uint32_t v = DELTA ? mx[i] : max(mx[i] & 0xFFFFu, mx[i] >> 16);
            v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
            v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
            v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
            v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 8));
            if (kq == i) mine = v;
        }
        const int r = rbase + 2 * kq;
        if (r < Tk) {
            // the delta: max1 = max |d| rounded up to binary16 (an anchor's d is
            // x itself, so its max1 is the plain one)
            const uint32_t mh = DELTA ? half_up_bits(__uint_as_float(mine)) : mine;
            s_m1[r] = (uint16_t)mh;
            max1_out[group_index(d, kv, l, t0 + r)] = (uint16_t)mh;
            nonfinite = DELTA ? mine >= 0x7F800000u : mine >= 0x7C00u;
        }
    }
    for (int n = tid; n <= Tk; n += kNT)
        s_ftab[n] = (uint16_t)(1u + ((uint32_t)n * (kTotal - (uint32_t)A)) / (uint32_t)Tk);
    for (int i = tid; i < AL::cnt_bytes / 4; i += kNT) cnt32[i] = 0;
    nonfinite = __syncthreads_or(nonfinite) != 0;
    if (tid < Tk) {
        const unsigned mb = s_m1[tid];
        s_fac[tid * FS] = mb ? __fdiv_rn(fmax, __half2float(__ushort_as_half((unsigned short)mb))) : 0.0f;
    }
    __syncthreads();

    // counter byte address of (q, channel 4 kq) is cnt_lane + 132 * (kMagic + q)
    const uint32_t cnt_lane = smem_u32(cnt32) + 8u * (uint32_t)kq - (uint32_t)(kCntRow * 2) * kMagic;
    Enc e;
    enc_init(e);
    for (int w = 0; w < nwin; w++) {
        const int c0 = w * kW;
        const int Wc = min(kW, d.C - c0);  // a multiple of 8
        if (!mbar_wait(bar0, ph0)) timed_out = true;
        ph0 ^= 1u;
        __syncwarp();  // this warp's coding of the previous window has read its symbol rows
        // 2. quantise + count
        if (4 * kq < Wc) {
            // a box that did not arrive in time holds stale values: clamp those too
            if (DELTA)
                quantise_window_delta<AL::SH>(box0, s_fac, s_anchor, s_m1, us, sym, cnt_lane, rbase, kq, Tk, fm, mg,
                                              qmax);
            else if (nonfinite || timed_out)
                quantise_window<true, AL::SH, FS>(box0, s_fac, sym, cnt_lane, rbase, kq, Tk, fm, mg, qmax);
            else
                quantise_window<false, AL::SH, FS>(box0, s_fac, sym, cnt_lane, rbase, kq, Tk, fm, mg, qmax);
        }
        __syncthreads();
        if (tid == 0 && w + 1 < nwin) tma_load(buf0, tm, c0 + kW, t0, l, bar0, box_bytes);
        // 3. CDF rows: thread (channel c, part p) owns symbols 8p .. 8p + 7
        build_cdf_window<V2, 1, AM>(tid, cnt16, s_ftab, cdfw, side_out, side_base, c0, Wc, A);
        __syncthreads();
        // 4. code my token's symbols of this window
        if (tid < Tk) encode_window<AM>(e, stream, sym + tid * kSymRow, cdfw, Wc);
    }

    // 5. stream lengths and the slice's total (offsets and packing follow in
    // k_pack, so no slice here waits on another)
    const uint32_t mylen = tid < Tk ? enc_finish(e, stream) : 0u;
    if (tid < Tk) len[sid] = mylen;
    uint32_t tot = mylen;  // a slice holds at most 256 * (2C + 8) bytes
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
    if (lane == 0) s_scan[warp] = tot;
    __syncthreads();
    if (tid == 0) {
        unsigned long long run = 0;
#pragma unroll
        for (int w = 0; w < kNW; w++) run += s_scan[w];
        state[2 + 2LL * d.L * d.nch + ticket] = run;
    }
    if (status && (nonfinite || timed_out) && (tid == 0 || timed_out))
        atomicOr(status, (nonfinite ? CG_FLAG_NONFINITE : 0) | (timed_out ? CG_FLAG_TIMEOUT : 0));
}

// Latency mode: launches of at most one slice per SM (a single chunk, say),
// where each slice's CTA has an SM to itself and the coders' time is set by the
// serial chain of each token stream, not by instruction issue. A CTA splits the
// work by warp: the first 256 / NC threads only code (thread t codes token
// R0 + t), the next 256 quantise and count window i + 1 and turn its counts into
// CDF rows while the coders code window i, so the coders never wait on those
// steps. The symbol tile and the CDF rows are double-buffered; one named
// barrier of all threads per window hands a window over (producers have
// finished window i, coders have finished window i - 1). The max1 pass uses all
// warps; the fp16 boxes come by TMA into two buffers, window i + 2's box
// loading while window i + 1 is quantised.
// NC = 2 (at most one slice per two SMs): a cluster of two CTAs shares a slice,
// CTA rank r taking rows [r h, r h + h), h = ceil(Tc_k / 2), so each SM codes
// half the streams and quantises half the rows. Each CTA counts its rows into
// one of two counter tables (alternating per window); its producers then tell
// the peer's producers (a remote arrive on the peer's mbarrier, release at
// cluster scope) and wait for the peer's word before both build the same CDF
// rows from both tables (the peer's through distributed shared memory). A
// CTA clears a table only after the peer has announced the next window's
// counts, by which time the peer has read it. Rank 0 writes the side output
// and the slice's byte total.
template <int NC>
struct LmSmem {
    static constexpr int rows = kNT / NC;
    static constexpr int sym_bytes = rows * kSymRow;
    static constexpr int cdfw = 0;
    static constexpr int cnt = cdfw + 2 * kCdfwBytes;
    static constexpr int sym = cnt + NC * kCntBytes;
    static constexpr int box = (sym + 2 * sym_bytes + 127) & ~127;
    static int bytes(int box_bytes) { return 128 + box + 2 * box_bytes; }
};

template <bool V2, int NC>
__global__ void __launch_bounds__(kNT / NC + kNT, 1) k_compress_lm(
    const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv, Dims d, MaxTab mt,
    int box_rows, uint16_t *__restrict__ max1_out, void *__restrict__ side_out, uint8_t *__restrict__ stage,
    uint32_t *__restrict__ len, unsigned long long *state, int32_t *status) {
    using S = LmSmem<NC>;
    constexpr int NCOD = kNT / NC;   // coder threads
    constexpr int NCW = NCOD / 32;   // coder warps
    constexpr int NTH = NCOD + kNT;  // threads
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ unsigned long long s_bar[4];  // box buffers 0 and 1; the peer's word on even / odd windows
    __shared__ unsigned long long s_scan[NCW + 1];
    __shared__ float s_fac[NCOD];
    __shared__ uint16_t s_m1[NCOD];
    __shared__ uint16_t s_ftab[kNT + 2];

    // the packing launch (programmatic dependent launch) may start placing its
    // CTAs now; they wait in griddepcontrol.wait until this grid has finished
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const uint32_t dyn = smem_u32(dsm);
    const uint32_t base = (dyn + 127u) & ~127u;
    unsigned char *sm = dsm + (base - dyn);
    uint2 *cdfw2 = reinterpret_cast<uint2 *>(sm + S::cdfw);
    uint16_t *cnt16 = reinterpret_cast<uint16_t *>(sm + S::cnt);
    uint32_t *cnt32 = reinterpret_cast<uint32_t *>(sm + S::cnt);
    uint8_t *sym2 = sm + S::sym;
    const uint32_t buf0 = base + S::box, buf1 = buf0 + (uint32_t)box_rows * (kW * 2);
    const uint32_t bar0 = smem_u32(&s_bar[0]), bar1 = smem_u32(&s_bar[1]);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = NC == 2 ? cluster_rank() : 0u;
    const int slice = blockIdx.x / NC;
    int k, kv, l;
    slice_coords(d, slice, k, kv, l);
    const int Tk = chunk_tokens(d, k);
    const int h = (Tk + NC - 1) / NC;
    const int R0 = (int)rank * h;
    const int nr = min(h, Tk - R0);  // this CTA's rows of the slice: [R0, R0 + nr)
    const int MAX = mt.v[kv][l];
    const int A = V2 ? 2 * MAX + 1 : d.A[kv];
    const CUtensorMap *tm = kv ? &tmv : &tmk;
    const int t0 = k * d.Tc;
    const int ty = t0 + R0;  // first row of this CTA's boxes
    const int nwin = (d.C + kW - 1) / kW;
    const uint32_t box_bytes = (uint32_t)box_rows * (kW * 2);
    const long long side_base = V2 ? record_slice_offset(d, mt, k, kv, l) : cdf_slice_offset(d, k, kv, l);
    const long long sid0 = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk + R0;
    bool timed_out = false;
    if (tid == 0) {
        mbar_init(bar0);
        mbar_init(bar1);
        mbar_init(smem_u32(&s_bar[2]));
        mbar_init(smem_u32(&s_bar[3]));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // the max1 pass reads window m from buffer m & 1; the coding pass reads
        // window i from buffer (nwin + i) & 1 (with one window, buffer 1 holds it)
        tma_load(buf0, tm, 0, ty, l, bar0, box_bytes);
        tma_load(buf1, tm, nwin > 1 ? kW : 0, ty, l, bar1, box_bytes);
    }
    if (NC == 2)
        cluster_sync();  // both CTAs' mbarriers exist before either arrives on the other's
    else
        __syncthreads();

    // 1. max1 pass, all warps: lane (quad kq) of warp w keeps rows 16 w + (lane >> 4) + 2 i
    const int kq = lane & 15;
    uint32_t ph0 = 0u, ph1 = 0u;
    {
        const int rb = 16 * warp + (lane >> 4);
        uint32_t mx[8];
#pragma unroll
        for (int i = 0; i < 8; i++) mx[i] = 0;
        for (int m = 0; m < nwin; m++) {
            const bool b = (m & 1) != 0;
            if (!mbar_wait(b ? bar1 : bar0, b ? ph1 : ph0)) timed_out = true;
            if (b)
                ph1 ^= 1u;
            else
                ph0 ^= 1u;
            const unsigned char *box = sm + ((b ? buf1 : buf0) - base);
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const int r = rb + 2 * i;
                if (r < nr) {
                    const uint2 x = *reinterpret_cast<const uint2 *>(box + r * (kW * 2) + 8 * kq);
                    mx[i] = __vmaxu2(mx[i], x.x & 0x7FFF7FFFu);
                    mx[i] = __vmaxu2(mx[i], x.y & 0x7FFF7FFFu);
                }
            }
            __syncthreads();  // the buffer is free again
            if (tid == 0) {
                const int j = m + 2 < nwin ? m + 2 : m + 2 - nwin;  // the coding pass starts over at 0 and 1
                if (m + 2 < nwin || (j < 2 && j < nwin))
                    tma_load(b ? buf1 : buf0, tm, j * kW, ty, l, b ? bar1 : bar0, box_bytes);
            }
        }
        uint32_t mine = 0;
#pragma unroll
        for (int i = 0; i < 8; i++) {
            uint32_t v = max(mx[i] & 0xFFFFu, mx[i] >> 16);
            v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 1));
            v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 2));
            v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 4));
            v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, 8));
            if (kq == i) mine = v;
        }
        bool nonfinite = false;
        const int r = rb + 2 * kq;
        if (kq < 8 && r < nr) {
            s_m1[r] = (uint16_t)mine;
            max1_out[group_index(d, kv, l, ty + r)] = (uint16_t)mine;
            nonfinite = mine >= 0x7C00u;
        }
        for (int n = tid; n <= Tk; n += NTH)
            s_ftab[n] = (uint16_t)(1u + ((uint32_t)n * (kTotal - (uint32_t)A)) / (uint32_t)Tk);
        for (int i = tid; i < NC * kCntBytes / 4; i += NTH) cnt32[i] = 0;
        nonfinite = __syncthreads_or(nonfinite) != 0;
        if (tid < nr) {
            const unsigned mb = s_m1[tid];
            s_fac[tid] = mb ? __fdiv_rn((float)MAX, __half2float(__ushort_as_half((unsigned short)mb))) : 0.0f;
        }
        timed_out = __syncthreads_or(timed_out) != 0;
        if (tid == 0 && status && (nonfinite || timed_out))
            atomicOr(status, (nonfinite ? CG_FLAG_NONFINITE : 0) | (timed_out ? CG_FLAG_TIMEOUT : 0));
        timed_out = timed_out || nonfinite;  // either takes the clamping quantiser
    }
    const bool safe = timed_out;

    if (warp >= NCW) {
        // producers: window i's symbols, counts and CDF rows into buffers i & 1
        const int pt = tid - NCOD;
        const int pw = warp - NCW;
        const int rbase = 32 * pw + (lane >> 4);
        const unsigned long long fm = pair((float)MAX, (float)MAX);
        const unsigned long long mg = pair(12582912.0f, 12582912.0f);
        const uint32_t qmax = 2u * (uint32_t)MAX;
        const uint32_t cnt_lane = smem_u32(cnt32) + 8u * (uint32_t)kq - (uint32_t)(kCntRow * 2) * kMagic;
        // the peer's word for window i arrives on s_bar[2 + (i & 1)], phase i >> 1:
        // it cannot run a phase ahead, as its word for window i + 2 needs this
        // CTA's word for window i + 1, sent after this wait
        const uint32_t xb0 = smem_u32(&s_bar[2]), xb1 = smem_u32(&s_bar[3]);
        const uint32_t xp0 = NC == 2 ? peer_addr(xb0, rank ^ 1u) : 0u, xp1 = NC == 2 ? peer_addr(xb1, rank ^ 1u) : 0u;
        bool late = false;
        for (int i = 0; i < nwin; i++) {
            const int c0 = i * kW;
            const int Wc = min(kW, d.C - c0);
            const int tb = NC == 2 ? (i & 1) * (kCntBytes / 2) : 0;  // this window's counter table (elements)
            const bool b = ((nwin + i) & 1) != 0;  // box buffer of window i in the coding pass
            if (!mbar_wait(b ? bar1 : bar0, b ? ph1 : ph0)) late = true;
            if (b)
                ph1 ^= 1u;
            else
                ph0 ^= 1u;
            uint8_t *sym = sym2 + (i & 1) * S::sym_bytes;
            const unsigned char *box = sm + ((b ? buf1 : buf0) - base);
            if (4 * kq < Wc) {
                if (safe || late)
                    quantise_window<true>(box, s_fac, sym, cnt_lane + 2u * tb, rbase, kq, nr, fm, mg, qmax);
                else
                    quantise_window<false>(box, s_fac, sym, cnt_lane + 2u * tb, rbase, kq, nr, fm, mg, qmax);
            }
            asm volatile("bar.sync 1, %0;" ::"n"(kNT) : "memory");  // counts in, box read
            if (pt == 0 && i + 2 < nwin) tma_load(b ? buf1 : buf0, tm, (i + 2) * kW, ty, l, b ? bar1 : bar0, box_bytes);
            if constexpr (NC == 2) {
                const bool odd = (i & 1) != 0;
                if (pt == 0) mbar_arrive_remote(odd ? xp1 : xp0);  // this CTA's counts of window i are in
                if (!mbar_wait_cluster(odd ? xb1 : xb0, (uint32_t)(i >> 1) & 1u)) late = true;  // and the peer's
            }
            build_cdf_window<V2, NC>(pt, cnt16, s_ftab, cdfw2 + (i & 1) * (kCdfwBytes / 8), side_out, side_base, c0,
                                     Wc, A, tb, rank);
            asm volatile("bar.sync 2, %0;" ::"n"(NTH) : "memory");  // window i handed over
        }
        if (late && lane == 0 && status) atomicOr(status, CG_FLAG_TIMEOUT);
    } else {
        // coders: window i from buffers i & 1
        Enc e;
        enc_init(e);
        uint8_t *stream = stage_stream(stage, sid0 + (tid < nr ? tid : 0), d);
        asm volatile("bar.sync 2, %0;" ::"n"(NTH) : "memory");  // window 0 is ready
        for (int i = 0; i < nwin; i++) {
            const int Wc = min(kW, d.C - i * kW);
            if (tid < nr)
                encode_window<kAmax, true>(e, stream, sym2 + (i & 1) * S::sym_bytes + tid * kSymRow,
                              cdfw2 + (i & 1) * (kCdfwBytes / 8), Wc);
            if (i + 1 < nwin) asm volatile("bar.sync 2, %0;" ::"n"(NTH) : "memory");
        }
        const uint32_t mylen = tid < nr ? enc_finish(e, stream) : 0u;
        if (tid < nr) len[sid0 + tid] = mylen;
        uint32_t tot = mylen;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, o);
        if (lane == 0) s_scan[warp] = tot;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned long long run = 0;
#pragma unroll
        for (int w = 0; w < NCW; w++) run += s_scan[w];
        s_scan[NCW] = run;
        if (NC == 1) state[2 + 2LL * d.L * d.nch + slice] = run;
    }
    if constexpr (NC == 2) {
        cluster_sync();  // both CTAs' totals are in
        if (rank == 0 && tid == 0)
            state[2 + 2LL * d.L * d.nch + slice] = s_scan[NCW] + ld_peer_u64(peer_addr(smem_u32(&s_scan[NCW]), 1u));
        cluster_sync();  // the peer's shared memory is read before either CTA exits
    }
}

// Copy one staged stream (n bytes; this lane's first word already loaded)
// to byte position dst of the packed buffer, a warp per stream, lane i taking
// the words i, i + 32, ... For streams past 128 bytes a full word goes out as
// one, two or three stores by the destination's alignment (the same for
// every word of the stream); the last word, and every word of shorter streams,
// byte by byte.
__device__ __forceinline__ void copy_stream(const uint8_t *src, uint32_t n, unsigned long long dst, uint8_t *packed,
                                            unsigned long long capacity, uint32_t first, int lane) {
    if (n > 128u) {
        const uint32_t al = (uint32_t)((reinterpret_cast<uintptr_t>(packed) + dst) & 3u);
        for (uint32_t b = 4u * lane; b < n; b += 128u) {
            const uint32_t wv = b < 128u ? first : *reinterpret_cast<const uint32_t *>(src + b);
            const unsigned long long pos = dst + b;
            if (b + 4u <= n && pos + 4u <= capacity) {
                uint8_t *pp = packed + pos;
                if (al == 0) {
                    *reinterpret_cast<uint32_t *>(pp) = wv;
                } else if (al == 2) {
                    reinterpret_cast<uint16_t *>(pp)[0] = (uint16_t)wv;
                    reinterpret_cast<uint16_t *>(pp)[1] = (uint16_t)(wv >> 16);
                } else {
                    pp[0] = (uint8_t)wv;
                    *reinterpret_cast<uint16_t *>(pp + 1) = (uint16_t)(wv >> 8);
                    pp[3] = (uint8_t)(wv >> 24);
                }
            } else {
                const uint32_t nb = min(4u, n - b);
#pragma unroll
                for (uint32_t q = 0; q < 4; q++)
                    if (q < nb && pos + q < capacity) packed[pos + q] = (uint8_t)(wv >> (8 * q));
            }
        }
    } else {
        // one word per lane at most; a stream inside the capacity (every
        // stream of a buffer large enough) needs no per-byte check against it
        const uint32_t b = 4u * lane;
        if (b < n) {
            if (dst + n <= capacity) {
                uint8_t *pp = packed + dst + b;
                pp[0] = (uint8_t)first;
                if (b + 1u < n) pp[1] = (uint8_t)(first >> 8);
                if (b + 2u < n) pp[2] = (uint8_t)(first >> 16);
                if (b + 3u < n) pp[3] = (uint8_t)(first >> 24);
            } else {
                const uint32_t nb = min(4u, n - b);
#pragma unroll
                for (uint32_t q = 0; q < 4; q++) {
                    const unsigned long long pos = dst + b + q;
                    if (q < nb && pos < capacity) packed[pos] = (uint8_t)(first >> (8 * q));
                }
            }
        }
    }
}

// Offsets and packing: CTA per slice in stream order (by ticket). Every
// slice's byte total is known when this kernel starts, so each CTA publishes
// its aggregate at once and its decoupled look-back (32 predecessors per step,
// bounded spins) never waits on slow work. Then a block scan of the lengths
// gives each stream's offset, and warps copy the streams from the staging
// area into place, clipped at the capacity; lane i takes word i of a stream,
// eight streams per batch of loads.
__global__ void __launch_bounds__(kNT) k_pack(Dims d, const uint8_t *__restrict__ stage,
                                              const uint32_t *__restrict__ len, uint64_t *__restrict__ off,
                                              uint8_t *__restrict__ packed, unsigned long long capacity,
                                              unsigned long long *state, int32_t *status) {
    __shared__ unsigned long long s_scan[kNW + 1];
    __shared__ uint32_t s_len[kNT], s_loc[kNT];
    __shared__ int s_ticket;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long nslices = 2LL * d.L * d.nch;
    if (tid == 0) {
        // take the next slice and publish its total at once
        const long long t = (long long)atomicAdd(state + 1, 1ull);
        s_ticket = (int)t;
        st_release(state + 2 + t, (t == 0 ? (2ull << 62) : kFlagAggregate) | state[2 + nslices + t]);
    }
    __syncthreads();
    const int ticket = s_ticket;
    int k, kv, l;
    slice_coords(d, ticket, k, kv, l);
    const int Tk = chunk_tokens(d, k);
    const long long sid0 = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk;
    bool timed_out = false;
    // offsets inside the slice
    const uint32_t mylen = tid < Tk ? len[sid0 + tid] : 0u;
    uint32_t incl = mylen;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s_scan[warp] = incl;
    s_len[tid] = mylen;
    __syncthreads();
    uint32_t wbase = 0;
#pragma unroll
    for (int w = 0; w < kNW; w++) wbase += w < warp ? (uint32_t)s_scan[w] : 0u;
    s_loc[tid] = wbase + incl - mylen;
    if (warp == 0) {
        const unsigned long long run = state[2 + nslices + ticket];
        unsigned long long *mine = state + 2 + ticket;
        unsigned long long base = 0;
        for (long long j = ticket - 1; j >= 0; j -= 32) {
            const long long idx = j - lane;
            unsigned long long v = idx >= 0 ? ld_acquire(state + 2 + idx) : (2ull << 62);
            for (int spins = 0; __any_sync(0xFFFFFFFFu, (v >> 62) == 0) && spins < kSpinLimit; spins++) {
                if ((v >> 62) == 0) {
                    __nanosleep(32);
                    v = ld_acquire(state + 2 + idx);
                }
            }
            if (__any_sync(0xFFFFFFFFu, (v >> 62) == 0)) {
                timed_out = true;
                break;
            }
            const unsigned pm = __ballot_sync(0xFFFFFFFFu, (v >> 62) == 2);
            const int first = pm ? __ffs(pm) - 1 : 31;
            unsigned long long x = lane <= first ? (v & kValueMask) : 0ull;
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
            base += x;
            if (pm) break;
        }
        if (lane == 0) {
            if (ticket > 0) st_release(mine, (2ull << 62) | ((base + run) & kValueMask));
            s_scan[kNW] = base;
            if (ticket == nslices - 1) {
                off[d.nstreams] = base + run;
                if (base + run > capacity && status) atomicOr(status, CG_FLAG_CAPACITY);
            }
        }
    }
    // the first batch of stage words is read while warp 0 looks back
    constexpr int kBatch = 8;
    uint32_t held[kBatch];
    auto load_batch = [&](int b0) {
#pragma unroll
        for (int u = 0; u < kBatch; u++) {
            const int t = warp + kNW * (b0 + u);
            held[u] = 0;
            if (t < Tk && 4u * lane < s_len[t])
                held[u] = *reinterpret_cast<const uint32_t *>(stage_stream(const_cast<uint8_t *>(stage), sid0 + t, d) +
                                                              4 * lane);
        }
    };
    load_batch(0);
    __syncthreads();
    const unsigned long long sbase = s_scan[kNW];
    if (tid < Tk) off[sid0 + tid] = sbase + s_loc[tid];
    const int nper = (Tk + kNW - 1) / kNW;  // streams per warp
    for (int b0 = 0; b0 < nper; b0 += kBatch) {
        if (b0 > 0) load_batch(b0);
#pragma unroll
        for (int u = 0; u < kBatch; u++) {
            const int t = warp + kNW * (b0 + u);
            if (t >= Tk) continue;
            const uint32_t n = s_len[t];
            const unsigned long long dst = sbase + s_loc[t];
            const uint8_t *src = stage_stream(const_cast<uint8_t *>(stage), sid0 + t, d);
            copy_stream(src, n, dst, packed, capacity, held[u], lane);
        }
    }
    if (timed_out && status && lane == 0) atomicOr(status, CG_FLAG_TIMEOUT);
}

// Packing after the latency-mode kernel (at most one slice per SM): four
// CTAs per slice, each placing a quarter of its streams. A slice's offset is
// the sum of the byte totals of the slices before it, read directly (at most
// one slice per SM precedes it): no look-back and no wait on another CTA.
constexpr int kPackParts = 4;

__global__ void __launch_bounds__(kNT, 4) k_pack_lm(Dims d, const uint8_t *__restrict__ stage,
                                                 const uint32_t *__restrict__ len, uint64_t *__restrict__ off,
                                                 uint8_t *__restrict__ packed, unsigned long long capacity,
                                                 const unsigned long long *__restrict__ totals, int32_t *status) {
    __shared__ unsigned long long s_red[kNW];
    __shared__ uint32_t s_len[kNT], s_loc[kNT], s_wtot[kNW];
    // launched as a programmatic dependent of the compress kernel: wait until
    // that grid has finished and its writes are visible (a no-op otherwise)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slice = blockIdx.x / kPackParts, part = blockIdx.x % kPackParts;
    const long long nslices = 2LL * d.L * d.nch;
    int k, kv, l;
    slice_coords(d, slice, k, kv, l);
    const int Tk = chunk_tokens(d, k);
    const long long sid0 = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk;
    // the slice's offset and the places of its streams
    unsigned long long b = 0;
    for (int j = tid; j < slice; j += kNT) b += totals[j];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) b += __shfl_xor_sync(0xFFFFFFFFu, b, o);
    const uint32_t mylen = tid < Tk ? len[sid0 + tid] : 0u;
    uint32_t incl = mylen;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 0) s_red[warp] = b;
    if (lane == 31) s_wtot[warp] = incl;
    s_len[tid] = mylen;
    __syncthreads();
    unsigned long long sbase = 0;
    uint32_t wbase = 0;
#pragma unroll
    for (int w = 0; w < kNW; w++) {
        sbase += s_red[w];
        wbase += w < warp ? s_wtot[w] : 0u;
    }
    s_loc[tid] = wbase + incl - mylen;
    __syncthreads();
    const int q0 = (int)((long long)Tk * part / kPackParts), q1 = (int)((long long)Tk * (part + 1) / kPackParts);
    if (tid >= q0 && tid < q1) off[sid0 + tid] = sbase + s_loc[tid];
    if (slice == nslices - 1 && part == kPackParts - 1 && tid == 0) {
        unsigned long long run = 0;
#pragma unroll
        for (int w = 0; w < kNW; w++) run += s_wtot[w];
        off[d.nstreams] = sbase + run;
        if (sbase + run > capacity && status) atomicOr(status, CG_FLAG_CAPACITY);
    }
    // warps take this part's streams in turn, lane i word i; all first words in flight at once
    constexpr int kBatch = 8;
    for (int t0 = q0; t0 < q1; t0 += kNW * kBatch) {
        uint32_t held[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; u++) {
            const int t = t0 + warp + kNW * u;
            held[u] = 0;
            if (t < q1 && 4u * lane < s_len[t])
                held[u] = *reinterpret_cast<const uint32_t *>(stage_stream(const_cast<uint8_t *>(stage), sid0 + t, d) +
                                                              4 * lane);
        }
#pragma unroll
        for (int u = 0; u < kBatch; u++) {
            const int t = t0 + warp + kNW * u;
            if (t >= q1) continue;
            const uint32_t n = s_len[t];
            const unsigned long long dst = sbase + s_loc[t];
            const uint8_t *src = stage_stream(const_cast<uint8_t *>(stage), sid0 + t, d);
            copy_stream(src, n, dst, packed, capacity, held[u], lane);
        }
    }
}

// cuTensorMapEncodeTiled, fetched once from the driver through the runtime.
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// [L][T][C] fp16 with the given layer stride, boxes of [box_rows][kW].
bool make_map(CUtensorMap *map, const uint16_t *base, const Dims &d, int box_rows) {
    EncodeTiled fn = encode_tiled();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d.C, (cuuint64_t)d.T, (cuuint64_t)d.L};
    const cuuint64_t strides[2] = {(cuuint64_t)d.C * 2, (cuuint64_t)d.layer_stride * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kW, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool compress_fused_applies(const Dims &d, const uint16_t *k, const uint16_t *v) {
    const int tmax = d.Tc < d.T ? d.Tc : d.T;
    const int A = d.A[0] > d.A[1] ? d.A[0] : d.A[1];
    const bool aligned = ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0 &&
                         d.layer_stride % 8 == 0;
    return d.T > 0 && tmax <= kNT && A <= 64 && d.C % 8 == 0 && aligned;
}

cudaError_t launch_compress_fused(const uint16_t *k, const uint16_t *v, const Dims &d, const MaxTab &mt,
                                  uint16_t *max1, uint16_t *cdf, uint8_t *rec, uint8_t *stage, uint32_t *len,
                                  uint64_t *off, uint8_t *packed, uint64_t capacity,
                                  unsigned long long *state, int32_t *status, cudaStream_t s) {
    const int box_rows = d.Tc < d.T ? d.Tc : d.T;
    CUtensorMap tmk, tmv;
    if (!make_map(&tmk, k, d, box_rows) || !make_map(&tmv, v, d, box_rows)) return cudaErrorNotSupported;
    const bool v2 = cdf == nullptr;
    void *side = v2 ? static_cast<void *>(rec) : static_cast<void *>(cdf);
    const long long nslices = 2LL * d.L * d.nch;
    cudaError_t err;
    const int sms = device_sm_count();
    // the largest alphabet the kernel codes: the tensors' (format 1) or the
    // largest layer alphabet 2 MAX + 1 (format 2)
    int amax = d.A[0] > d.A[1] ? d.A[0] : d.A[1];
    if (v2) {
        amax = 0;
        for (int kv = 0; kv < 2; kv++)
            for (int l = 0; l < d.L; l++) amax = 2 * mt.v[kv][l] + 1 > amax ? 2 * mt.v[kv][l] + 1 : amax;
    }
    if (d.G == 1 && sms > 0 && nslices <= sms && amax <= 32) {
        // latency mode: coders and producers per slice, one slice per SM (or a
        // cluster of two CTAs per slice, one slice per two SMs); the slice
        // totals go to state[2 + nslices ..], which the packing reads directly
        // (no tickets, no look-back)
        const int tmax = d.Tc < d.T ? d.Tc : d.T;
        if (2 * nslices <= sms && tmax >= 2) {
            const int rows = (tmax + 1) / 2;
            CUtensorMap hk, hv;
            if (!make_map(&hk, k, d, rows) || !make_map(&hv, v, d, rows)) return cudaErrorNotSupported;
            const int dyn = LmSmem<2>::bytes(rows * kW * 2);
            auto kern = v2 ? k_compress_lm<true, 2> : k_compress_lm<false, 2>;
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
            if (err != cudaSuccess) return err;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3((unsigned)(2 * nslices));
            cfg.blockDim = dim3(kNT / 2 + kNT);
            cfg.dynamicSmemBytes = (size_t)dyn;
            cfg.stream = s;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            err = cudaLaunchKernelEx(&cfg, kern, hk, hv, d, mt, rows, max1, side, stage, len, state, status);
            if (err != cudaSuccess) return err;
        } else {
            const int dyn = LmSmem<1>::bytes(box_rows * kW * 2);
            auto kern = v2 ? k_compress_lm<true, 1> : k_compress_lm<false, 1>;
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
            if (err != cudaSuccess) return err;
            kern<<<(unsigned)nslices, 2 * kNT, dyn, s>>>(tmk, tmv, d, mt, box_rows, max1, side, stage, len, state,
                                                       status);
        }
        // the packing as a programmatic dependent launch: its CTAs are placed
        // while the compress grid runs and start as soon as it has finished
        cudaLaunchConfig_t pcfg = {};
        pcfg.gridDim = dim3((unsigned)(kPackParts * nslices));
        pcfg.blockDim = dim3(kNT);
        pcfg.dynamicSmemBytes = 0;
        pcfg.stream = s;
        cudaLaunchAttribute pattr[1];
        pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        pattr[0].val.programmaticStreamSerializationAllowed = 1;
        pcfg.attrs = pattr;
        pcfg.numAttrs = 1;
        const unsigned long long *totals = state + 2 + nslices;
        err = cudaLaunchKernelEx(&pcfg, k_pack_lm, d, static_cast<const uint8_t *>(stage),
                                 static_cast<const uint32_t *>(len), off, packed, (unsigned long long)capacity, totals,
                                 status);
        if (err != cudaSuccess) return err;
        return cudaGetLastError();
    }
    k_compress_init<<<(unsigned)((nslices + 2 + 255) / 256), 256, 0, s>>>(state, nslices);
    {
        // AM = 64: the union follows the box buffer
        const int dyn = amax <= 32 ? 128 + box_rows * kW * 2
                                   : 128 + box_rows * kW * 2 + Alpha<64>::union_bytes;
        using Kern = void (*)(const CUtensorMap, const CUtensorMap, const uint16_t *, const uint16_t *, Dims, MaxTab,
                              int, uint16_t *, void *, uint8_t *, uint32_t *, unsigned long long *, int32_t *);
        Kern kern;
        if (amax <= 32)
            kern = d.G > 1 ? (v2 ? k_compress_tma<true, true, 32> : k_compress_tma<false, true, 32>)
                           : (v2 ? k_compress_tma<true, false, 32> : k_compress_tma<false, false, 32>);
        else
            kern = d.G > 1 ? (v2 ? k_compress_tma<true, true, 64> : k_compress_tma<false, true, 64>)
                           : (v2 ? k_compress_tma<true, false, 64> : k_compress_tma<false, false, 64>);
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
        if (err != cudaSuccess) return err;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                   cudaSharedmemCarveoutMaxShared);
        if (err != cudaSuccess) return err;
        kern<<<(unsigned)nslices, kNT, dyn, s>>>(tmk, tmv, k, v, d, mt, box_rows, max1, side, stage, len, state,
                                                  status);
    }
    k_pack<<<(unsigned)nslices, kNT, 0, s>>>(d, stage, len, off, packed, capacity, state, status);
    return cudaGetLastError();
}

}  // namespace cg
