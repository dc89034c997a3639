// codec.cu - CDF construction [CG §2.3(2)], range encoding [CG §1.2(3)] and
// decoding with fused dequantisation [CG §2.4] on sm_103a.
//
// Work unit: one (chunk k, kv, layer l) slice per CTA, one thread per token
// stream (Tc_k <= 1024 threads). The CTA walks the channels in windows of W:
//   1. stage the [Tc_k x W] symbol tile in shared memory (coalesced 16 B loads),
//   2. count symbols per channel (a warp owns a channel; equal symbols of 32
//      tokens merge with one match), normalise to 16-bit frequencies with a
//      warp scan (or load the caller's CDF rows),
//   3. every thread codes its token's W symbols with the window's CDF rows,
//      which all lanes of a warp read from the same shared-memory row.
// Coder state lives in registers: 32-bit low/range plus a 64-bit accumulator
// of emitted-but-unwritten bits, so a carry is a plain add into the
// accumulator; words leave the accumulator one behind ("prev"), so only a
// carry through 32+ one-bits ever touches memory again. The decoder mirrors
// it with a 64-bit bit buffer and a branch-free binary search of the CDF row.
#include <cuda_fp16.h>

#include "cg_internal.cuh"
#include "coder.cuh"

namespace cg {
namespace {

constexpr uint32_t kM = 65536u;

// Window width for alphabet A: a power of two in [16, 64] with W*A <= 4096
// (so a 16-byte symbol vector never straddles a window when C % 16 == 0).
__host__ __device__ inline int window_for(int A) {
    int w = 64;
    while (w > 16 && w * A > 2048) w >>= 1;
    return w;
}

__host__ __device__ inline int pow2_at_least(int a) {
    int p = 1;
    while (p < a) p <<= 1;
    return p;
}

struct EncSmem {
    int W, tile_stride;
    size_t tile_off, cdf_off, total_off, ftab_off, bytes;
};

__host__ __device__ inline EncSmem enc_smem_layout(int NT, int A) {
    EncSmem s;
    s.W = window_for(A);
    s.tile_stride = s.W + 4;  // odd word stride: row-per-lane reads hit distinct banks
    size_t o = 0;
    s.tile_off = o;
    o += (size_t)NT * s.tile_stride;
    o = (o + 15) & ~(size_t)15;
    s.cdf_off = o;  // W*A uint32: lo | f << 16
    o += (size_t)s.W * A * 4;
    s.total_off = o;  // A x (W + 1) uint32 symbol counts, [symbol][channel]
    o += (size_t)(s.W + 1) * A * 4;
    s.ftab_off = o;  // f(n) for n = 0..NT, uint16
    o += (size_t)(NT + 1) * 2;
    s.bytes = (o + 15) & ~(size_t)15;
    return s;
}

// ---- CDF normalisation of one channel (specification F), one warp -------
// counts[s * cs] for s in [0, A) -> packed[s] = lo | f << 16 and, when out != nullptr, the
// uint16 row lo[0..A); when rec != nullptr, the channel's format-2 count
// record (the mode, then the other symbols' counts in increasing s).
// ftab[n] = 1 + floor(n * (65536 - A) / Tk).
__device__ __forceinline__ void build_cdf_row_warp(const uint32_t *counts, int cs, int A,
                                                   const uint16_t *ftab, uint32_t *packed,
                                                   uint16_t *out, uint8_t *rec, int lane) {
    unsigned key = 0, sum = 0;
    for (int s = lane; s < A; s += 32) {
        const unsigned n = counts[s * cs];
        key = max(key, (n << 8) | (255u - (unsigned)s));  // largest n, then smallest s
        sum += ftab[n];
    }
    key = __reduce_max_sync(0xFFFFFFFFu, key);
    sum = __reduce_add_sync(0xFFFFFFFFu, sum);
    const int best = 255 - (int)(key & 255u);
    const unsigned extra = kM - sum;
    if (rec)  // a count other than the mode's is at most Tk / 2 <= 128
        for (int s = lane; s < A; s += 32)
            rec[s == best ? 0 : s + (s < best ? 1 : 0)] = (uint8_t)(s == best ? best : counts[s * cs]);
    unsigned run = 0;
    for (int base = 0; base < A; base += 32) {
        const int s = base + lane;
        const unsigned f = (s < A) ? (unsigned)ftab[counts[s * cs]] + (s == best ? extra : 0u) : 0u;
        unsigned incl = f;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        const unsigned lo = run + incl - f;
        if (s < A) {
            packed[s] = lo | (f << 16);
            if (out) out[s] = (uint16_t)lo;
        }
        run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
}

// ---- slice coder kernel ---------------------------------------------------
// mode 0: counts -> CDF rows only; 1: code with the caller's CDF rows;
// 2: counts -> CDF rows -> code. rec_out != nullptr (modes 0 and 2): format 2,
// the layer's own alphabet 2 MAX + 1 and count records out instead of CDF
// entries.
__global__ void __launch_bounds__(1024, 1) k_code_slices(const uint8_t *__restrict__ sym,
                                                      const uint16_t *__restrict__ cdf_in,
                                                      uint16_t *__restrict__ cdf_out,
                                                      uint8_t *__restrict__ stage,
                                                      uint32_t *__restrict__ len, Dims d,
                                                      int mode, int vec_rows, int32_t *status, MaxTab mt,
                                                      uint8_t *__restrict__ rec_out) {
    extern __shared__ __align__(16) unsigned char smem[];
    int k, kv, l;
    slice_coords(d, blockIdx.x, k, kv, l);
    const int A = rec_out ? 2 * mt.v[kv][l] + 1 : d.A[kv];
    const long long rec_base = rec_out ? record_slice_offset(d, mt, k, kv, l) : 0;
    const int Tk = chunk_tokens(d, k);
    const int NT = blockDim.x;
    const int nwarps = NT >> 5;
    const EncSmem lay = enc_smem_layout(NT, A);
    const int W = lay.W;
    const int ts = lay.tile_stride;
    uint8_t *tile = smem + lay.tile_off;
    uint32_t *cdfw = reinterpret_cast<uint32_t *>(smem + lay.cdf_off);
    uint32_t *total = reinterpret_cast<uint32_t *>(smem + lay.total_off);
    const int cs = W + 1;  // counter row stride: channel c of symbol q at q * cs + c
    uint16_t *ftab = reinterpret_cast<uint16_t *>(smem + lay.ftab_off);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const bool do_count = (mode != 1);
    const bool do_encode = (mode != 0);
    const long long t0 = (long long)k * d.Tc;
    const uint8_t *rows = sym + group_index(d, kv, l, t0) * d.C;
    const long long cdf_base = cdf_slice_offset(d, k, kv, l);
    const long long sid = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk + tid;
    uint8_t *stream = stage_stream(stage, tid < Tk ? sid : 0, d);
    // vec_rows: C % 16 == 0 and sym 16-byte aligned, so with W % 16 == 0 a
    // 16-byte vector never straddles a window
    const int vshift = (W == 64) ? 2 : (W == 32) ? 1 : 0;  // log2(W / 16)

    if (do_count) {
        for (int n = tid; n <= Tk; n += NT)
            ftab[n] = (uint16_t)(1u + ((uint32_t)n * (kM - (uint32_t)A)) / (uint32_t)Tk);
    }

    Enc e;
    enc_init(e);
    int bad = 0;

    for (int c0 = 0; c0 < d.C; c0 += W) {
        const int Wc = min(W, d.C - c0);
        // 1. symbol tile [Tk][Wc]
        if (vec_rows) {
            const int vpr = Wc >> 4;  // vectors per row: 1 << vshift or fewer at the end
            for (int i = tid; i < (Tk << vshift); i += NT) {
                const int r = i >> vshift, j = i & ((1 << vshift) - 1);
                if (j < vpr) {
                    const uint4 q = __ldg(reinterpret_cast<const uint4 *>(rows + (long long)r * d.C + c0) + j);
                    uint32_t *dst = reinterpret_cast<uint32_t *>(tile + r * ts + 16 * j);
                    dst[0] = q.x;
                    dst[1] = q.y;
                    dst[2] = q.z;
                    dst[3] = q.w;
                }
            }
        } else {
            for (int r = warp; r < Tk; r += nwarps)
                for (int j = lane; j < Wc; j += 32) tile[r * ts + j] = rows[(long long)r * d.C + c0 + j];
        }
        if (do_count)
            for (int i = tid; i < cs * A; i += NT) total[i] = 0;
        __syncthreads();

        // 2. per-channel CDF rows for this window
        if (do_count) {
            // each thread counts its token's Wc symbols by shared adds, lane l
            // starting at channel l mod Wc so that the lanes of a warp add to
            // different channels (the padded stride puts them in different banks)
            if (tid < Tk) {
                const uint8_t *my = tile + tid * ts;
                int c = lane % Wc;
                for (int j = 0; j < Wc; j++) {
                    unsigned q = my[c];
                    if (q >= (unsigned)A) {
                        bad = 1;
                        q = A - 1;
                    }
                    atomicAdd(total + q * cs + c, 1u);
                    c = c + 1 == Wc ? 0 : c + 1;
                }
            }
            __syncthreads();
            for (int c = warp; c < Wc; c += nwarps)
                build_cdf_row_warp(total + c, cs, A, ftab, cdfw + c * A,
                                   cdf_out && !rec_out ? cdf_out + cdf_base + (long long)(c0 + c) * A : nullptr,
                                   rec_out ? rec_out + rec_base + (long long)(c0 + c) * A : nullptr, lane);
        } else {
            const uint16_t *src = cdf_in + cdf_base + (long long)c0 * A;
            for (int i = tid; i < Wc * A; i += NT) {
                const int s = i % A;
                const uint32_t lo = src[i];
                const uint32_t hi = (s + 1 < A) ? (uint32_t)src[i + 1] : kM;
                cdfw[i] = lo | ((hi - lo) << 16);
            }
        }
        __syncthreads();

        // 3. code this window's symbols of my token
        if (do_encode && tid < Tk) {
            const uint8_t *my = tile + tid * ts;
            const uint32_t amax = (uint32_t)A - 1;
            int c = 0;
            for (; c + 4 <= Wc; c += 4) {
                const uint32_t q4 = *reinterpret_cast<const uint32_t *>(my + c);
                uint32_t q0 = q4 & 0xFF, q1 = (q4 >> 8) & 0xFF, q2 = (q4 >> 16) & 0xFF, q3 = q4 >> 24;
                if (max(max(q0, q1), max(q2, q3)) > amax) {
                    bad = 1;
                    q0 = min(q0, amax);
                    q1 = min(q1, amax);
                    q2 = min(q2, amax);
                    q3 = min(q3, amax);
                }
                const uint32_t *row = cdfw + c * A;
                if (e.nbits >= 32) enc_flush_word(e, stream);
                enc_symbol(e, row[q0]);
                enc_symbol(e, row[A + q1]);
                if (e.nbits >= 32) enc_flush_word(e, stream);
                enc_symbol(e, row[2 * A + q2]);
                enc_symbol(e, row[3 * A + q3]);
            }
            for (; c < Wc; c++) {
                uint32_t q = my[c];
                if (q > amax) {
                    bad = 1;
                    q = amax;
                }
                if (e.nbits >= 32) enc_flush_word(e, stream);
                enc_symbol(e, cdfw[c * A + q]);
            }
        }
        __syncthreads();
    }
    if (do_encode && tid < Tk) len[sid] = enc_finish(e, stream);
    if (bad && status) atomicOr(status, CG_FLAG_BAD_SYMBOL);
}

// ---- decoder ----------------------------------------------------------------
struct DecSmem {
    int W, tile_stride, P, row_stride;
    size_t tile_off, cdf_off, unit_off, m1_off, bytes;
};

__host__ __device__ inline DecSmem dec_smem_layout(int NT, int A) {
    DecSmem s;
    s.W = window_for(A);
    s.tile_stride = s.W + 4;
    s.P = pow2_at_least(A);
    s.row_stride = s.P + 1;
    size_t o = 0;
    s.tile_off = o;
    o += (size_t)NT * s.tile_stride;
    o = (o + 15) & ~(size_t)15;
    s.cdf_off = o;
    o += (size_t)s.W * s.row_stride * 4;
    s.unit_off = o;
    o += 256 * 4;
    s.m1_off = o;
    o += (size_t)NT * 4;
    s.bytes = (o + 15) & ~(size_t)15;
    return s;
}

struct Dec {
    uint32_t code, range;
    uint64_t bb;       // bit buffer, next bits at the top
    int nb;            // valid bits in bb
    long long wa;      // next aligned word to load (byte offset into packed)
    long long start;   // first byte of the stream
    long long end;     // one past the last readable byte of the stream
};

__device__ __forceinline__ uint32_t load_be_word(const uint8_t *packed, long long wa, long long start,
                                                 long long end) {
    if (wa >= start && wa + 4 <= end) {
        return __byte_perm(__ldg(reinterpret_cast<const uint32_t *>(packed + wa)), 0, 0x0123);
    }
    uint32_t w = 0;
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const long long p = wa + i;
        const uint32_t b = (p >= start && p < end) ? (uint32_t)__ldg(packed + p) : 0u;
        w = (w << 8) | b;
    }
    return w;
}

__device__ __forceinline__ void dec_refill(Dec &s, const uint8_t *packed) {
    const uint32_t w = load_be_word(packed, s.wa, s.start, s.end);
    s.bb |= (uint64_t)w << (32 - s.nb);
    s.nb += 32;
    s.wa += 4;
}

__device__ __forceinline__ void dec_init(Dec &s, const uint8_t *packed, long long start, long long end) {
    s.start = start;
    s.end = end;
    const int a = (int)(start & 3);
    s.wa = start - a;
    const uint32_t w = load_be_word(packed, s.wa, start, end);
    s.wa += 4;
    s.bb = ((uint64_t)w << 32) << (8 * a);
    s.nb = 32 - 8 * a;
    dec_refill(s, packed);  // nb >= 40
    s.code = (uint32_t)(s.bb >> 32);
    s.bb <<= 32;
    s.nb -= 32;
    s.range = 0xFFFFFFFFu;
    dec_refill(s, packed);  // nb >= 40
}

// One symbol; row holds cdf[0..A-1] then 65536 up to index P.
__device__ __forceinline__ uint32_t dec_symbol(Dec &s, const uint32_t *row, int P, int A) {
    const uint32_t r = s.range >> 16;
    int q = 0;
    for (int step = P >> 1; step > 0; step >>= 1) {
        if (r * row[q + step] <= s.code) q += step;
    }
    q = min(q, A - 1);
    const uint32_t lo = row[q];
    const uint32_t hi = row[q + 1];
    s.code -= r * lo;
    s.range = r * (hi - lo);
    const int sh = __clz(s.range) & 24;
    s.code = __funnelshift_l((uint32_t)(s.bb >> 32), s.code, sh);
    s.bb <<= sh;
    s.nb -= sh;
    s.range <<= sh;
    return (uint32_t)q;
}

__global__ void __launch_bounds__(1024, 1) k_decode(const uint8_t *__restrict__ packed,
                                                 long long packed_bytes,
                                                 const uint64_t *__restrict__ off,
                                                 const uint32_t *__restrict__ len,
                                                 const uint16_t *__restrict__ cdf,
                                                 const uint16_t *__restrict__ max1, Dims d,
                                                 MaxTab mt, int mode, uint8_t *__restrict__ sym,
                                                 float *__restrict__ out_k,
                                                 float *__restrict__ out_v, int32_t *status) {
    extern __shared__ __align__(16) unsigned char smem[];
    int k, kv, l;
    slice_coords(d, blockIdx.x, k, kv, l);
    const int A = d.A[kv];
    const int Tk = chunk_tokens(d, k);
    const int NT = blockDim.x;
    const DecSmem lay = dec_smem_layout(NT, A);
    const int W = lay.W, P = lay.P;
    uint8_t *tile = smem + lay.tile_off;
    uint32_t *rows = reinterpret_cast<uint32_t *>(smem + lay.cdf_off);
    float *unit = reinterpret_cast<float *>(smem + lay.unit_off);
    float *m1s = reinterpret_cast<float *>(smem + lay.m1_off);
    const int tid = threadIdx.x;
    const long long t0 = (long long)k * d.Tc;
    const long long cdf_base = cdf_slice_offset(d, k, kv, l);
    const long long sid = chunk_stream_base(d, k) + ((long long)kv * d.L + l) * Tk + tid;

    if (mode == 1) {
        const int MAX = mt.v[kv][l];
        for (int q = tid; q < 256; q += NT)
            unit[q] = __fdiv_rn((float)(q - MAX), (float)MAX);
        for (int t = tid; t < Tk; t += NT)
            m1s[t] = __half2float(__ushort_as_half(max1[group_index(d, kv, l, t0 + t)]));
    }

    Dec s;
    bool corrupt = false;
    if (tid < Tk) {
        long long start = (long long)off[sid];
        long long end = start + (long long)len[sid];
        if (start > packed_bytes || end > packed_bytes) {
            corrupt = true;
            start = min(start, packed_bytes);
            end = min(end, packed_bytes);
        }
        dec_init(s, packed, start, end);
    }

    for (int c0 = 0; c0 < d.C; c0 += W) {
        const int Wc = min(W, d.C - c0);
        const uint16_t *src = cdf + cdf_base + (long long)c0 * A;
        for (int i = tid; i < Wc * (P + 1); i += NT) {
            const int c = i / (P + 1), j = i % (P + 1);
            rows[c * lay.row_stride + j] = (j < A) ? (uint32_t)src[c * A + j] : kM;
        }
        __syncthreads();
        if (tid < Tk) {
            uint8_t *my = tile + tid * lay.tile_stride;
            int c = 0;
            for (; c + 2 <= Wc; c += 2) {
                if (s.nb < 32) dec_refill(s, packed);
                my[c] = (uint8_t)dec_symbol(s, rows + c * lay.row_stride, P, A);
                my[c + 1] = (uint8_t)dec_symbol(s, rows + (c + 1) * lay.row_stride, P, A);
            }
            if (c < Wc) {
                if (s.nb < 32) dec_refill(s, packed);
                my[c] = (uint8_t)dec_symbol(s, rows + c * lay.row_stride, P, A);
            }
        }
        __syncthreads();
        // write the window out, coalesced
        if (mode == 0) {
            uint8_t *dst = sym + group_index(d, kv, l, t0) * d.C + c0;
            for (int r = tid >> 5; r < Tk; r += NT >> 5)
                for (int j = tid & 31; j < Wc; j += 32) dst[(long long)r * d.C + j] = tile[r * lay.tile_stride + j];
        } else {
            float *out = (kv ? out_v : out_k) + ((long long)l * d.T + t0) * d.C + c0;
            if ((d.C & 3) == 0) {
                // Wc is a power of two W except in a ragged last window
                const int per_row = Wc >> 2;
                const int lg = (per_row & (per_row - 1)) == 0 ? __ffs(per_row) - 1 : -1;
                for (int i = tid; i < Tk * per_row; i += NT) {
                    const int r = lg >= 0 ? (i >> lg) : i / per_row;
                    const int j = lg >= 0 ? (i & (per_row - 1)) : i % per_row;
                    const uint32_t q4 = *reinterpret_cast<const uint32_t *>(tile + r * lay.tile_stride + 4 * j);
                    const float m = m1s[r];
                    float4 o;
                    o.x = __fmul_rn(unit[q4 & 0xFF], m);
                    o.y = __fmul_rn(unit[(q4 >> 8) & 0xFF], m);
                    o.z = __fmul_rn(unit[(q4 >> 16) & 0xFF], m);
                    o.w = __fmul_rn(unit[q4 >> 24], m);
                    reinterpret_cast<float4 *>(out + (long long)r * d.C)[j] = o;
                }
            } else {
                for (int r = tid >> 5; r < Tk; r += NT >> 5)
                    for (int j = tid & 31; j < Wc; j += 32)
                        out[(long long)r * d.C + j] = __fmul_rn(unit[tile[r * lay.tile_stride + j]], m1s[r]);
            }
        }
        __syncthreads();
    }
    if (tid < Tk) {
        const long long consumed = (s.wa - s.start) - s.nb / 8;
        if ((corrupt || consumed != (long long)len[sid] + 3) && status) atomicOr(status, CG_FLAG_CORRUPT);
    }
}

int block_threads(const Dims &d) {
    const int tmax = d.Tc < d.T ? d.Tc : d.T;
    return ((tmax + 31) / 32) * 32;
}

}  // namespace

cudaError_t launch_code_slices(const uint8_t *sym, const uint16_t *cdf_in, uint16_t *cdf_out,
                               uint8_t *stage, uint32_t *len, const Dims &d, int mode,
                               int32_t *status, cudaStream_t s, const MaxTab *mt, uint8_t *rec) {
    const long long nslices = 2LL * d.L * d.nch;
    const int NT = block_threads(d);
    size_t smem = 0;
    MaxTab m{};
    if (rec) {  // format 2: every layer's own alphabet
        m = *mt;
        for (int kv = 0; kv < 2; kv++)
            for (int l = 0; l < d.L; l++) {
                const size_t b = enc_smem_layout(NT, 2 * m.v[kv][l] + 1).bytes;
                smem = b > smem ? b : smem;
            }
    } else {
        const size_t s0 = enc_smem_layout(NT, d.A[0]).bytes, s1 = enc_smem_layout(NT, d.A[1]).bytes;
        smem = s0 > s1 ? s0 : s1;
    }
    cudaError_t err = cudaFuncSetAttribute(k_code_slices, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    const int vec_rows = (d.C % 16) == 0 && (reinterpret_cast<uintptr_t>(sym) & 15) == 0;
    k_code_slices<<<(unsigned)nslices, NT, smem, s>>>(sym, cdf_in, cdf_out, stage, len, d, mode, vec_rows,
                                                      status, m, rec);
    return cudaGetLastError();
}

cudaError_t launch_decode_generic(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                                  const uint32_t *len, const uint16_t *cdf, const uint16_t *max1,
                                  const Dims &d, const MaxTab &mt, int mode, uint8_t *sym,
                                  float *out_k, float *out_v, int32_t *status, cudaStream_t s) {
    const long long nslices = 2LL * d.L * d.nch;
    const int NT = block_threads(d);
    const size_t s0 = dec_smem_layout(NT, d.A[0]).bytes, s1 = dec_smem_layout(NT, d.A[1]).bytes;
    const size_t smem = s0 > s1 ? s0 : s1;
    cudaError_t err = cudaFuncSetAttribute(k_decode, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    k_decode<<<(unsigned)nslices, NT, smem, s>>>(packed, (long long)packed_bytes, off, len, cdf, max1,
                                                 d, mt, mode, sym, out_k, out_v, status);
    return cudaGetLastError();
}

}  // namespace cg
