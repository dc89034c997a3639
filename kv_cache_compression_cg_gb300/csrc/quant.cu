// quant.cu - adaptive quantisation [CG §2.3(1)] and dequantisation
// [CG §2.4(2)] kernels for sm_103a.
//
// One warp owns one (kv, layer, token) group: 128-bit fp16 loads kept in
// registers, the group's amax taken on the fp16 magnitude bits (for finite
// halves the order of |x| is the order of (bits & 0x7FFF)), a warp max
// reduction, then q = rint((x * factor) + MAX) in binary32 with explicitly
// rounded operations (no contraction into FMA). HBM-bound: 2 B read and 1 B
// written per element.
#include <cuda_fp16.h>

#include "cg_internal.cuh"

namespace cg {
namespace {

__device__ __forceinline__ float half_bits_to_float(unsigned h) {
    return __half2float(__ushort_as_half((unsigned short)h));
}

// Quantise one fp16 value (bits h) to a symbol in [0, 2*MAX].
__device__ __forceinline__ unsigned quant_one(unsigned h, float factor, float fmax, int MAX,
                                              bool zero_group) {
    if (zero_group) return (unsigned)MAX;
    float x = half_bits_to_float(h);
    float y = __fadd_rn(__fmul_rn(x, factor), fmax);
    int q = __float2int_rn(y);
    q = q < 0 ? 0 : q;
    q = q > 2 * MAX ? 2 * MAX : q;
    return (unsigned)q;
}

// 4 halves (two 32-bit words) -> 4 symbols packed little-endian in 32 bits.
__device__ __forceinline__ unsigned quant_word2(unsigned w0, unsigned w1, float factor, float fmax,
                                                int MAX, bool z) {
    unsigned q0 = quant_one(w0 & 0xFFFFu, factor, fmax, MAX, z);
    unsigned q1 = quant_one(w0 >> 16, factor, fmax, MAX, z);
    unsigned q2 = quant_one(w1 & 0xFFFFu, factor, fmax, MAX, z);
    unsigned q3 = quant_one(w1 >> 16, factor, fmax, MAX, z);
    return q0 | (q1 << 8) | (q2 << 16) | (q3 << 24);
}

__device__ __forceinline__ void group_coords(const Dims &d, long long row, int &kv, int &l,
                                             long long &t) {
    t = row % d.T;
    long long r = row / d.T;
    l = (int)(r % d.L);
    kv = (int)(r / d.L);
}

// Vector path: C % 8 == 0 and 16-byte aligned rows; VPL 8-half vectors per lane.
template <int VPL>
__global__ void __launch_bounds__(256) k_quantize_vec(const uint16_t *__restrict__ kin,
                                                      const uint16_t *__restrict__ vin, Dims d,
                                                      MaxTab mt, uint8_t *__restrict__ sym,
                                                      uint16_t *__restrict__ max1,
                                                      int32_t *status) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long rows = 2LL * d.L * d.T;
    const int nvec = d.C >> 3;
    for (long long row = warp; row < rows; row += nwarps) {
        int kv, l;
        long long t;
        group_coords(d, row, kv, l, t);
        const uint16_t *x = (kv ? vin : kin) + (long long)l * d.layer_stride + t * d.C;
        uint4 val[VPL];
        unsigned m = 0;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            int vi = lane + 32 * i;
            if (vi < nvec) {
                val[i] = __ldg(reinterpret_cast<const uint4 *>(x) + vi);
            } else {
                val[i] = make_uint4(0, 0, 0, 0);
            }
            m = __vmaxu2(m, val[i].x & 0x7FFF7FFFu);
            m = __vmaxu2(m, val[i].y & 0x7FFF7FFFu);
            m = __vmaxu2(m, val[i].z & 0x7FFF7FFFu);
            m = __vmaxu2(m, val[i].w & 0x7FFF7FFFu);
        }
        unsigned mm = max(m & 0xFFFFu, m >> 16);
        mm = __reduce_max_sync(0xFFFFFFFFu, mm);
        const int MAX = mt.v[kv][l];
        if (lane == 0) {
            max1[row] = (uint16_t)mm;
            if (mm >= 0x7C00u && status) atomicOr(status, CG_FLAG_NONFINITE);
        }
        const bool z = (mm == 0);
        const float fmax = (float)MAX;
        const float factor = z ? 0.0f : __fdiv_rn(fmax, half_bits_to_float(mm));
        uint8_t *out = sym + row * d.C;
#pragma unroll
        for (int i = 0; i < VPL; i++) {
            int vi = lane + 32 * i;
            if (vi < nvec) {
                uint2 o;
                o.x = quant_word2(val[i].x, val[i].y, factor, fmax, MAX, z);
                o.y = quant_word2(val[i].z, val[i].w, factor, fmax, MAX, z);
                reinterpret_cast<uint2 *>(out)[vi] = o;
            }
        }
    }
}

// Generic path: any C and alignment; reads the group twice (second read from cache).
__global__ void __launch_bounds__(256) k_quantize_any(const uint16_t *__restrict__ kin,
                                                      const uint16_t *__restrict__ vin, Dims d,
                                                      MaxTab mt, uint8_t *__restrict__ sym,
                                                      uint16_t *__restrict__ max1,
                                                      int32_t *status) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long rows = 2LL * d.L * d.T;
    for (long long row = warp; row < rows; row += nwarps) {
        int kv, l;
        long long t;
        group_coords(d, row, kv, l, t);
        const uint16_t *x = (kv ? vin : kin) + (long long)l * d.layer_stride + t * d.C;
        unsigned mm = 0;
        for (int c = lane; c < d.C; c += 32) mm = max(mm, (unsigned)(x[c] & 0x7FFFu));
        mm = __reduce_max_sync(0xFFFFFFFFu, mm);
        const int MAX = mt.v[kv][l];
        if (lane == 0) {
            max1[row] = (uint16_t)mm;
            if (mm >= 0x7C00u && status) atomicOr(status, CG_FLAG_NONFINITE);
        }
        const bool z = (mm == 0);
        const float fmax = (float)MAX;
        const float factor = z ? 0.0f : __fdiv_rn(fmax, half_bits_to_float(mm));
        uint8_t *out = sym + row * d.C;
        for (int c = lane; c < d.C; c += 32) out[c] = (uint8_t)quant_one(x[c], factor, fmax, MAX, z);
    }
}

// Dequantisation, standalone: one warp per group, 4 symbols per lane step.
__global__ void __launch_bounds__(256) k_dequantize(const uint8_t *__restrict__ sym,
                                                    const uint16_t *__restrict__ max1, Dims d,
                                                    MaxTab mt, float *__restrict__ out_k,
                                                    float *__restrict__ out_v) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long rows = 2LL * d.L * d.T;
    const bool vec = (d.C & 3) == 0;
    for (long long row = warp; row < rows; row += nwarps) {
        int kv, l;
        long long t;
        group_coords(d, row, kv, l, t);
        const int MAX = mt.v[kv][l];
        const float fmax = (float)MAX;
        const float m1 = half_bits_to_float(max1[row]);
        const uint8_t *q = sym + row * d.C;
        float *o = (kv ? out_v : out_k) + ((long long)l * d.T + t) * d.C;
        if (vec) {
            for (int c4 = lane; c4 < (d.C >> 2); c4 += 32) {
                unsigned w = reinterpret_cast<const unsigned *>(q)[c4];
                float4 r;
                r.x = __fmul_rn(__fdiv_rn((float)((int)(w & 0xFF) - MAX), fmax), m1);
                r.y = __fmul_rn(__fdiv_rn((float)((int)((w >> 8) & 0xFF) - MAX), fmax), m1);
                r.z = __fmul_rn(__fdiv_rn((float)((int)((w >> 16) & 0xFF) - MAX), fmax), m1);
                r.w = __fmul_rn(__fdiv_rn((float)((int)(w >> 24) - MAX), fmax), m1);
                reinterpret_cast<float4 *>(o)[c4] = r;
            }
        } else {
            for (int c = lane; c < d.C; c += 32)
                o[c] = __fmul_rn(__fdiv_rn((float)((int)q[c] - MAX), fmax), m1);
        }
    }
}

// ---- token-locality delta [CG §1.2(1)] -----------------------------------
// One warp per token group: the anchor row first (plain quantisation, its
// reconstruction kept), then each other row as d = x - a^ with max1 the
// binary16 value rounded up from max |d| (65504 above it), q clamped to
// [0, 2 MAX]. HBM-bound like the plain kernels.

// Smallest binary16 >= m (m >= 0; NaN and values above 65504 give 65504).
__device__ __forceinline__ unsigned half_up_bits(float m) {
    const unsigned h = __half_as_ushort(__float2half_ru(m));
    return h >= 0x7C00u ? 0x7BFFu : h;
}

__device__ __forceinline__ float dequant_one(unsigned q, int MAX, float fmax, float m1) {
    return __fmul_rn(__fdiv_rn((float)((int)q - MAX), fmax), m1);
}

__device__ __forceinline__ unsigned quant_delta_one(float dv, float factor, float fmax, int MAX, bool z) {
    if (z) return (unsigned)MAX;
    int q = __float2int_rn(__fadd_rn(__fmul_rn(dv, factor), fmax));
    q = q < 0 ? 0 : q;
    return (unsigned)(q > 2 * MAX ? 2 * MAX : q);
}

// Vector path: C % 8 == 0, 16-byte aligned rows, C <= 256 VPL.
template <int VPL>
__global__ void __launch_bounds__(256) k_quantize_delta_vec(const uint16_t *__restrict__ kin,
                                                            const uint16_t *__restrict__ vin, Dims d,
                                                            MaxTab mt, uint8_t *__restrict__ sym,
                                                            uint16_t *__restrict__ max1,
                                                            int32_t *status) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long tasks = 2LL * d.L * d.nch * delta_groups_per_chunk(d);
    const int nvec = d.C >> 3;
    for (long long task = warp; task < tasks; task += nwarps) {
        int kv, l, n;
        long long ta;
        delta_task(d, task, kv, l, ta, n);
        if (n <= 0) continue;
        const int MAX = mt.v[kv][l];
        const float fmax = (float)MAX;
        const uint16_t *xb = (kv ? vin : kin) + (long long)l * d.layer_stride;
        float a[VPL][8];
        bool bad = false;
        for (int r = 0; r < n; r++) {
            const long long t = ta + r;
            const long long row = group_index(d, kv, l, t);
            const uint16_t *x = xb + t * d.C;
            uint4 val[VPL];
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const int vi = lane + 32 * i;
                val[i] = vi < nvec ? __ldg(reinterpret_cast<const uint4 *>(x) + vi) : make_uint4(0, 0, 0, 0);
            }
            // max1: the anchor's |x| (as fp16 bits), the others' |x - a^| rounded up
            unsigned mh;
            if (r == 0) {
                unsigned m = 0;
#pragma unroll
                for (int i = 0; i < VPL; i++) {
                    m = __vmaxu2(m, val[i].x & 0x7FFF7FFFu);
                    m = __vmaxu2(m, val[i].y & 0x7FFF7FFFu);
                    m = __vmaxu2(m, val[i].z & 0x7FFF7FFFu);
                    m = __vmaxu2(m, val[i].w & 0x7FFF7FFFu);
                }
                mh = __reduce_max_sync(0xFFFFFFFFu, max(m & 0xFFFFu, m >> 16));
                bad |= mh >= 0x7C00u;
            } else {
                unsigned mb = 0;  // |d| bits: non-negative floats order like their bits
#pragma unroll
                for (int i = 0; i < VPL; i++) {
                    if (lane + 32 * i >= nvec) continue;  // no channels (and no a^) there
                    const uint32_t *w = reinterpret_cast<const uint32_t *>(&val[i]);
#pragma unroll
                    for (int j = 0; j < 8; j++) {
                        const float dv = __fsub_rn(half_bits_to_float((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu), a[i][j]);
                        mb = max(mb, __float_as_uint(dv) & 0x7FFFFFFFu);
                    }
                }
                mb = __reduce_max_sync(0xFFFFFFFFu, mb);
                bad |= mb >= 0x7F800000u;
                mh = half_up_bits(__uint_as_float(mb));
            }
            if (lane == 0) max1[row] = (uint16_t)mh;
            const bool z = mh == 0;
            const float m1 = half_bits_to_float(mh);
            const float factor = z ? 0.0f : __fdiv_rn(fmax, m1);
            uint8_t *out = sym + row * d.C;
#pragma unroll
            for (int i = 0; i < VPL; i++) {
                const int vi = lane + 32 * i;
                if (vi >= nvec) continue;
                const uint32_t *w = reinterpret_cast<const uint32_t *>(&val[i]);
                unsigned q[8];
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    const float xv = half_bits_to_float((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
                    if (r == 0) {
                        q[j] = quant_one((w[j >> 1] >> (16 * (j & 1))) & 0xFFFFu, factor, fmax, MAX, z);
                        a[i][j] = dequant_one(q[j], MAX, fmax, m1);
                    } else {
                        q[j] = quant_delta_one(__fsub_rn(xv, a[i][j]), factor, fmax, MAX, z);
                    }
                }
                uint2 o;
                o.x = q[0] | (q[1] << 8) | (q[2] << 16) | (q[3] << 24);
                o.y = q[4] | (q[5] << 8) | (q[6] << 16) | (q[7] << 24);
                reinterpret_cast<uint2 *>(out)[vi] = o;
            }
        }
        if (bad && lane == 0 && status) atomicOr(status, CG_FLAG_NONFINITE);
    }
}

// Generic path: any C and alignment. A lane reads back the anchor symbols it
// wrote itself (same channels), so no cross-lane ordering is needed.
__global__ void __launch_bounds__(256) k_quantize_delta_any(const uint16_t *__restrict__ kin,
                                                            const uint16_t *__restrict__ vin, Dims d,
                                                            MaxTab mt, uint8_t *sym,
                                                            uint16_t *__restrict__ max1,
                                                            int32_t *status) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long tasks = 2LL * d.L * d.nch * delta_groups_per_chunk(d);
    for (long long task = warp; task < tasks; task += nwarps) {
        int kv, l, n;
        long long ta;
        delta_task(d, task, kv, l, ta, n);
        if (n <= 0) continue;
        const int MAX = mt.v[kv][l];
        const float fmax = (float)MAX;
        const uint16_t *xb = (kv ? vin : kin) + (long long)l * d.layer_stride;
        const long long arow = group_index(d, kv, l, ta);
        const uint8_t *qa = sym + arow * d.C;
        bool bad = false;
        float m1a = 0.0f;
        for (int r = 0; r < n; r++) {
            const long long t = ta + r;
            const long long row = group_index(d, kv, l, t);
            const uint16_t *x = xb + t * d.C;
            unsigned mh;
            if (r == 0) {
                unsigned m = 0;
                for (int c = lane; c < d.C; c += 32) m = max(m, (unsigned)(x[c] & 0x7FFFu));
                mh = __reduce_max_sync(0xFFFFFFFFu, m);
                bad |= mh >= 0x7C00u;
            } else {
                unsigned mb = 0;
                for (int c = lane; c < d.C; c += 32) {
                    const float dv = __fsub_rn(half_bits_to_float(x[c]), dequant_one(qa[c], MAX, fmax, m1a));
                    mb = max(mb, __float_as_uint(dv) & 0x7FFFFFFFu);
                }
                mb = __reduce_max_sync(0xFFFFFFFFu, mb);
                bad |= mb >= 0x7F800000u;
                mh = half_up_bits(__uint_as_float(mb));
            }
            if (lane == 0) max1[row] = (uint16_t)mh;
            const bool z = mh == 0;
            const float m1 = half_bits_to_float(mh);
            const float factor = z ? 0.0f : __fdiv_rn(fmax, m1);
            uint8_t *out = sym + row * d.C;
            for (int c = lane; c < d.C; c += 32) {
                if (r == 0)
                    out[c] = (uint8_t)quant_one(x[c], factor, fmax, MAX, z);
                else
                    out[c] = (uint8_t)quant_delta_one(
                        __fsub_rn(half_bits_to_float(x[c]), dequant_one(qa[c], MAX, fmax, m1a)), factor, fmax, MAX, z);
            }
            if (r == 0) m1a = m1;
        }
        if (bad && lane == 0 && status) atomicOr(status, CG_FLAG_NONFINITE);
    }
}

// Dequantisation with the delta: warp per group; x^ = a^ + D(q) off the anchor.
__global__ void __launch_bounds__(256) k_dequantize_delta(const uint8_t *__restrict__ sym,
                                                          const uint16_t *__restrict__ max1, Dims d,
                                                          MaxTab mt, float *__restrict__ out_k,
                                                          float *__restrict__ out_v) {
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long tasks = 2LL * d.L * d.nch * delta_groups_per_chunk(d);
    for (long long task = warp; task < tasks; task += nwarps) {
        int kv, l, n;
        long long ta;
        delta_task(d, task, kv, l, ta, n);
        if (n <= 0) continue;
        const int MAX = mt.v[kv][l];
        const float fmax = (float)MAX;
        const long long arow = group_index(d, kv, l, ta);
        const uint8_t *qa = sym + arow * d.C;
        const float m1a = half_bits_to_float(max1[arow]);
        for (int r = 0; r < n; r++) {
            const long long row = arow + r;
            const float m1 = half_bits_to_float(max1[row]);
            const uint8_t *q = sym + row * d.C;
            float *o = (kv ? out_v : out_k) + ((long long)l * d.T + ta + r) * d.C;
            for (int c = lane; c < d.C; c += 32) {
                float x = dequant_one(q[c], MAX, fmax, m1);
                if (r > 0) x = __fadd_rn(dequant_one(qa[c], MAX, fmax, m1a), x);
                o[c] = x;
            }
        }
    }
}

int grid_for_rows(long long rows) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long want = (rows + 7) / 8;           // 8 warps (rows) per 256-thread block
    long long cap = (long long)sms * 8;        // up to 8 resident blocks per SM
    return (int)(want < cap ? (want < 1 ? 1 : want) : cap);
}

}  // namespace

cudaError_t launch_quantize(const uint16_t *k, const uint16_t *v, const Dims &d,
                            const MaxTab &mt, uint8_t *sym, uint16_t *max1, int32_t *status,
                            cudaStream_t s) {
    const long long rows = 2LL * d.L * d.T;
    const int grid = grid_for_rows(rows);
    const bool aligned = ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(sym) & 7) == 0 && (d.layer_stride % 8) == 0 &&
                         (d.C % 8) == 0;
    const int nvec = d.C / 8;
    if (aligned && nvec <= 32) {
        k_quantize_vec<1><<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    } else if (aligned && nvec <= 64) {
        k_quantize_vec<2><<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    } else if (aligned && nvec <= 128) {
        k_quantize_vec<4><<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    } else if (aligned && nvec <= 256) {
        k_quantize_vec<8><<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    } else {
        k_quantize_any<<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t *sym, const uint16_t *max1, const Dims &d,
                              const MaxTab &mt, float *out_k, float *out_v, cudaStream_t s) {
    const long long rows = 2LL * d.L * d.T;
    k_dequantize<<<grid_for_rows(rows), 256, 0, s>>>(sym, max1, d, mt, out_k, out_v);
    return cudaGetLastError();
}

cudaError_t launch_quantize_delta(const uint16_t *k, const uint16_t *v, const Dims &d,
                                  const MaxTab &mt, uint8_t *sym, uint16_t *max1, int32_t *status,
                                  cudaStream_t s) {
    const long long tasks = 2LL * d.L * d.nch * delta_groups_per_chunk(d);
    const int grid = grid_for_rows(tasks);
    const bool aligned = ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0 &&
                         (reinterpret_cast<uintptr_t>(sym) & 7) == 0 && (d.layer_stride % 8) == 0 &&
                         (d.C % 8) == 0;
    const int nvec = d.C / 8;
    if (aligned && nvec <= 32) {
        k_quantize_delta_vec<1><<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    } else if (aligned && nvec <= 64) {
        k_quantize_delta_vec<2><<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    } else if (aligned && nvec <= 128) {
        k_quantize_delta_vec<4><<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    } else {
        k_quantize_delta_any<<<grid, 256, 0, s>>>(k, v, d, mt, sym, max1, status);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize_delta(const uint8_t *sym, const uint16_t *max1, const Dims &d,
                                    const MaxTab &mt, float *out_k, float *out_v, cudaStream_t s) {
    const long long tasks = 2LL * d.L * d.nch * delta_groups_per_chunk(d);
    k_dequantize_delta<<<grid_for_rows(tasks), 256, 0, s>>>(sym, max1, d, mt, out_k, out_v);
    return cudaGetLastError();
}

}  // namespace cg
