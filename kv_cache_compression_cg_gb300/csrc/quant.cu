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

}  // namespace cg
