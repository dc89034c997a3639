// synth_gpu.cu - the seeded synthetic KV generator on the device: the same
// arithmetic as synth.c (synth_core.h, built with -fmad=false), so the device
// writes the bytes the host would. One thread per (kv, layer, channel) runs
// that channel's sequence over the tokens; per-channel sigmas come from the
// host (syn_slice_sigma). Input generation only: none of the codec is here.
#include <cstdint>

extern "C" {
#include "synth_core.h"
}

namespace {

__global__ void k_synth(syn_params p, const double *__restrict__ sigma, uint16_t *__restrict__ k,
                        uint16_t *__restrict__ v, long long layer_stride) {
    const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (gid >= 2LL * p.L * p.C) return;
    const int c = (int)(gid % p.C);
    const long long r = gid / p.C;
    const int layer = (int)(r % p.L);
    const int kv = (int)(r / p.L);
    const uint64_t key_val = sm64(slice_key(&p, kv, layer), 3);
    uint16_t *out = (kv ? v : k) + (long long)layer * layer_stride + c;
    if (p.kind == SYN_UNIFORM) {
        for (int t = 0; t < p.T; t++) out[(long long)t * p.C] = syn_to_half(u01(sm64(key_val, elem_ctr(c, t))));
    } else if (p.kind == SYN_AR1) {
        const double stat = sqrt(1.0 - p.rho * p.rho);
        const double sg = sigma[gid];
        double x = 0.0;
        for (int t = 0; t < p.T; t++) {
            x = syn_ar1_next(&p, key_val, c, t, sg, stat, x);
            out[(long long)t * p.C] = syn_to_half(x);
        }
    } else {
        const double sg = sigma[gid];
        for (int t = 0; t < p.T; t++) out[(long long)t * p.C] = syn_to_half(syn_student_value(key_val, c, t, sg));
    }
}

}  // namespace

// Fill device K and V ([L][T][C], layers layer_stride elements apart).
// sigma: device doubles [2][L][C] from syn_slice_sigma (ignored for uniform).
extern "C" int syn_generate_device(const syn_params *p, const double *sigma, uint16_t *k, uint16_t *v,
                                   long long layer_stride, void *stream) {
    const long long n = 2LL * p->L * p->C;
    const int threads = 128;
    k_synth<<<(unsigned)((n + threads - 1) / threads), threads, 0, (cudaStream_t)stream>>>(*p, sigma, k, v,
                                                                                         layer_stride);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
