// decode.cu - range decoding [CG §2.4(1)] fused with dequantisation
// [CG §2.4(2)] for chunks of up to 256 tokens: the launchers of the plain
// (no delta) instantiations of the pipelined kernel in decode_pipe.cuh.
#include "decode_pipe.cuh"

namespace cg {
cudaError_t launch_decode(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                          const uint32_t *len, const uint16_t *cdf, const uint16_t *max1,
                          const Dims &d, const MaxTab &mt, int mode, uint8_t *sym, float *out_k,
                          float *out_v, int32_t *status, cudaStream_t s) {
    const int tmax = d.Tc < d.T ? d.Tc : d.T;
    if (tmax > kThreads || mode == 0)  // symbols out (the step API) or long chunks: one thread per stream
        return launch_decode_generic(packed, packed_bytes, off, len, cdf, max1, d, mt, mode, sym, out_k,
                                     out_v, status, s);
    return launch_decode_pipe(packed, packed_bytes, off, len, cdf, nullptr, max1, d, mt, 1, out_k, out_v,
                              (long long)d.T * d.C, status, s);
}

cudaError_t launch_decode_pipe(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                               const uint32_t *len, const uint16_t *cdf, const uint8_t *rec, const uint16_t *max1,
                               const Dims &d, const MaxTab &mt, int out_dtype, void *out_k, void *out_v,
                               long long ols, int32_t *status, cudaStream_t s) {
    if (d.G > 1)
        return launch_decode_pipe_delta(packed, packed_bytes, off, len, cdf, rec, max1, d, mt, out_dtype, out_k,
                                        out_v, ols, status, s);
    return launch_pipe_any<false>(packed, packed_bytes, off, len, cdf, rec, max1, d, mt, out_dtype, out_k, out_v,
                                  ols, status, s);
}

}  // namespace cg
