// decode_delta.cu - the token-locality delta [CG §1.2(1)] instantiations of
// the pipelined decode kernel in decode_pipe.cuh (their own translation unit,
// so the library's objects compile in parallel).
#include "decode_pipe.cuh"

namespace cg {

cudaError_t launch_decode_pipe_delta(const uint8_t *packed, uint64_t packed_bytes, const uint64_t *off,
                                     const uint32_t *len, const uint16_t *cdf, const uint8_t *rec,
                                     const uint16_t *max1, const Dims &d, const MaxTab &mt, int out_dtype,
                                     void *out_k, void *out_v, long long ols, int32_t *status, cudaStream_t s) {
    return launch_pipe_any<true>(packed, packed_bytes, off, len, cdf, rec, max1, d, mt, out_dtype, out_k, out_v,
                                 ols, status, s);
}

}  // namespace cg
