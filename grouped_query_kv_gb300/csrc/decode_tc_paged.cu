// decode_tc_paged.cu -- launches of the tensor-core decode kernel
// (decode_tc.cuh) over a paged cache; a translation unit of its own so the
// paged instantiations compile beside the contiguous ones.
#include "decode_tc.cuh"

namespace kvattn {

cudaError_t tc_prepare_paged(int D, int np, bool several_tokens) {
    KVATTN_TC_DISPATCH_MT(prepare_t, several_tokens, true)
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_tc_paged(const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   const CUtensorMap &tmq, const DecodeParams &p, int np,
                                   int num_ctas, cudaStream_t stream) {
    const int D = p.D;
    KVATTN_TC_DISPATCH_MT(launch_t, p.T > 1, true, tmk, tmv, tmq, p, num_ctas, stream)
    return cudaErrorInvalidValue;
}

}  // namespace kvattn
