// decode_tc16.cu -- launches of the one-token tensor-core kernel
// (decode_tc.cuh) with 16 columns per pass over a contiguous cache: the
// multi-query and grouped-query passes of up to 16 heads per K/V head.  A
// translation unit of its own, so that its code does not move when the
// other passes' code changes.
#include "decode_tc.cuh"

namespace kvattn {

cudaError_t tc_prepare_one16(int D) {
    if (D == 128) return prepare_t<128, 16, false, false>();
    if (D == 256) return prepare_t<256, 16, false, false>();
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_tc_one16(const CUtensorMap &tmk, const CUtensorMap &tmv,
                                   const CUtensorMap &tmq, const DecodeParams &p, int num_ctas,
                                   cudaStream_t stream) {
    if (p.D == 128) return launch_t<128, 16, false, false>(tmk, tmv, tmq, p, num_ctas, stream);
    if (p.D == 256) return launch_t<256, 16, false, false>(tmk, tmv, tmq, p, num_ctas, stream);
    return cudaErrorInvalidValue;
}

}  // namespace kvattn
