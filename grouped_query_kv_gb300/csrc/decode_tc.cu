// decode_tc.cu -- host side of the tensor-core decode kernel (decode_tc.cuh)
// for contiguous caches: pass sizes, shared memory, and the launches.
#include "decode_tc.cuh"

namespace kvattn {

// Heads per pass: at most 64 (D = 128) or 48 (D = 256, where a 64-head pass
// would not leave room for the K/V ring), spread evenly over the passes.
static int tc_max_heads(int D) { return D == 256 ? 48 : 64; }
int tc_heads_per_seg(int G, int D) {
    const int groups = (G + tc_max_heads(D) - 1) / tc_max_heads(D);
    return (G + groups - 1) / groups;
}
int tc_np(int G, int D) { return (tc_heads_per_seg(G, D) + 15) / 16 * 16; }
// Columns one several-token pass holds: 64 at either head width (at D = 256
// the 64-column configuration keeps one probability stage to fit)
int tc_max_cols_several(int D) { return D == 256 || D == 128 ? 64 : 0; }
int tc_tile() { return kT; }
int tc_threads(int D, int np) {
    return np >= 32 || D == 256 ? TcGroups<256, 32, false>::THREADS
                                : TcGroups<128, 16, false>::THREADS;
}
bool tc_supported(int D, int G) { return (D == 128 || D == 256) && G >= 1; }

template <int D, int NP>
int smem_of() { return TcCfg<D, NP>::alloc; }
template <int D, int NP>
int stages_of() { return TcCfg<D, NP>::NCH; }

int tc_smem_bytes(int D, int np) {
    KVATTN_TC_DISPATCH(smem_of)
    return -1;
}
int tc_stages(int D, int np) {
    KVATTN_TC_DISPATCH(stages_of)
    return -1;
}

// The one-token 16-column kernels (the PaLM-8B and Llama-70B passes) are
// compiled in decode_tc16.cu, so that changes to the other passes' code do
// not move theirs: this kernel's speed has shifted by a percent or more with
// code that never runs.
cudaError_t tc_prepare(int D, int np, bool several_tokens) {
    if (np == 16 && !several_tokens) return tc_prepare_one16(D);
    KVATTN_TC_DISPATCH_MT_NOT16(prepare_t, several_tokens, false)
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_tc(const CUtensorMap &tmk, const CUtensorMap &tmv,
                             const CUtensorMap &tmq, const DecodeParams &p, int np, int num_ctas,
                             cudaStream_t stream) {
    const int D = p.D;
    if (np == 16 && p.T == 1) return launch_decode_tc_one16(tmk, tmv, tmq, p, num_ctas, stream);
    KVATTN_TC_DISPATCH_MT_NOT16(launch_t, p.T > 1, false, tmk, tmv, tmq, p, num_ctas, stream)
    return cudaErrorInvalidValue;
}

}  // namespace kvattn
