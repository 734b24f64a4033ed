// noalloc.cu -- gqa_decode_attn_noalloc: decode attention that never
// allocates device memory.
//
// Why it exists.  The regular entry point keeps a per-(device, stream)
// workspace for the partial results of sequences that the persistent grid
// splits across several CTAs, and grows it with cudaMalloc/cudaFree the
// first time a larger one is needed.  Some callers cannot allow that: a
// serving process that hands all free device memory to its own pool at
// start-up (a later cudaMalloc fails or fragments that pool), or a
// latency-critical loop where the device-wide synchronisation that cudaFree
// implies is not acceptable.  This variant runs the same CUDA-core split-KV
// kernel and combine, but keeps its partials in one fixed array that is part
// of the library image and is therefore created when the library is loaded.
//
// The scratch array.  kNoallocScratchBytes (4 MiB) of device memory, one
// copy per GPU that loads the library, held until the process exits.  Host
// code must not pass `g_noalloc_scratch` itself to a kernel: on the host that
// name only stands for the device symbol.  The device address is looked up
// with cudaGetSymbolAddress once per device, on the first call made while
// that device is current; make that first call before capturing work on the
// device's streams into anything.  Every call on a device shares the array
// and it keeps the previous call's contents; nothing in it needs to start at
// zero, because each call writes every partial slot it later reads.  Two
// calls whose kernels overlap on the GPU (different streams, no ordering
// between them) race on the array and may produce wrong results.
#include <cstdio>
#include <mutex>

#include "../../include/kvattn.h"
#include "internal.h"

namespace {

constexpr size_t kNoallocScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

struct NoallocDevice {
    bool ready;
    int num_sms;
    void *scratch;      // device address of g_noalloc_scratch on this device
    unsigned int *err;  // device address of the sticky error word
};

std::mutex g_noalloc_mu;
NoallocDevice g_noalloc_dev[kMaxDevices];

// Once per device, with that device current.
int noalloc_setup(int dev, NoallocDevice **out) {
    if (dev < 0 || dev >= kMaxDevices)
        return kvattn::api_fail(KVATTN_ERR_UNSUPPORTED, "device ordinal beyond 63");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    NoallocDevice &d = g_noalloc_dev[dev];
    if (!d.ready) {
        cudaError_t e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return kvattn::api_cuda_fail(e, "cudaDeviceGetAttribute");
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return kvattn::api_cuda_fail(e, "cudaGetSymbolAddress(scratch)");
        int rc = kvattn::api_error_word(&d.err);
        if (rc) return rc;
        d.scratch = p;
        d.ready = true;
    }
    *out = &d;
    return KVATTN_OK;
}

}  // namespace

extern "C" int gqa_decode_attn_noalloc(const void *q, const void *k_cache,
                                       const void *v_cache, const int32_t *seq_lens,
                                       float *out, int B, int Hq, int Hkv, int D, int Lmax,
                                       float scale, kvattn_stream_t stream_) {
    using namespace kvattn;
    int rc = api_check_args(q, k_cache, v_cache, seq_lens, out, B, Hq, Hkv, D, Lmax, scale);
    if (rc) return rc;

    const int G = Hq / Hkv;
    const int hps = fma_heads_per_seg(G);
    const int tile = fma_tile(D);
    const int smem = fma_smem_bytes(D, hps);

    int num_ctas = api_forced_ctas();
    NoallocDevice *nd = nullptr;
    int dev = 0;
    if (num_ctas <= 0) {
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return api_cuda_fail(e, "cudaGetDevice");
        if ((rc = noalloc_setup(dev, &nd))) return rc;
        num_ctas = nd->num_sms;
    }
    // partial (o, m, l) for up to two pieces per CTA, and one combine record per CTA
    const size_t need = size_t(2) * num_ctas * hps * (D + 2) * sizeof(float) + size_t(16) * num_ctas;
    if (need > kNoallocScratchBytes) {
        char msg[192];
        snprintf(msg, sizeof msg,
                 "needs %zu bytes of scratch for %d CTAs; the no-alloc variant holds %zu",
                 need, num_ctas, kNoallocScratchBytes);
        return api_fail(KVATTN_ERR_UNSUPPORTED, msg);
    }
    if (!nd) {
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return api_cuda_fail(e, "cudaGetDevice");
        if ((rc = noalloc_setup(dev, &nd))) return rc;
    }

    CUtensorMap tmk, tmv;
    if ((rc = api_encode_cache_maps(&tmk, &tmv, k_cache, v_cache, D, Lmax, B * Hkv, tile)))
        return rc;

    DecodeParams p = {};
    p.q = static_cast<const uint16_t *>(q);
    p.seq_lens = seq_lens;
    p.len_add = 0;
    p.k_new = p.v_new = nullptr;
    p.k_cache = p.v_cache = nullptr;
    p.out = out;
    p.ws_o = static_cast<float *>(nd->scratch);
    p.ws_ml = p.ws_o + size_t(2) * num_ctas * hps * D;
    p.split = reinterpret_cast<int *>(p.ws_ml + size_t(2) * num_ctas * hps * 2);
    p.err = nd->err;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.Lmax = Lmax;
    p.G = G;
    p.heads_per_seg = hps;
    p.hpg = hps;
    p.head_groups = (G + hps - 1) / hps;
    p.tile = tile;
    p.cost_piece = 16;  // the regular entry point's schedule weight for this path
    p.window = Lmax;    // full attention
    p.qwin = Lmax;
    p.walign = 0;
    p.T = 1;
    p.q_bytes = 0;      // (the CUDA-core kernel reads q itself)
    p.block_table = nullptr;  // contiguous cache
    p.block_lg = 0;
    p.max_blocks = 0;
    p.num_blocks = 0;
    p.k_scale = nullptr;
    p.v_scale = nullptr;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    cudaError_t e = fma_prepare(D, hps, smem);
    if (e != cudaSuccess) return api_cuda_fail(e, "cudaFuncSetAttribute");
    e = launch_decode_fma(tmk, tmv, p, num_ctas, smem, stream);
    if (e != cudaSuccess) return api_cuda_fail(e, "decode kernel launch");
    e = launch_combine(p, num_ctas, stream);
    if (e != cudaSuccess) return api_cuda_fail(e, "combine kernel launch");
    return KVATTN_OK;
}
