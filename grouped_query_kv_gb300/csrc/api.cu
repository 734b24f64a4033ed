// api.cu -- the C ABI declared in include/kvattn.h: argument checks, the
// split plan, TMA descriptors, per-(device, stream) workspaces and launches.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <vector>
#include <mutex>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/kvattn.h"
#include "internal.h"

using namespace kvattn;

// The sticky device error word (one copy per device, as for every __device__
// variable).  Kernels receive its address as a plain pointer.
__device__ unsigned int g_kvattn_device_error;

namespace {

thread_local char t_last_error[512] = "";

int fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_last_error, sizeof t_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(KVATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

std::mutex g_mu;
int g_force_path = 0;
int g_force_ctas = 0;
unsigned int g_wait_limit = 0;           // 0: the kernels' default wait limits
cudaEvent_t g_ev_before = nullptr;       // measurement hook around the split-KV kernel
cudaEvent_t g_ev_after = nullptr;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    unsigned int *err = nullptr;
};
std::map<int, DeviceState> g_dev;

struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
    // buffers outgrown by this one: kept until kvattn_release, because work
    // captured earlier (a CUDA graph) may still use them
    std::vector<void *> retired;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

// cuTensorMapEncodeTiled, fetched through the runtime so the library needs no
// link-time dependency on the driver library.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    return KVATTN_OK;
}

// Per-device lazy set-up (under g_mu).
int device_state(int dev, DeviceState **out) {
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        cudaError_t e = cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&s.err), g_kvattn_device_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
        s.ready = true;
    }
    *out = &s;
    return KVATTN_OK;
}

int get_encoder() {
    if (g_encode) return KVATTN_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(KVATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return KVATTN_OK;
}

// 3-D map over one cache: dims (D, Lmax, B*Hkv), box (64, tile, 1),
// 128-byte swizzle; rows past Lmax read as zeros.
int encode_cache_map(CUtensorMap *m, const void *base, int D, int Lmax, int BH, int tile) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Lmax, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * (cuuint64_t)Lmax};
    cuuint32_t box[3] = {64, (cuuint32_t)tile, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return KVATTN_OK;
}

// 3-D map over a paged pool [num_blocks, Hkv, block_size, D] viewed as
// (D, block_size, num_blocks*Hkv): box (64, min(block_size, 128), 1), the
// same 128-byte swizzle; a tile is min(block_size, 128)-row boxes stacked.
int encode_pool_map(CUtensorMap *m, const void *base, int D, int block_size, long long rows) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)block_size, (cuuint64_t)rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)D * 2 * (cuuint64_t)block_size};
    cuuint32_t box[3] = {64, (cuuint32_t)(block_size < 128 ? block_size : 128), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVATTN_ERR_CUDA, "cuTensorMapEncodeTiled(pool) failed (%d)", (int)r);
    return KVATTN_OK;
}

// A paged cache: pools [num_blocks, Hkv, block_size, D] and the block table.
struct Paged {
    const int32_t *table;  // [B, max_blocks]
    int block_size, max_blocks, num_blocks;
};

// Checks a paged cache's sizes; on success *lg = log2(block_size) and
// *Lmax = the positions a table row can address.
int check_paged(const Paged &pg, int Hkv, const char *who, int *lg, int *Lmax) {
    if (!pg.table) return fail(KVATTN_ERR_INVALID_ARG, "%s: null block table", who);
    if (reinterpret_cast<uintptr_t>(pg.table) & 3u)
        return fail(KVATTN_ERR_INVALID_ARG, "%s: block table must be 4-byte aligned", who);
    const int bs = pg.block_size;
    if (bs < 16 || bs > (1 << 20) || (bs & (bs - 1)))
        return fail(KVATTN_ERR_UNSUPPORTED, "%s: block_size must be a power of two in [16, 2^20] (got %d)",
                    who, bs);
    if (pg.max_blocks <= 0 || pg.num_blocks <= 0)
        return fail(KVATTN_ERR_INVALID_ARG, "%s: max_blocks and num_blocks must be positive", who);
    if ((long long)pg.num_blocks * Hkv > 0x7fffffffLL)
        return fail(KVATTN_ERR_UNSUPPORTED, "%s: num_blocks * Hkv beyond 2^31", who);
    if ((long long)pg.max_blocks * bs > (1LL << 24))
        return fail(KVATTN_ERR_UNSUPPORTED, "%s: max_blocks * block_size beyond 2^24", who);
    int l = 0;
    while ((1 << l) < bs) ++l;
    *lg = l;
    *Lmax = pg.max_blocks * bs;
    return KVATTN_OK;
}

// 3-D map over an 8-bit cache [B*Hkv, Lmax, D] of one-byte codes: dims
// (D, Lmax, B*Hkv), box (128, tile, 1), 128-byte swizzle: one box is the
// tile's codes of 128 head dims (D / 128 boxes per tile).
int encode_fp8_map(CUtensorMap *m, const void *base, int D, int Lmax, int BH, int tile) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Lmax, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D, (cuuint64_t)D * (cuuint64_t)Lmax};
    cuuint32_t box[3] = {128, (cuuint32_t)tile, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVATTN_ERR_CUDA, "cuTensorMapEncodeTiled(fp8) failed (%d)", (int)r);
    return KVATTN_OK;
}

struct Plan {
    kvattn_plan pub;
    int heads_per_seg;  // query rows per pass (heads, or hpg heads x T tokens)
    int hpg;            // query heads per pass
    int np;  // tensor-core path: heads per pass rounded up to 16
    int cost_piece;  // schedule weight of a piece (a tile weighs 32)
};

// Path choice: the tensor-core kernel whenever D is 128 or 256, for every
// group size G (heads are padded to a multiple of 16 MMA columns, which the
// tensor pipe absorbs: measured on GB300 it streams at copy bandwidth even
// at G = 1, where the CUDA-core kernel is instruction-bound); the CUDA-core
// kernel for D = 64.
int make_plan(int B, int Hq, int Hkv, int D, int Lmax, int num_sms, Plan *pl, int T = 1) {
    (void)Lmax;
    (void)B;
    const int G = Hq / Hkv;
    kvattn_plan &p = pl->pub;
    memset(&p, 0, sizeof p);
    const bool tc_ok = (D == 128 || D == 256);
    int path = tc_ok ? 2 : 1;
    if (g_force_path == 1) path = 1;
    if (g_force_path == 2 || T > 1) {
        if (!tc_ok)
            return fail(KVATTN_ERR_UNSUPPORTED, "tensor-core path needs D in {128, 256} (D=%d)", D);
        path = 2;
    }
    if (T > 1 && g_force_path == 1)
        return fail(KVATTN_ERR_UNSUPPORTED, "several new tokens need the tensor-core path");
    p.path = path;
    if (T > 1) {
        // one pass takes hpg of the group's heads for all T tokens as its
        // columns; a group whose G x T query rows exceed one pass is split
        // into passes of (nearly) equal head counts, each re-reading the K/V
        const int maxcols = tc_max_cols_several(D);  // columns one pass holds
        if (T > maxcols)
            return fail(KVATTN_ERR_UNSUPPORTED, "T = %d new tokens exceed one pass (%d at D=%d)",
                        T, maxcols, D);
        const int hmax = maxcols / T;
        const int passes = (G + hmax - 1) / hmax;
        pl->hpg = (G + passes - 1) / passes;
        pl->heads_per_seg = pl->hpg * T;
        pl->np = (pl->heads_per_seg + 15) / 16 * 16;
        p.tile_positions = tc_tile();
        p.stages = tc_stages(D, pl->np);
        p.threads = tc_threads(D, pl->np);
        p.smem_bytes = tc_smem_bytes(D, pl->np);
    } else if (path == 2) {
        pl->heads_per_seg = pl->hpg = tc_heads_per_seg(G, D);
        pl->np = tc_np(G, D);
        p.tile_positions = tc_tile();
        p.stages = tc_stages(D, pl->np);
        p.threads = tc_threads(D, pl->np);
        p.smem_bytes = tc_smem_bytes(D, pl->np);
    } else {
        pl->heads_per_seg = pl->hpg = fma_heads_per_seg(G);
        pl->np = 0;
        p.tile_positions = fma_tile(D);
        p.stages = fma_stages(D);
        p.threads = fma_threads();
        p.smem_bytes = fma_smem_bytes(D, pl->heads_per_seg);
    }
    p.heads_per_cta = pl->heads_per_seg;
    p.head_groups = (G + pl->hpg - 1) / pl->hpg;
    // CTA ranges balance cost: a tile costs W and a piece (q load, the first
    // tile's exact max, the output's read-out and stores) costs P more.
    // Measured on GB300 with the tensor-core kernel, a piece takes about
    // (0.6 + 0.05 NP) tiles' time at D = 128 and half as many D = 256 tiles
    // (twice the bytes each).
    pl->cost_piece = path == 2 ? (int)lround(32.0 * (0.6 + 0.05 * pl->np) * 128.0 / D) : 16;
    const int ctas = g_force_ctas > 0 ? g_force_ctas : num_sms;
    p.num_ctas = ctas;
    p.workspace_bytes = (int64_t)2 * ctas * pl->heads_per_seg * (D + 2) * (int64_t)sizeof(float) +
                        (int64_t)ctas * 16;
    return KVATTN_OK;
}

// 3-D map over q, 128-byte swizzle.  One token per sequence: q viewed as
// (D, B*Hq, 1) with box (64, np, 1).  T tokens: q [B, T, Hq, D] viewed as
// (D, Hq, B*T) with box (64, hpg, T) -- one pass's heads of every token.
int encode_q_map(CUtensorMap *m, const void *base, int D, int B, int T, int Hq, int hpg, int np) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)(T == 1 ? B * Hq : Hq),
                          (cuuint64_t)(T == 1 ? 1 : B * T)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)(T == 1 ? B * Hq : Hq) * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)(T == 1 ? np : hpg), (cuuint32_t)T};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KVATTN_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed (%d)", (int)r);
    return KVATTN_OK;
}

int check_sizes(int B, int Hq, int Hkv, int D, int Lmax) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Lmax <= 0)
        return fail(KVATTN_ERR_INVALID_ARG, "sizes must be positive (B=%d Hq=%d Hkv=%d D=%d Lmax=%d)",
                    B, Hq, Hkv, D, Lmax);
    if (Hq % Hkv != 0)
        return fail(KVATTN_ERR_INVALID_ARG, "Hq (%d) is not a multiple of Hkv (%d)", Hq, Hkv);
    if (D != 64 && D != 128 && D != 256)
        return fail(KVATTN_ERR_UNSUPPORTED, "head dimension D=%d not in {64, 128, 256}", D);
    if (B > 65535 || Hkv > 4096 || Hq > 8192 || Lmax > (1 << 24))
        return fail(KVATTN_ERR_UNSUPPORTED,
                    "sizes beyond limits (B<=65535, Hkv<=4096, Hq<=8192, Lmax<=2^24)");
    // the kernels count one segment's tiles of all sequences in 32 bits
    if ((long long)B * ((Lmax + 63) / 64) > (1LL << 30))
        return fail(KVATTN_ERR_UNSUPPORTED, "B * ceil(Lmax / 64) beyond 2^30 (B=%d Lmax=%d)", B, Lmax);
    return KVATTN_OK;
}

int get_workspace(int dev, cudaStream_t stream, size_t bytes, void **ptr) {
    Workspace &w = g_ws[std::make_pair(dev, stream)];
    if (w.bytes < bytes) {
        // grow at least twofold; the old buffer is retired, not freed
        size_t want = bytes < (1u << 20) ? (1u << 20) : bytes;
        if (want < 2 * w.bytes) want = 2 * w.bytes;
        void *fresh = nullptr;
        cudaError_t e = cudaMalloc(&fresh, want);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return fail(KVATTN_ERR_OOM, "workspace allocation of %zu bytes failed", want);
        }
        if (w.ptr) w.retired.push_back(w.ptr);
        w.ptr = fresh;
        w.bytes = want;
    }
    *ptr = w.ptr;
    return KVATTN_OK;
}

}  // namespace

// Entry points for the allocation-free variant (noalloc.cu): they reuse the
// checks, the descriptor encoding and the error word above without touching
// the workspace cache.
namespace kvattn {

int api_fail(int status, const char *msg) { return fail(status, "%s", msg); }

int api_check_args(const void *q, const void *k_cache, const void *v_cache,
                   const int32_t *seq_lens, const float *out, int B, int Hq, int Hkv, int D,
                   int Lmax, float scale) {
    t_last_error[0] = 0;
    if (!q || !k_cache || !v_cache || !seq_lens || !out)
        return fail(KVATTN_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return fail(KVATTN_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
    if (!std::isfinite(scale)) return fail(KVATTN_ERR_INVALID_ARG, "scale must be finite");
    return check_sizes(B, Hq, Hkv, D, Lmax);
}

int api_forced_ctas() {
    std::lock_guard<std::mutex> lk(g_mu);
    return g_force_ctas;
}

int api_encode_cache_maps(CUtensorMap *tmk, CUtensorMap *tmv, const void *k_cache,
                          const void *v_cache, int D, int Lmax, int BH, int tile) {
    int rc;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if ((rc = get_encoder())) return rc;
    }
    if ((rc = encode_cache_map(tmk, k_cache, D, Lmax, BH, tile))) return rc;
    return encode_cache_map(tmv, v_cache, D, Lmax, BH, tile);
}

int api_error_word(unsigned int **word) {
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(word), g_kvattn_device_error);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    return KVATTN_OK;
}

int api_cuda_fail(cudaError_t e, const char *what) { return cuda_fail(e, what); }

}  // namespace kvattn

namespace {

int append_rows(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                const int32_t *seq_lens, int B, int T, int Hkv, int D, int Lmax,
                kvattn_stream_t stream, const char *who, const Paged *pg = nullptr) {
    if (!k_cache || !v_cache || !k_new || !v_new || !seq_lens)
        return fail(KVATTN_ERR_INVALID_ARG, "%s: null pointer", who);
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return fail(KVATTN_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", who);
    int rc, lg = 0;
    if (pg && (rc = check_paged(*pg, Hkv, who, &lg, &Lmax))) return rc;
    if ((rc = check_sizes(B, Hkv, Hkv, D, Lmax))) return rc;
    int dev;
    if ((rc = current_device(&dev))) return rc;
    DeviceState *ds;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if ((rc = device_state(dev, &ds))) return rc;
    }
    cudaError_t e = launch_kv_append(k_cache, v_cache, k_new, v_new, seq_lens, B, T, Hkv, D,
                                     Lmax, pg ? pg->table : nullptr, lg, pg ? pg->max_blocks : 0,
                                     pg ? pg->num_blocks : 0, ds->err,
                                     reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return KVATTN_OK;
}

}  // namespace

extern "C" {

const char *kvattn_status_string(int status) {
    switch (status) {
        case KVATTN_OK: return "KVATTN_OK";
        case KVATTN_ERR_INVALID_ARG: return "KVATTN_ERR_INVALID_ARG";
        case KVATTN_ERR_UNSUPPORTED: return "KVATTN_ERR_UNSUPPORTED";
        case KVATTN_ERR_CUDA: return "KVATTN_ERR_CUDA";
        case KVATTN_ERR_OOM: return "KVATTN_ERR_OOM";
        case KVATTN_ERR_DEVICE_BOUNDS: return "KVATTN_ERR_DEVICE_BOUNDS";
        case KVATTN_ERR_TIMEOUT: return "KVATTN_ERR_TIMEOUT";
        default: return "KVATTN_ERR_UNKNOWN";
    }
}

const char *kvattn_last_error(void) { return t_last_error; }

int kvattn_set_tuning(int force_path, int num_ctas) {
    if (force_path < 0 || force_path > 2 || num_ctas < 0 || num_ctas > 65535)
        return fail(KVATTN_ERR_INVALID_ARG, "kvattn_set_tuning: value out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    g_force_path = force_path;
    g_force_ctas = num_ctas;
    return KVATTN_OK;
}

int kvattn_set_wait_limit(unsigned int polls) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_wait_limit = polls;
    return KVATTN_OK;
}

int kvattn_set_kernel_events(void *before, void *after) {
    if ((before == nullptr) != (after == nullptr))
        return fail(KVATTN_ERR_INVALID_ARG, "kvattn_set_kernel_events: give both events or neither");
    std::lock_guard<std::mutex> lk(g_mu);
    g_ev_before = static_cast<cudaEvent_t>(before);
    g_ev_after = static_cast<cudaEvent_t>(after);
    return KVATTN_OK;
}

int kvattn_get_plan(int B, int Hq, int Hkv, int D, int Lmax, int num_sms, kvattn_plan *plan) {
    t_last_error[0] = 0;
    if (!plan) return fail(KVATTN_ERR_INVALID_ARG, "plan is null");
    int rc = check_sizes(B, Hq, Hkv, D, Lmax);
    if (rc) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    if (num_sms <= 0) {
        int dev;
        if ((rc = current_device(&dev))) return rc;
        DeviceState *ds;
        if ((rc = device_state(dev, &ds))) return rc;
        num_sms = ds->num_sms;
    }
    Plan pl;
    if ((rc = make_plan(B, Hq, Hkv, D, Lmax, num_sms, &pl))) return rc;
    *plan = pl.pub;
    return KVATTN_OK;
}

int kv_append_multi(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                    const int32_t *seq_lens, int B, int T, int Hkv, int D, int Lmax,
                    kvattn_stream_t stream) {
    t_last_error[0] = 0;
    if (T < 1 || T > 64)
        return fail(KVATTN_ERR_INVALID_ARG, "kv_append_multi: T must be in [1, 64] (got %d)", T);
    return append_rows(k_cache, v_cache, k_new, v_new, seq_lens, B, T, Hkv, D, Lmax, stream,
                       "kv_append_multi");
}

int kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
              const int32_t *seq_lens, int B, int Hkv, int D, int Lmax, kvattn_stream_t stream) {
    t_last_error[0] = 0;
    return append_rows(k_cache, v_cache, k_new, v_new, seq_lens, B, 1, Hkv, D, Lmax, stream,
                       "kv_append");
}

int kv_append_paged(void *k_pool, void *v_pool, const void *k_new, const void *v_new,
                    const int32_t *block_table, const int32_t *seq_lens, int B, int T, int Hkv,
                    int D, int num_blocks, int block_size, int max_blocks,
                    kvattn_stream_t stream) {
    t_last_error[0] = 0;
    if (T < 1 || T > 64)
        return fail(KVATTN_ERR_INVALID_ARG, "kv_append_paged: T must be in [1, 64] (got %d)", T);
    const Paged pg{block_table, block_size, max_blocks, num_blocks};
    return append_rows(k_pool, v_pool, k_new, v_new, seq_lens, B, T, Hkv, D, 0, stream,
                       "kv_append_paged", &pg);
}

}  // extern "C"

namespace {

// A window no sequence reaches: the full attention.
constexpr int kFullWindow = 0x7fffffff;

// Shared body of gqa_decode_attn and gqa_decode_step (k_new != nullptr:
// append this step's rows first; seq_lens then count tokens cached before).
int run_decode(const void *q, const void *k_cache, const void *v_cache, const void *k_new,
               const void *v_new, const int32_t *seq_lens, float *out, int B, int Hq, int Hkv,
               int D, int Lmax, float scale, int window, kvattn_stream_t stream_,
               const char *who, int T = 1, const Paged *pg = nullptr) {
    t_last_error[0] = 0;
    const bool fused = k_new != nullptr || v_new != nullptr;
    if (!q || !k_cache || !v_cache || !seq_lens || !out || (fused && (!k_new || !v_new)))
        return fail(KVATTN_ERR_INVALID_ARG, "%s: null pointer", who);
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (fused && (!aligned16(k_new) || !aligned16(v_new))) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return fail(KVATTN_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned", who);
    if (!std::isfinite(scale))
        return fail(KVATTN_ERR_INVALID_ARG, "%s: scale must be finite", who);
    if (window < 1)
        return fail(KVATTN_ERR_INVALID_ARG, "%s: window must be >= 1 (got %d)", who, window);
    if (T < 1 || T > 64)
        return fail(KVATTN_ERR_INVALID_ARG, "%s: T must be in [1, 64] (got %d)", who, T);
    int rc, lg = 0;
    if (pg) {
        if ((rc = check_paged(*pg, Hkv, who, &lg, &Lmax))) return rc;
        if (D != 128 && D != 256)
            return fail(KVATTN_ERR_UNSUPPORTED, "%s: a paged cache needs D in {128, 256} (D=%d)", who, D);
    }
    if ((rc = check_sizes(B, Hq, Hkv, D, Lmax))) return rc;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

    int dev;
    if ((rc = current_device(&dev))) return rc;
    DeviceState *ds;
    Plan pl;
    void *ws = nullptr;
    unsigned int wait_limit = 0;
    cudaEvent_t ev_before = nullptr, ev_after = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        wait_limit = g_wait_limit;
        ev_before = g_ev_before;
        ev_after = g_ev_after;
        if ((rc = device_state(dev, &ds))) return rc;
        if ((rc = get_encoder())) return rc;
        if ((rc = make_plan(B, Hq, Hkv, D, Lmax, ds->num_sms, &pl, T))) return rc;
        if (pg && pl.pub.path != 2)
            return fail(KVATTN_ERR_UNSUPPORTED, "%s: a paged cache needs the tensor-core path", who);
        if ((rc = get_workspace(dev, stream, (size_t)pl.pub.workspace_bytes, &ws))) return rc;
    }
    const kvattn_plan &P = pl.pub;

    CUtensorMap tmk, tmv;
    if (pg) {
        const long long rows = (long long)pg->num_blocks * Hkv;
        if ((rc = encode_pool_map(&tmk, k_cache, D, pg->block_size, rows))) return rc;
        if ((rc = encode_pool_map(&tmv, v_cache, D, pg->block_size, rows))) return rc;
    } else {
        if ((rc = encode_cache_map(&tmk, k_cache, D, Lmax, B * Hkv, P.tile_positions))) return rc;
        if ((rc = encode_cache_map(&tmv, v_cache, D, Lmax, B * Hkv, P.tile_positions))) return rc;
    }

    DecodeParams p = {};
    p.q = static_cast<const uint16_t *>(q);
    p.seq_lens = seq_lens;
    p.len_add = fused ? 1 : 0;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    // written only by the fused append
    p.k_cache = const_cast<uint16_t *>(static_cast<const uint16_t *>(k_cache));
    p.v_cache = const_cast<uint16_t *>(static_cast<const uint16_t *>(v_cache));
    p.out = out;
    p.ws_o = static_cast<float *>(ws);
    p.ws_ml = p.ws_o + (size_t)2 * P.num_ctas * pl.heads_per_seg * D;
    p.split = reinterpret_cast<int *>(p.ws_ml + (size_t)2 * P.num_ctas * pl.heads_per_seg * 2);
    p.err = ds->err;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.Lmax = Lmax;
    p.G = Hq / Hkv;
    p.heads_per_seg = pl.heads_per_seg;
    p.hpg = pl.hpg;
    p.head_groups = P.head_groups;
    p.tile = P.tile_positions;
    p.cost_piece = pl.cost_piece;
    // each query's window, and the positions the T queries' windows span
    // together (token t's ends T - 1 - t positions before the last)
    p.qwin = window < Lmax ? window : Lmax;
    p.window = (long long)p.qwin + T - 1 < Lmax ? p.qwin + T - 1 : Lmax;
    // a paged cache's tiles start on block boundaries: a local window's
    // first tile starts at the tile boundary before it
    p.walign = (pg && p.qwin < Lmax) ? P.tile_positions - 1 : 0;
    p.T = T;
    // bytes of one piece's q box: (64 columns x rows) per 64-column slab
    p.q_bytes = (D / 64) * (T == 1 ? pl.np : pl.hpg * T) * 128;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.block_table = pg ? pg->table : nullptr;
    p.block_lg = lg;
    p.max_blocks = pg ? pg->max_blocks : 0;
    p.num_blocks = pg ? pg->num_blocks : 0;
    p.k_scale = nullptr;
    p.v_scale = nullptr;
    p.wait_limit = wait_limit;

    cudaError_t e;
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess)
        return cuda_fail(e, "recording the event before the split-KV kernel");
    if (P.path == 2) {
        CUtensorMap tmq;
        if ((rc = encode_q_map(&tmq, q, D, B, T, Hq, pl.hpg, pl.np))) return rc;
        e = pg ? tc_prepare_paged(D, pl.np, T > 1) : tc_prepare(D, pl.np, T > 1);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        e = pg ? launch_decode_tc_paged(tmk, tmv, tmq, p, pl.np, P.num_ctas, stream)
               : launch_decode_tc(tmk, tmv, tmq, p, pl.np, P.num_ctas, stream);
    } else {
        e = fma_prepare(D, pl.heads_per_seg, P.smem_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
        e = launch_decode_fma(tmk, tmv, p, P.num_ctas, P.smem_bytes, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
    if (ev_after && (e = cudaEventRecord(ev_after, stream)) != cudaSuccess)
        return cuda_fail(e, "recording the event after the split-KV kernel");
    e = launch_combine(p, P.num_ctas, stream);
    if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    return KVATTN_OK;
}

// gqa_decode_attn over an 8-bit cache (decode_fp8.cu), D = 128 or 256;
// with k_new / v_new (gqa_decode_step_fp8) the kernel first writes this
// step's rows, quantized, at seq_lens[b] and attends over one more position.
int run_decode_fp8(const void *q, const void *k_codes, const void *v_codes, const float *k_scale,
                   const float *v_scale, const int32_t *seq_lens, float *out, int B, int Hq,
                   int Hkv, int D, int Lmax, float scale, kvattn_stream_t stream_,
                   const void *k_new = nullptr, const void *v_new = nullptr) {
    const bool fused = k_new != nullptr || v_new != nullptr;
    const char *who = fused ? "gqa_decode_step_fp8" : "gqa_decode_attn_fp8";
    t_last_error[0] = 0;
    if (!q || !k_codes || !v_codes || !k_scale || !v_scale || !seq_lens || !out ||
        (fused && (!k_new || !v_new)))
        return fail(KVATTN_ERR_INVALID_ARG, "%s: null pointer", who);
    if (!aligned16(q) || !aligned16(k_codes) || !aligned16(v_codes) || !aligned16(out) ||
        (fused && (!aligned16(k_new) || !aligned16(v_new))) ||
        (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return fail(KVATTN_ERR_INVALID_ARG, "%s: pointers must be 16-byte aligned (scales 4)", who);
    if (!std::isfinite(scale)) return fail(KVATTN_ERR_INVALID_ARG, "%s: scale must be finite", who);
    int rc = check_sizes(B, Hq, Hkv, D, Lmax);
    if (rc) return rc;
    if (D != 128 && D != 256)
        return fail(KVATTN_ERR_UNSUPPORTED,
                    "%s: the 8-bit kernel reads 128-code rows per copy and needs D = 128 or 256 "
                    "(D=%d)", who, D);
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int dev;
    if ((rc = current_device(&dev))) return rc;
    DeviceState *ds;
    Plan pl;
    void *ws = nullptr;
    cudaEvent_t ev_before = nullptr, ev_after = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        ev_before = g_ev_before;
        ev_after = g_ev_after;
        if ((rc = device_state(dev, &ds))) return rc;
        if ((rc = get_encoder())) return rc;
        const int saved = g_force_path;
        g_force_path = 2;  // the plan of the tensor-core kernel (heads per pass, grid)
        rc = make_plan(B, Hq, Hkv, D, Lmax, ds->num_sms, &pl);
        g_force_path = saved;
        if (rc) return rc;
        if ((rc = get_workspace(dev, stream, (size_t)pl.pub.workspace_bytes, &ws))) return rc;
    }
    const kvattn_plan &P = pl.pub;
    CUtensorMap tmk, tmv;
    if ((rc = encode_fp8_map(&tmk, k_codes, D, Lmax, B * Hkv, P.tile_positions))) return rc;
    if ((rc = encode_fp8_map(&tmv, v_codes, D, Lmax, B * Hkv, P.tile_positions))) return rc;

    DecodeParams p = {};
    memset(&p, 0, sizeof p);
    p.q = static_cast<const uint16_t *>(q);
    p.seq_lens = seq_lens;
    p.len_add = fused ? 1 : 0;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    // the codes (one byte each), written only by the fused append
    p.k_cache = const_cast<uint16_t *>(static_cast<const uint16_t *>(k_codes));
    p.v_cache = const_cast<uint16_t *>(static_cast<const uint16_t *>(v_codes));
    p.out = out;
    p.ws_o = static_cast<float *>(ws);
    p.ws_ml = p.ws_o + (size_t)2 * P.num_ctas * pl.heads_per_seg * D;
    p.split = reinterpret_cast<int *>(p.ws_ml + (size_t)2 * P.num_ctas * pl.heads_per_seg * 2);
    p.err = ds->err;
    p.B = B; p.Hq = Hq; p.Hkv = Hkv; p.D = D; p.Lmax = Lmax;
    p.G = Hq / Hkv;
    p.heads_per_seg = pl.heads_per_seg;
    p.hpg = pl.hpg;
    p.head_groups = P.head_groups;
    p.tile = P.tile_positions;
    // a tile carries half the bytes of a bf16 tile; a piece's fixed work
    // weighs twice as many tiles
    p.cost_piece = 2 * pl.cost_piece;
    p.window = Lmax;
    p.qwin = Lmax;
    p.walign = 0;
    p.T = 1;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    cudaError_t e;
    if (ev_before && (e = cudaEventRecord(ev_before, stream)) != cudaSuccess)
        return cuda_fail(e, "recording the event before the split-KV kernel");
    e = launch_decode_q8(tmk, tmv, p, pl.np, P.num_ctas, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fp8 decode kernel launch");
    if (ev_after && (e = cudaEventRecord(ev_after, stream)) != cudaSuccess)
        return cuda_fail(e, "recording the event after the split-KV kernel");
    e = launch_combine(p, P.num_ctas, stream);
    if (e != cudaSuccess) return cuda_fail(e, "combine kernel launch");
    return KVATTN_OK;
}

}  // namespace

extern "C" {

int gqa_decode_attn(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *seq_lens, float *out, int B, int Hq, int Hkv, int D, int Lmax,
                    float scale, kvattn_stream_t stream) {
    return run_decode(q, k_cache, v_cache, nullptr, nullptr, seq_lens, out, B, Hq, Hkv, D, Lmax,
                      scale, Lmax, stream, "gqa_decode_attn");
}

int gqa_decode_attn_multi(const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *seq_lens, float *out, int B, int T, int Hq, int Hkv,
                          int D, int Lmax, float scale, kvattn_stream_t stream) {
    return run_decode(q, k_cache, v_cache, nullptr, nullptr, seq_lens, out, B, Hq, Hkv, D, Lmax,
                      scale, Lmax, stream, "gqa_decode_attn_multi", T);
}

int gqa_decode_attn_window(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *seq_lens, float *out, int B, int Hq, int Hkv, int D,
                           int Lmax, float scale, int window, kvattn_stream_t stream) {
    return run_decode(q, k_cache, v_cache, nullptr, nullptr, seq_lens, out, B, Hq, Hkv, D, Lmax,
                      scale, window, stream, "gqa_decode_attn_window");
}

int gqa_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache,
                    void *v_cache, const int32_t *seq_lens, float *out, int B, int Hq, int Hkv,
                    int D, int Lmax, float scale, kvattn_stream_t stream) {
    if (!k_new || !v_new) {
        t_last_error[0] = 0;
        return fail(KVATTN_ERR_INVALID_ARG, "gqa_decode_step: null pointer");
    }
    return run_decode(q, k_cache, v_cache, k_new, v_new, seq_lens, out, B, Hq, Hkv, D, Lmax,
                      scale, Lmax, stream, "gqa_decode_step");
}

int gqa_decode_step_window(const void *q, const void *k_new, const void *v_new, void *k_cache,
                           void *v_cache, const int32_t *seq_lens, float *out, int B, int Hq,
                           int Hkv, int D, int Lmax, float scale, int window,
                           kvattn_stream_t stream) {
    if (!k_new || !v_new) {
        t_last_error[0] = 0;
        return fail(KVATTN_ERR_INVALID_ARG, "gqa_decode_step_window: null pointer");
    }
    return run_decode(q, k_cache, v_cache, k_new, v_new, seq_lens, out, B, Hq, Hkv, D, Lmax,
                      scale, window, stream, "gqa_decode_step_window");
}

int gqa_decode_attn_paged(const void *q, const void *k_pool, const void *v_pool,
                          const int32_t *block_table, const int32_t *seq_lens, float *out, int B,
                          int T, int Hq, int Hkv, int D, int num_blocks, int block_size,
                          int max_blocks, float scale, kvattn_stream_t stream) {
    const Paged pg{block_table, block_size, max_blocks, num_blocks};
    return run_decode(q, k_pool, v_pool, nullptr, nullptr, seq_lens, out, B, Hq, Hkv, D, 0, scale,
                      kFullWindow, stream, "gqa_decode_attn_paged", T, &pg);
}

int gqa_decode_step_paged(const void *q, const void *k_new, const void *v_new, void *k_pool,
                          void *v_pool, const int32_t *block_table, const int32_t *seq_lens,
                          float *out, int B, int Hq, int Hkv, int D, int num_blocks,
                          int block_size, int max_blocks, float scale, kvattn_stream_t stream) {
    if (!k_new || !v_new) {
        t_last_error[0] = 0;
        return fail(KVATTN_ERR_INVALID_ARG, "gqa_decode_step_paged: null pointer");
    }
    const Paged pg{block_table, block_size, max_blocks, num_blocks};
    return run_decode(q, k_pool, v_pool, k_new, v_new, seq_lens, out, B, Hq, Hkv, D, 0, scale,
                      kFullWindow, stream, "gqa_decode_step_paged", 1, &pg);
}

int gqa_decode_attn_multi_window(const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *seq_lens, float *out, int B, int T, int Hq,
                                 int Hkv, int D, int Lmax, float scale, int window,
                                 kvattn_stream_t stream) {
    return run_decode(q, k_cache, v_cache, nullptr, nullptr, seq_lens, out, B, Hq, Hkv, D, Lmax,
                      scale, window, stream, "gqa_decode_attn_multi_window", T);
}

int gqa_decode_attn_paged_window(const void *q, const void *k_pool, const void *v_pool,
                                 const int32_t *block_table, const int32_t *seq_lens, float *out,
                                 int B, int T, int Hq, int Hkv, int D, int num_blocks,
                                 int block_size, int max_blocks, float scale, int window,
                                 kvattn_stream_t stream) {
    const Paged pg{block_table, block_size, max_blocks, num_blocks};
    return run_decode(q, k_pool, v_pool, nullptr, nullptr, seq_lens, out, B, Hq, Hkv, D, 0, scale,
                      window, stream, "gqa_decode_attn_paged_window", T, &pg);
}

int gqa_decode_step_paged_window(const void *q, const void *k_new, const void *v_new,
                                 void *k_pool, void *v_pool, const int32_t *block_table,
                                 const int32_t *seq_lens, float *out, int B, int Hq, int Hkv,
                                 int D, int num_blocks, int block_size, int max_blocks,
                                 float scale, int window, kvattn_stream_t stream) {
    if (!k_new || !v_new) {
        t_last_error[0] = 0;
        return fail(KVATTN_ERR_INVALID_ARG, "gqa_decode_step_paged_window: null pointer");
    }
    const Paged pg{block_table, block_size, max_blocks, num_blocks};
    return run_decode(q, k_pool, v_pool, k_new, v_new, seq_lens, out, B, Hq, Hkv, D, 0, scale,
                      window, stream, "gqa_decode_step_paged_window", 1, &pg);
}

int gqa_decode_attn_fp8(const void *q, const void *k_codes, const void *v_codes,
                        const float *k_scale, const float *v_scale, const int32_t *seq_lens,
                        float *out, int B, int Hq, int Hkv, int D, int Lmax, float scale,
                        kvattn_stream_t stream) {
    return run_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, seq_lens, out, B, Hq, Hkv, D,
                          Lmax, scale, stream);
}

int gqa_decode_step_fp8(const void *q, const void *k_new, const void *v_new, void *k_codes,
                        void *v_codes, float *k_scale, float *v_scale, const int32_t *seq_lens,
                        float *out, int B, int Hq, int Hkv, int D, int Lmax, float scale,
                        kvattn_stream_t stream) {
    if (!k_new || !v_new) {
        t_last_error[0] = 0;
        return fail(KVATTN_ERR_INVALID_ARG, "gqa_decode_step_fp8: null pointer");
    }
    return run_decode_fp8(q, k_codes, v_codes, k_scale, v_scale, seq_lens, out, B, Hq, Hkv, D,
                          Lmax, scale, stream, k_new, v_new);
}

int kv_quantize_fp8(const void *src, void *codes, float *scales, long long rows, int D,
                    kvattn_stream_t stream) {
    t_last_error[0] = 0;
    if (!src || !codes || !scales) return fail(KVATTN_ERR_INVALID_ARG, "kv_quantize_fp8: null pointer");
    if (!aligned16(src) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3u))
        return fail(KVATTN_ERR_INVALID_ARG, "kv_quantize_fp8: pointers must be 16-byte aligned (scales 4)");
    if (rows < 0 || rows > (1LL << 40))
        return fail(KVATTN_ERR_INVALID_ARG, "kv_quantize_fp8: rows out of range");
    if (D != 64 && D != 128 && D != 256)
        return fail(KVATTN_ERR_UNSUPPORTED, "kv_quantize_fp8: D=%d not in {64, 128, 256}", D);
    if ((rows + 3) / 4 > 0x7fffffffLL)
        return fail(KVATTN_ERR_UNSUPPORTED, "kv_quantize_fp8: too many rows for one launch");
    cudaError_t e = launch_quantize_fp8(src, codes, scales, rows, D,
                                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    return KVATTN_OK;
}

int kv_append_fp8(void *k_codes, void *v_codes, float *k_scale, float *v_scale,
                  const void *k_new, const void *v_new, const int32_t *seq_lens, int B, int Hkv,
                  int D, int Lmax, kvattn_stream_t stream) {
    t_last_error[0] = 0;
    if (!k_codes || !v_codes || !k_scale || !v_scale || !k_new || !v_new || !seq_lens)
        return fail(KVATTN_ERR_INVALID_ARG, "kv_append_fp8: null pointer");
    if (!aligned16(k_codes) || !aligned16(v_codes) || !aligned16(k_new) || !aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return fail(KVATTN_ERR_INVALID_ARG, "kv_append_fp8: pointers must be 16-byte aligned (scales 4)");
    int rc = check_sizes(B, Hkv, Hkv, D, Lmax);
    if (rc) return rc;
    int dev;
    if ((rc = current_device(&dev))) return rc;
    DeviceState *ds;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if ((rc = device_state(dev, &ds))) return rc;
    }
    cudaError_t e = launch_kv_append_fp8(k_codes, v_codes, k_scale, v_scale, k_new, v_new, seq_lens,
                                         B, Hkv, D, Lmax, ds->err,
                                         reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "fp8 append launch");
    return KVATTN_OK;
}

int kvattn_check_device_error(kvattn_stream_t stream) {
    t_last_error[0] = 0;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    unsigned int word = 0;
    e = cudaMemcpyFromSymbol(&word, g_kvattn_device_error, sizeof word);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (word) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_kvattn_device_error, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        return fail((int)word, "device reported %s", kvattn_status_string((int)word));
    }
    return KVATTN_OK;
}

void kvattn_release(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto &kv : g_ws) {
        cudaSetDevice(kv.first.first);
        if (kv.second.ptr) cudaFree(kv.second.ptr);
        for (void *old : kv.second.retired) cudaFree(old);
    }
    g_ws.clear();
    cudaSetDevice(cur);
}

}  // extern "C"
