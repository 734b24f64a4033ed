// kv_fp8.cu -- writing an 8-bit KV cache ("The Basics of Transformer
// Inference", item "Quantization"; "Machine Learning Engineering and AI
// Systems at Scale", section "Quantization": FP8 E4M3).  Each cached row
// (one position of one K/V head, D values) is stored as D E4M3 codes and
// one fp32 scale:
//     scale  = absmax(row) / 448   (1 for an all-zero row),
//     code_d = E4M3(row_d / scale), nearest with ties to even, saturating
// -- both divisions IEEE binary32 (so the codes are a deterministic
// function of the bf16 row).  One warp per row; D in {64, 128, 256}.
#include <cuda_bf16.h>

#include "fp8_codec.cuh"
#include "internal.h"

namespace kvattn {

namespace {

template <int D>
__global__ void __launch_bounds__(128)
    quantize_rows_kernel(const uint16_t *__restrict__ src, uint8_t *__restrict__ codes,
                         float *__restrict__ scales, long long rows) {
    const long long r = (long long)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (r >= rows) return;
    quantize_row_warp<D / 32>(src + r * D, codes + r * D, scales + r, threadIdx.x & 31);
}

// The new token's rows (b, kvh) -> position seq_lens[b] of the 8-bit cache.
template <int D>
__global__ void __launch_bounds__(128)
    kv_append_fp8_kernel(uint8_t *__restrict__ k_codes, uint8_t *__restrict__ v_codes,
                         float *__restrict__ k_scale, float *__restrict__ v_scale,
                         const uint16_t *__restrict__ k_new, const uint16_t *__restrict__ v_new,
                         const int32_t *__restrict__ seq_lens, int B, int Hkv, int Lmax,
                         unsigned int *err) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int row = blockIdx.x * 4 + (threadIdx.x >> 5);  // (b, kvh)
    const int lane = threadIdx.x & 31;
    if (row >= B * Hkv) return;
    const int b = row / Hkv;
    const int pos = seq_lens[b];
    if (pos < 0 || pos >= Lmax) {
        if (lane == 0) atomicCAS(err, 0u, (unsigned int)DEV_ERR_BOUNDS);
        return;
    }
    const size_t dst = (size_t)row * Lmax + pos;
    quantize_row_warp<D / 32>(k_new + (size_t)row * D, k_codes + dst * D, k_scale + dst, lane);
    quantize_row_warp<D / 32>(v_new + (size_t)row * D, v_codes + dst * D, v_scale + dst, lane);
}

}  // namespace

cudaError_t launch_quantize_fp8(const void *src, void *codes, float *scales, long long rows,
                                int D, cudaStream_t stream) {
    const long long blocks = (rows + 3) / 4;
    if (blocks == 0) return cudaSuccess;
    const auto *s = static_cast<const uint16_t *>(src);
    auto *c = static_cast<uint8_t *>(codes);
    switch (D) {
        case 64: quantize_rows_kernel<64><<<(unsigned)blocks, 128, 0, stream>>>(s, c, scales, rows); break;
        case 128: quantize_rows_kernel<128><<<(unsigned)blocks, 128, 0, stream>>>(s, c, scales, rows); break;
        case 256: quantize_rows_kernel<256><<<(unsigned)blocks, 128, 0, stream>>>(s, c, scales, rows); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_kv_append_fp8(void *k_codes, void *v_codes, float *k_scale, float *v_scale,
                                 const void *k_new, const void *v_new, const int32_t *seq_lens,
                                 int B, int Hkv, int D, int Lmax, unsigned int *err,
                                 cudaStream_t stream) {
    const int blocks = (B * Hkv + 3) / 4;
    auto *kc = static_cast<uint8_t *>(k_codes);
    auto *vc = static_cast<uint8_t *>(v_codes);
    const auto *kn = static_cast<const uint16_t *>(k_new);
    const auto *vn = static_cast<const uint16_t *>(v_new);
    switch (D) {
        case 64: kv_append_fp8_kernel<64><<<blocks, 128, 0, stream>>>(kc, vc, k_scale, v_scale, kn, vn, seq_lens, B, Hkv, Lmax, err); break;
        case 128: kv_append_fp8_kernel<128><<<blocks, 128, 0, stream>>>(kc, vc, k_scale, v_scale, kn, vn, seq_lens, B, Hkv, Lmax, err); break;
        case 256: kv_append_fp8_kernel<256><<<blocks, 128, 0, stream>>>(kc, vc, k_scale, v_scale, kn, vn, seq_lens, B, Hkv, Lmax, err); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace kvattn
