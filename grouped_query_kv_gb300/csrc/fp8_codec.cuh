// fp8_codec.cuh -- the row quantizer of the 8-bit KV cache, shared by the
// stand-alone writers (kv_fp8.cu) and the fused append of the 8-bit
// attention kernel (decode_fp8.cu), so that both write the same bytes.
// A cached row (one position of one K/V head, D values) is stored as D E4M3
// codes and one fp32 scale ("The Basics of Transformer Inference", item
// "Quantization"; "Machine Learning Engineering and AI Systems at Scale",
// section "Quantization"):
//     scale  = absmax(row) / 448   (1 for an all-zero row),
//     code_d = E4M3(row_d / scale), nearest with ties to even, saturating,
// both divisions IEEE binary32.
#pragma once

#include <cstdint>

namespace kvattn {

// Two binary32 values -> two E4M3 codes, a in the low byte.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float a, float b) {
    uint16_t r;
    // the first source goes to the upper byte
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
    return r;
}

// Quantize one row of D bf16 values held by a warp (D / 32 values per
// lane, lane l holding values [l * D/32, (l+1) * D/32)).
template <int VPL>
__device__ __forceinline__ void quantize_row_warp(const uint16_t *src, uint8_t *codes,
                                                  float *scale, int lane) {
    float x[VPL];
    if (VPL == 8) {
        const uint4 raw = reinterpret_cast<const uint4 *>(src)[lane];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            x[2 * u] = __uint_as_float(w[u] << 16);
            x[2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u);
        }
    } else if (VPL == 4) {
        const uint2 raw = reinterpret_cast<const uint2 *>(src)[lane];
        x[0] = __uint_as_float(raw.x << 16);
        x[1] = __uint_as_float(raw.x & 0xFFFF0000u);
        x[2] = __uint_as_float(raw.y << 16);
        x[3] = __uint_as_float(raw.y & 0xFFFF0000u);
    } else {
        const uint32_t raw = reinterpret_cast<const uint32_t *>(src)[lane];
        x[0] = __uint_as_float(raw << 16);
        x[1] = __uint_as_float(raw & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int v = 0; v < VPL; ++v) amax = fmaxf(amax, fabsf(x[v]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
    uint32_t packed[VPL / 4 > 0 ? VPL / 4 : 1];
#pragma unroll
    for (int v = 0; v < VPL; v += 2) {
        const uint16_t two = e4m3x2_from_f32(__fdiv_rn(x[v], s), __fdiv_rn(x[v + 1], s));
        if (VPL >= 4) {
            if ((v & 2) == 0)
                packed[v / 4] = two;
            else
                packed[v / 4] |= (uint32_t)two << 16;
        } else {
            reinterpret_cast<uint16_t *>(codes)[lane] = two;
        }
    }
    if (VPL == 8)
        reinterpret_cast<uint2 *>(codes)[lane] = make_uint2(packed[0], packed[1]);
    else if (VPL == 4)
        reinterpret_cast<uint32_t *>(codes)[lane] = packed[0];
    if (lane == 0) *scale = s;
}

}  // namespace kvattn
