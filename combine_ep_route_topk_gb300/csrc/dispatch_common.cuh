// Row-moving helpers shared by the dispatch kernels (dispatch.cu) and the
// fused layout + dispatch kernel (layout_dispatch.cu): bf16 unpacking and the
// FP8 E4M3 1x128 block quantisation ("Expert Parallelism" (SGLang docs),
// deep_gemm row: FP8 block-wise quantisation).  A 128-column scale block is 8
// lanes x 16 values; amax = max |x| over the block, scale = amax / 448 by IEEE
// division (1 when amax == 0), code = E4M3(x / scale) by IEEE division and
// the hardware round-to-nearest-even satfinite conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ep_kernels.cuh"

namespace ep {
namespace mv {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two values -> two E4M3 codes, low byte = first value.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// E4M3 codes of 16 values as 16 bytes (value j in byte j).
__device__ __forceinline__ uint4 quantize16(const uint4& lo, const uint4& hi, float scale) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t p[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        p[j] = e4m3x2(__fdiv_rn(bf16_lo(w[j]), scale), __fdiv_rn(bf16_hi(w[j]), scale));
    return make_uint4(p[0] | (p[1] << 16), p[2] | (p[3] << 16), p[4] | (p[5] << 16),
                      p[6] | (p[7] << 16));
}

__device__ __forceinline__ float amax16(const uint4& lo, const uint4& hi) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    float m = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[j])), fabsf(bf16_hi(w[j]))));
    return m;
}

// Scale of one 128-column block from the amax of this lane's 16 values: the
// amax of the 8 lanes (an aligned group of the warp), every lane taking part.
__device__ __forceinline__ float block_scale(float amax) {
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    return (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
}

}  // namespace mv
}  // namespace ep
