// Dispatch for sm_103a: "Anatomy of a High-Performance EP Kernel", "Dispatch"
// -- gather each expert's tokens into one dense buffer for the grouped GEMM;
// "Expert Parallelism" (SGLang docs), deep_gemm row -- contiguous layout for
// prefill, masked fixed-capacity layout for decode, FP8 block-wise
// quantisation.
//
// On one GPU the all-to-all is an HBM scatter.  One block per token reads
// the token's row once (16-byte streaming loads, all of a thread's vectors in
// flight before any store) and writes it to the K destination rows
// (16-byte stores for bf16, 8-byte for FP8 codes).  The FP8 variant
// quantises once per token: a 128-column block is 16 lanes x 8 values, its
// amax is a 4-step shuffle reduction within the half-warp, scale = amax/448
// and x/scale use IEEE division, and the E4M3 conversion is the hardware
// round-to-nearest-even satfinite cvt.  Bytes moved per token:
// H*2 read + K*(H*b_out + scales) written; the kernel is HBM-bound.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Destination row of pick (t, k), or -1 when the pick is not delivered.
__device__ __forceinline__ long long dest_row(const MoveArgs& a, int t, int k) {
    const int p = __ldg(a.pos + (size_t)t * a.K + k);
    const int e = __ldg(a.topk_idx + (size_t)t * a.K + k);
    if (p < 0 || e < 0 || e >= a.E) return -1;
    if (a.layout == 0) return (p < a.N * a.K) ? (long long)p : -1;
    const int slot = p - __ldg(a.expert_offsets + e);
    if (slot < 0 || slot >= a.cap) return -1;
    return (long long)e * a.cap + slot;
}

template <int NT, int U>
__global__ void __launch_bounds__(NT) dispatch_bf16_kernel(MoveArgs a) {
    __shared__ long long s_dst[kMaxK];
    const int t = blockIdx.x;
    if (threadIdx.x < a.K) s_dst[threadIdx.x] = dest_row(a, t, threadIdx.x);
    __syncthreads();
    const int V = a.H >> 3;  // 16-byte vectors per row
    const uint4* src = reinterpret_cast<const uint4*>(a.src) + (size_t)t * V;
    uint4* dst = reinterpret_cast<uint4*>(a.dst);
    for (int c0 = threadIdx.x; c0 < V; c0 += NT * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * NT;
            if (c < V) v[u] = __ldcs(src + c);
        }
        for (int k = 0; k < a.K; ++k) {
            const long long row = s_dst[k];
            if (row < 0) continue;
            uint4* d = dst + row * V;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT;
                if (c < V) __stcs(d + c, v[u]);
            }
        }
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two values -> two E4M3 codes, low byte = first value.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

template <int NT, int U>
__global__ void __launch_bounds__(NT) dispatch_fp8_kernel(MoveArgs a) {
    __shared__ long long s_dst[kMaxK];
    const int t = blockIdx.x;
    if (threadIdx.x < a.K) s_dst[threadIdx.x] = dest_row(a, t, threadIdx.x);
    __syncthreads();
    const int V = a.H >> 3;   // 8-value vectors per row; 16 per 128-block
    const int SB = a.H >> 7;  // scale blocks per row
    const uint4* src = reinterpret_cast<const uint4*>(a.src) + (size_t)t * V;
    uint2* dst = reinterpret_cast<uint2*>(a.dst);
    const bool lead = (threadIdx.x & 15) == 0;
    const int lane = threadIdx.x & 31;
    // warp-uniform trip count: every lane takes part in the half-warp shuffles
    for (int c0 = threadIdx.x; c0 - lane < V; c0 += NT * U) {
        uint4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * NT;
            v[u] = (c < V) ? __ldcs(src + c) : make_uint4(0, 0, 0, 0);
        }
        uint2 q[U];
        float sc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
            float f[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                f[2 * j] = bf16_lo(w[j]);
                f[2 * j + 1] = bf16_hi(w[j]);
            }
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
            const float scale = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
            uint32_t p[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                p[j] = e4m3x2(__fdiv_rn(f[2 * j], scale), __fdiv_rn(f[2 * j + 1], scale));
            q[u] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
            sc[u] = scale;
        }
        for (int k = 0; k < a.K; ++k) {
            const long long row = s_dst[k];
            if (row < 0) continue;
            uint2* d = dst + row * V;
            float* srow = a.scales + row * SB;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT;
                if (c < V) {
                    __stcs(d + c, q[u]);
                    if (lead) __stcs(srow + (c >> 4), sc[u]);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_dispatch(const MoveArgs& a, cudaStream_t s) {
    if (a.N == 0) return cudaSuccess;
    if (a.dtype == 0) dispatch_bf16_kernel<128, 8><<<a.N, 128, 0, s>>>(a);
    else dispatch_fp8_kernel<128, 4><<<a.N, 128, 0, s>>>(a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace ep
