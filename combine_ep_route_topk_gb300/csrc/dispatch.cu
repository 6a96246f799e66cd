// Dispatch for sm_103a: "Anatomy of a High-Performance EP Kernel", "Dispatch"
// -- gather each expert's tokens into one dense buffer for the grouped GEMM;
// "Expert Parallelism" (SGLang docs), deep_gemm row -- contiguous layout for
// prefill, masked fixed-capacity layout for decode, FP8 block-wise
// quantisation.
//
// On one GPU the all-to-all is an HBM scatter.  One block per token reads
// the token's row once (16-byte streaming loads, all of a thread's vectors in
// flight before any store) and writes it to the K destination rows
// (16-byte stores).  The FP8 variant quantises once per token: a 128-column
// block is 8 lanes x 16 values, its amax a 3-step shuffle reduction within
// the 8 lanes, scale = amax/448
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
    pdl_prologue();
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

// Each thread owns 16 consecutive values; 8 lanes make one 128-column scale
// block.  One 16-byte code store per destination, and one scale store per
// block and destination (lane 0 of the 8).
template <int NT, int U>
__global__ void __launch_bounds__(NT) dispatch_fp8_kernel(MoveArgs a) {
    __shared__ long long s_dst[kMaxK];
    pdl_prologue();
    const int t = blockIdx.x;
    if (threadIdx.x < a.K) s_dst[threadIdx.x] = dest_row(a, t, threadIdx.x);
    __syncthreads();
    const int G = a.H >> 4;   // 16-value groups per row; 8 per scale block
    const int SB = a.H >> 7;  // scale blocks per row
    const uint4* src = reinterpret_cast<const uint4*>(a.src) + (size_t)t * (a.H >> 3);
    uint4* dst = reinterpret_cast<uint4*>(a.dst);
    const int lane = threadIdx.x & 31;
    const bool lead = (lane & 7) == 0;
    // warp-uniform trip count: every lane takes part in the 8-lane shuffles
    for (int g0 = threadIdx.x; g0 - lane < G; g0 += NT * U) {
        uint4 lo[U], hi[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int g = g0 + u * NT;
            if (g < G) {
                lo[u] = __ldcs(src + 2 * g);
                hi[u] = __ldcs(src + 2 * g + 1);
            } else {
                lo[u] = make_uint4(0, 0, 0, 0);
                hi[u] = lo[u];
            }
        }
        uint4 q[U];
        float sc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            float amax = amax16(lo[u], hi[u]);
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
            sc[u] = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 448.0f);
            q[u] = quantize16(lo[u], hi[u], sc[u]);
        }
        for (int k = 0; k < a.K; ++k) {
            const long long row = s_dst[k];
            if (row < 0) continue;
            uint4* d = dst + row * G;
            float* srow = a.scales + row * SB;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int g = g0 + u * NT;
                if (g < G) {
                    __stcs(d + g, q[u]);
                    if (lead) __stcs(srow + (g >> 3), sc[u]);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_dispatch(const MoveArgs& a, cudaStream_t s) {
    if (a.N == 0) return cudaSuccess;
    const cudaError_t err =
        a.dtype == 0 ? launch(dispatch_bf16_kernel<128, 8>, dim3(a.N), dim3(128), 0, s, a)
                     : launch(dispatch_fp8_kernel<256, 2>, dim3(a.N), dim3(256), 0, s, a);
    note_launch();
    return err;
}

}  // namespace ep
