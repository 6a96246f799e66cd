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
#include "dispatch_common.cuh"

namespace ep {
namespace {

using namespace mv;

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

// Destination rows of token t's picks into s_dst.  For the masked layout the
// expert-offset table is staged in shared memory by the whole block at the
// same time as the picks are read (one round of global loads, not two).
// Every thread calls it.
template <int NT>
__device__ __forceinline__ void load_dests(const MoveArgs& a, int t, long long* s_dst,
                                           int* s_eoff) {
    if (a.layout == 1) {
        for (int e = threadIdx.x; e < a.E; e += NT) s_eoff[e] = __ldg(a.expert_offsets + e);
        int p = -1, e = -1;
        if (threadIdx.x < a.K) {
            p = __ldg(a.pos + (size_t)t * a.K + threadIdx.x);
            e = __ldg(a.topk_idx + (size_t)t * a.K + threadIdx.x);
        }
        __syncthreads();
        if (threadIdx.x < a.K) {
            long long row = -1;
            if (p >= 0 && e >= 0 && e < a.E) {
                const int slot = p - s_eoff[e];
                if (slot >= 0 && slot < a.cap) row = (long long)e * a.cap + slot;
            }
            s_dst[threadIdx.x] = row;
        }
    } else if (threadIdx.x < a.K) {
        s_dst[threadIdx.x] = dest_row(a, t, threadIdx.x);
    }
    __syncthreads();
}

template <int NT, int U>
__global__ void __launch_bounds__(NT) dispatch_bf16_kernel(MoveArgs a) {
    __shared__ long long s_dst[kMaxK];
    __shared__ int s_eoff[kMaxE];
    pdl_prologue();
    const int t = blockIdx.x;
    load_dests<NT>(a, t, s_dst, s_eoff);
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

// Each thread owns 16 consecutive values; 8 lanes make one 128-column scale
// block.  One 16-byte code store per destination, and one scale store per
// block and destination (lane 0 of the 8).
template <int NT, int U>
__global__ void __launch_bounds__(NT) dispatch_fp8_kernel(MoveArgs a) {
    __shared__ long long s_dst[kMaxK];
    __shared__ int s_eoff[kMaxE];
    pdl_prologue();
    const int t = blockIdx.x;
    load_dests<NT>(a, t, s_dst, s_eoff);
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
            sc[u] = block_scale(amax16(lo[u], hi[u]));
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
