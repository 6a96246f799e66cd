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
//
// From 4096 tokens on, the row (bf16) or its codes (FP8) are staged in shared
// memory and each destination row is written by one bulk shared-to-global
// copy (cp.async.bulk, L2 evict-first), issued by one thread per pick; the
// FP8 scales stay plain stores.  With fewer tokens the threads store the rows
// themselves: there the grid is about one wave and the staging barrier costs
// more than the bulk copies save.
#include <cstdlib>

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

// One bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// from shared to global memory, with an L2 evict-first hint: the rows are
// streamed out like the threads' __stcs stores.
__device__ __forceinline__ void bulk_store_row(void* gdst, const void* ssrc, unsigned bytes) {
    const unsigned sa = (unsigned)__cvta_generic_to_shared(ssrc);
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;"
                 :: "l"(gdst), "r"(sa), "r"(bytes), "l"(pol) : "memory");
}

// Commit this thread's bulk copies and wait until they have completed (the
// rows are written, and shared memory may be released).
__device__ __forceinline__ void bulk_commit_and_wait() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// The threads' shared-memory writes, made visible to the bulk copies, and
// then thread k < K writes destination row k from s_row.
__device__ __forceinline__ void bulk_store_dests(const long long* s_dst, int K, void* dst,
                                                 size_t row_bytes, const void* s_row) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if ((int)threadIdx.x < K) {
        const long long row = s_dst[threadIdx.x];
        if (row >= 0) {
            bulk_store_row(static_cast<unsigned char*>(dst) + row * row_bytes, s_row,
                           (unsigned)row_bytes);
            bulk_commit_and_wait();
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(NT) dispatch_bf16_bulk_kernel(MoveArgs a) {
    extern __shared__ __align__(128) unsigned char s_row[];  // H * 2 bytes
    __shared__ long long s_dst[kMaxK];
    __shared__ int s_eoff[kMaxE];
    pdl_prologue();
    const int t = blockIdx.x;
    load_dests<NT>(a, t, s_dst, s_eoff);
    const int V = a.H >> 3;
    const uint4* src = reinterpret_cast<const uint4*>(a.src) + (size_t)t * V;
    uint4* sr = reinterpret_cast<uint4*>(s_row);
    for (int c = threadIdx.x; c < V; c += NT) sr[c] = __ldcs(src + c);
    bulk_store_dests(s_dst, a.K, a.dst, (size_t)V * 16, s_row);
}

template <int NT, int U>
__global__ void __launch_bounds__(NT) dispatch_fp8_bulk_kernel(MoveArgs a) {
    extern __shared__ __align__(128) unsigned char s_codes[];  // H bytes
    __shared__ long long s_dst[kMaxK];
    __shared__ int s_eoff[kMaxE];
    pdl_prologue();
    const int t = blockIdx.x;
    load_dests<NT>(a, t, s_dst, s_eoff);
    const int G = a.H >> 4;
    const int SB = a.H >> 7;
    const uint4* src = reinterpret_cast<const uint4*>(a.src) + (size_t)t * (a.H >> 3);
    uint4* sq = reinterpret_cast<uint4*>(s_codes);
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
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int g = g0 + u * NT;
            const float sc = block_scale(amax16(lo[u], hi[u]));
            const uint4 q = quantize16(lo[u], hi[u], sc);
            if (g < G) {
                sq[g] = q;
                if (lead)
                    for (int k = 0; k < a.K; ++k) {
                        const long long row = s_dst[k];
                        if (row >= 0) __stcs(a.scales + row * SB + (g >> 3), sc);
                    }
            }
        }
    }
    bulk_store_dests(s_dst, a.K, a.dst, (size_t)a.H, s_codes);
}

constexpr int kDispatchBulkFrom = 4096;           // tokens
constexpr size_t kDispatchBulkMaxRow = 32768;     // staged bytes per block

// EP_DISPATCH_BULK=0 in the environment (read at every call) keeps the
// thread-store kernels at every size.
bool dispatch_bulk(const MoveArgs& a) {
    const char* v = std::getenv("EP_DISPATCH_BULK");
    if (v && v[0] == '0') return false;
    const size_t row = a.dtype == 0 ? (size_t)a.H * 2 : (size_t)a.H;
    return a.N >= kDispatchBulkFrom && row <= kDispatchBulkMaxRow &&
           (reinterpret_cast<uintptr_t>(a.dst) & 15u) == 0;
}

}  // namespace

cudaError_t launch_dispatch(const MoveArgs& a, cudaStream_t s) {
    if (a.N == 0) return cudaSuccess;
    cudaError_t err;
    if (dispatch_bulk(a))
        err = a.dtype == 0
                  ? launch(dispatch_bf16_bulk_kernel<128>, dim3(a.N), dim3(128), (size_t)a.H * 2, s, a)
                  : launch(dispatch_fp8_bulk_kernel<256, 2>, dim3(a.N), dim3(256), (size_t)a.H, s, a);
    else
        err = a.dtype == 0 ? launch(dispatch_bf16_kernel<128, 8>, dim3(a.N), dim3(128), 0, s, a)
                           : launch(dispatch_fp8_kernel<256, 2>, dim3(a.N), dim3(256), 0, s, a);
    note_launch();
    return err;
}

}  // namespace ep
