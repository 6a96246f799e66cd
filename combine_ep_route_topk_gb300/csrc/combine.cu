// Combine for sm_103a: "Anatomy of a High-Performance EP Kernel" -- after the
// expert GEMM, bring each token's K expert outputs home; "Expert Parallelism"
// (SGLang docs), framework overview -- Dispatcher.combine produces
// final_hidden_states.
//
//   out[t] = bf16_rn( sum_{k=0..K-1} w[t,k] * y[row(t,k)] )
//
// fp32 accumulation, one fused multiply-add per pick in pick order (so the
// result is reproducible bit for bit), undelivered picks skipped.  One block
// per token (256 threads, picked by a block-size sweep; 128 for 1024..8192
// tokens); each thread owns
// 16-byte column vectors and issues the loads of all K rows before the FMAs (K templated for 1/2/4/8, so up to 8 x 16 B per
// vector are in flight per thread).  Bytes per token: K*H*2 read + H*2
// written; HBM-bound.
#include <cuda_bf16.h>

#include "ep_kernels.cuh"

namespace ep {
namespace {

// Token counts served by 128-thread blocks; see launch_combine.
constexpr int kCombineSmallLo = 1024, kCombineSmallHi = 8192;

__device__ __forceinline__ long long src_row(const MoveArgs& a, int t, int k) {
    const int p = __ldg(a.pos + (size_t)t * a.K + k);
    const int e = __ldg(a.topk_idx + (size_t)t * a.K + k);
    if (p < 0 || e < 0 || e >= a.E) return -1;
    if (a.layout == 0) return (p < a.N * a.K) ? (long long)p : -1;
    const int slot = p - __ldg(a.expert_offsets + e);
    if (slot < 0 || slot >= a.cap) return -1;
    return (long long)e * a.cap + slot;
}

__device__ __forceinline__ void fma8(float* acc, float w, const uint4& v) {
    const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc[2 * j] = fmaf(w, __uint_as_float(x[j] << 16), acc[2 * j]);
        acc[2 * j + 1] = fmaf(w, __uint_as_float(x[j] & 0xffff0000u), acc[2 * j + 1]);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Rows of token t's picks (-1: not delivered) and their weights into s_row /
// s_w.  For the masked layout the expert-offset table is staged in shared
// memory by the whole block at the same time as the picks are read, so the
// rows need one round of global loads instead of two.  Every thread calls it.
template <int NT>
__device__ __forceinline__ void load_rows(const MoveArgs& a, int t, int K, long long* s_row,
                                          float* s_w, int* s_eoff) {
    if (a.layout == 1) {
        for (int e = threadIdx.x; e < a.E; e += NT) s_eoff[e] = __ldg(a.expert_offsets + e);
        int p = -1, e = -1;
        float w = 0.0f;
        if (threadIdx.x < K) {
            p = __ldg(a.pos + (size_t)t * a.K + threadIdx.x);
            e = __ldg(a.topk_idx + (size_t)t * a.K + threadIdx.x);
            w = __ldg(a.topk_w + (size_t)t * a.K + threadIdx.x);
        }
        __syncthreads();
        if (threadIdx.x < K) {
            long long row = -1;
            if (p >= 0 && e >= 0 && e < a.E) {
                const int slot = p - s_eoff[e];
                if (slot >= 0 && slot < a.cap) row = (long long)e * a.cap + slot;
            }
            s_row[threadIdx.x] = row;
            s_w[threadIdx.x] = w;
        }
    } else if (threadIdx.x < K) {
        s_row[threadIdx.x] = src_row(a, t, threadIdx.x);
        s_w[threadIdx.x] = __ldg(a.topk_w + (size_t)t * a.K + threadIdx.x);
    }
    __syncthreads();
}

// KC > 0: K known at compile time; KC == 0: runtime K, one row at a time.
template <int NT, int KC>
__global__ void __launch_bounds__(NT) combine_kernel(MoveArgs a) {
    __shared__ long long s_row[kMaxK];
    __shared__ float s_w[kMaxK];
    __shared__ int s_eoff[kMaxE];
    pdl_prologue();
    const int t = blockIdx.x;
    const int K = KC > 0 ? KC : a.K;
    load_rows<NT>(a, t, K, s_row, s_w, s_eoff);
    const int V = a.H >> 3;
    const uint4* y = reinterpret_cast<const uint4*>(a.src);
    uint4* out = reinterpret_cast<uint4*>(a.dst) + (size_t)t * V;
    for (int c = threadIdx.x; c < V; c += NT) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        if (KC > 0) {
            uint4 v[KC > 0 ? KC : 1];
#pragma unroll
            for (int k = 0; k < KC; ++k) {
                const long long row = s_row[k];
                v[k] = (row >= 0) ? __ldcs(y + row * V + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < KC; ++k)
                if (s_row[k] >= 0) fma8(acc, s_w[k], v[k]);
        } else {
            for (int k = 0; k < K; ++k) {
                const long long row = s_row[k];
                if (row >= 0) fma8(acc, s_w[k], __ldcs(y + row * V + c));
            }
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        __stcs(out + c, o);
    }
}

template <int NT>
cudaError_t launch_nt(const MoveArgs& a, cudaStream_t s) {
    switch (a.K) {
        case 1: return launch(combine_kernel<NT, 1>, dim3(a.N), dim3(NT), 0, s, a);
        case 2: return launch(combine_kernel<NT, 2>, dim3(a.N), dim3(NT), 0, s, a);
        case 4: return launch(combine_kernel<NT, 4>, dim3(a.N), dim3(NT), 0, s, a);
        case 8: return launch(combine_kernel<NT, 8>, dim3(a.N), dim3(NT), 0, s, a);
        default: return launch(combine_kernel<NT, 0>, dim3(a.N), dim3(NT), 0, s, a);
    }
}

}  // namespace

// Blocks of 256 threads, or of 128 for 1024..8192 tokens: a sweep on GB300
// (E = 256, K = 8, H = 7168, L2 clean, CUDA events) gave 128 / 256 threads
// 24.6 / 26.6 us at 1024 tokens, 41.0 / 45.1 at 2048, 75.8 / 77.8 at 4096
// and 151.6 / 153.6 at 8192, but 18.4 / 16.4 at 512 and 16.3 / 14.3 at 256.
// At 1024 tokens the 128-thread grid is one wave (all blocks resident), the
// 256-thread one 1.35 waves.
cudaError_t launch_combine(const MoveArgs& a, cudaStream_t s) {
    if (a.N == 0) return cudaSuccess;
    const bool small = a.N >= kCombineSmallLo && a.N <= kCombineSmallHi;
    const cudaError_t err = small ? launch_nt<128>(a, s) : launch_nt<256>(a, s);
    note_launch();
    return err;
}

}  // namespace ep
