// Route -> layout -> dispatch of a small (decode-sized) problem in two
// launches: "Anatomy of a High-Performance EP Kernel", "What we have to do"
// (route locally), "High throughput: ask first, then send" and "Dispatch";
// "Expert Parallelism" (SGLang docs), "Supported backends" (the low-latency
// mode) and the deep_gemm row (masked layout for decode).
//
// The routing kernel (route_hist_kernel) routes 8 tokens per block and writes
// each block's expert histogram H[e][c] and its exclusive prefix over experts
// P[e][c], expert-major.  These columns are all that is needed to place any
// pick, so one more kernel does the whole layout and the row copies, with no
// block waiting for another:
//   token blocks t (N of them, first in the grid): see below.
//   expert blocks e (E of them): the column H[e][.] scanned over the blocks
//       gives e's picks before any token boundary (plus the few ids of a
//       partial block), hence counts[r][e] and rank_expert_offsets[r][e];
//       sum_c P[e][c] is expert_offsets[e]; masked_m[e]; e's overflow is
//       added to the counter the routing kernel zeroed.
//   one totals block: expert_offsets[E] (the valid picks) and the -1 tail of
//       row_src.
//   token blocks t: issue the loads of the token's row first,
//       then for each pick (t, k) of expert e:
//           slot = sum_{c < t/8} H[e][c] + #{e's picks in t's block before (t, k)}
//           pos  = sum_c P[e][c] + slot       (the stable counting sort's answer)
//       write pos and row_src, and store (or quantise and store) the row to
//       its destinations, as ep_dispatch does.
// A token block reads two contiguous runs of at most 256 ints per pick (8 KB
// per token at the decode size) from L2; the expert and totals blocks are off
// the critical path.
#include "dispatch_common.cuh"
#include "layout_common.cuh"

namespace ep {
namespace {

using namespace mv;

__device__ __forceinline__ int clamp_tok(int v, int N) { return v < 0 ? 0 : (v > N ? N : v); }

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
    return v;
}

// Expert e's column of the layout.
template <int NT>
__device__ void expert_part(const RouteDispatchArgs& a, int e, int* smem) {
    const int C = a.C, E = a.E, K = a.K, N = a.N, R = a.R;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int* H = a.hist + (size_t)e * C;             // e's picks in each routing block
    const int* P = a.hist + ((size_t)E + e) * C;       // picks of lower experts in each block
    int* s_pre = smem;                       // [C+1] e's picks before block c
    int* s_o = s_pre + lay::round_up4(C + 1);  // [R+1] rank starts, then picks before them
    int* s_tmp = s_o + lay::round_up4(R + 1);  // [32]
    int eo = 0;
    for (int c = threadIdx.x; c <= C; c += NT) {
        s_pre[c] = (c == 0) ? 0 : __ldg(H + c - 1);
        if (c < C) eo += __ldg(P + c);
    }
    for (int r = threadIdx.x; r <= R; r += NT) s_o[r] = clamp_tok(__ldg(a.rank_offsets + r), N);
    eo = warp_sum(eo);
    if (lane == 0) s_tmp[warp] = eo;
    __syncthreads();
    eo = 0;
    for (int w = 0; w < NT / 32; ++w) eo += s_tmp[w];
    __syncthreads();
    lay::block_scan_inplace<NT, false>(s_pre, C + 1, s_tmp);  // inclusive: picks before c
    lay::block_scan_inplace<NT, true>(s_o, R + 1, s_tmp);     // non-decreasing rank starts
    const int total = s_pre[C];
    // picks of e among tokens < o_r: whole blocks, then the partial block
    for (int r = threadIdx.x; r <= R; r += NT) {
        const int T = s_o[r];
        const int c = T / kRouteTokensPerBlock;
        int f = s_pre[c];
        const int i1 = T * K;
#pragma unroll 8
        for (int i = c * kRouteTokensPerBlock * K; i < i1; ++i) f += (__ldg(a.topk_idx + i) == e);
        s_o[r] = f;  // only thread r reads or writes entry r from here on
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += NT) {
        a.counts[(size_t)r * E + e] = s_o[r + 1] - s_o[r];
        a.rank_expert_offsets[(size_t)r * E + e] = eo + s_o[r];
    }
    if (threadIdx.x == 0) {
        a.expert_offsets[e] = eo;
        if (a.cap > 0) {
            if (a.masked_m) a.masked_m[e] = min(total, a.cap);
            if (a.overflow && total > a.cap) atomicAdd(a.overflow, total - a.cap);
        }
    }
}

// expert_offsets[E] (the valid picks: sum_c of P[E-1][c] + H[E-1][c]) and
// row_src = -1 past them.
template <int NT>
__device__ void totals_part(const RouteDispatchArgs& a, int* smem) {
    const int C = a.C, E = a.E, NK = a.N * a.K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int v = 0;
    for (int c = threadIdx.x; c < C; c += NT)
        v += __ldg(a.hist + (size_t)(E - 1) * C + c) + __ldg(a.hist + (size_t)(2 * E - 1) * C + c);
    v = warp_sum(v);
    if (lane == 0) smem[warp] = v;
    __syncthreads();
    int total = 0;
    for (int w = 0; w < NT / 32; ++w) total += smem[w];
    if (threadIdx.x == 0) a.expert_offsets[E] = total;
    for (int p = total + threadIdx.x; p < NK; p += NT) a.row_src[p] = -1;
}

// Token t's positions: pos, row_src, and the destination row of each pick in
// s_dst (-1: not delivered).  Every thread calls it.
template <int NT>
__device__ void token_layout(const RouteDispatchArgs& a, int t, long long* s_dst) {
    const int C = a.C, E = a.E, K = a.K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c0 = t / kRouteTokensPerBlock;
    const int i0 = c0 * kRouteTokensPerBlock * K;  // first id of t's routing block
    for (int k = warp; k < K; k += NT / 32) {  // a warp per pick
        int e = __ldg(a.topk_idx + (size_t)t * K + k);  // the same address in every lane
        if (e < 0 || e >= E) e = -1;
        int before = 0, eo = 0, in = 0;
        if (e >= 0) {
            const int* H = a.hist + (size_t)e * C;        // contiguous over blocks
            const int* P = a.hist + ((size_t)E + e) * C;
#pragma unroll 4
            for (int c = lane; c < C; c += 32) {
                eo += __ldg(P + c);
                if (c < c0) before += __ldg(H + c);
            }
            for (int i = i0 + lane; i < t * K + k; i += 32) in += (__ldg(a.topk_idx + i) == e);
        }
        before = warp_sum(before + in);
        eo = warp_sum(eo);
        if (lane == 0) {
            long long dst = -1;
            int p = -1;
            if (e >= 0) {
                p = eo + before;
                a.row_src[p] = t;
                if (a.layout == 0) dst = p;
                else if (before < a.cap) dst = (long long)e * a.cap + before;
            }
            a.pos[(size_t)t * K + k] = p;
            s_dst[k] = dst;
        }
    }
    __syncthreads();
}

// At most 56 registers (9 blocks of 128 threads per SM): the decode grid of
// 1024 token blocks + 257 layout blocks then fits in one wave (8 per SM,
// at 64 registers, left 65 blocks for a second one).  Decode step in a CUDA
// graph: 55.2-55.4 -> 54.5-55.0 us.
template <int NT, int U>
__global__ void __launch_bounds__(NT, 9) route_dispatch_bf16_kernel(RouteDispatchArgs a) {
    extern __shared__ int smem[];
    __shared__ long long s_dst[kMaxK];
    pdl_prologue();
    if ((int)blockIdx.x >= a.N) {  // after the token blocks, which are on the critical path
        const int b = (int)blockIdx.x - a.N;
        if (b < a.E) expert_part<NT>(a, b, smem);
        else totals_part<NT>(a, smem);
        return;
    }
    const int t = blockIdx.x;
    const int V = a.H >> 3;  // 16-byte vectors per row
    const uint4* src = reinterpret_cast<const uint4*>(a.x) + (size_t)t * V;
    uint4* dst = reinterpret_cast<uint4*>(a.out);
    uint4 v[U];  // the row's first vectors are in flight during the layout
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int c = threadIdx.x + u * NT;
        if (c < V) v[u] = __ldcs(src + c);
    }
    token_layout<NT>(a, t, s_dst);
    for (int c0 = threadIdx.x; c0 < V; c0 += NT * U) {
        if (c0 != (int)threadIdx.x) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * NT;
                if (c < V) v[u] = __ldcs(src + c);
            }
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

template <int NT, int U>
__global__ void __launch_bounds__(NT) route_dispatch_fp8_kernel(RouteDispatchArgs a) {
    extern __shared__ int smem[];
    __shared__ long long s_dst[kMaxK];
    pdl_prologue();
    if ((int)blockIdx.x >= a.N) {  // after the token blocks, which are on the critical path
        const int b = (int)blockIdx.x - a.N;
        if (b < a.E) expert_part<NT>(a, b, smem);
        else totals_part<NT>(a, smem);
        return;
    }
    const int t = blockIdx.x;
    const int G = a.H >> 4;   // 16-value groups per row; 8 per scale block
    const int SB = a.H >> 7;  // scale blocks per row
    const uint4* src = reinterpret_cast<const uint4*>(a.x) + (size_t)t * (a.H >> 3);
    uint4* dst = reinterpret_cast<uint4*>(a.out);
    const int lane = threadIdx.x & 31;
    const bool lead = (lane & 7) == 0;
    uint4 lo[U], hi[U];
    auto load = [&](int g0) {
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
    };
    load(threadIdx.x);
    token_layout<NT>(a, t, s_dst);
    // warp-uniform trip count: every lane takes part in the 8-lane shuffles
    for (int g0 = threadIdx.x; g0 - lane < G; g0 += NT * U) {
        if (g0 != (int)threadIdx.x) load(g0);
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

bool route_dispatch_fits(int N, int E, int K, int R) {
    (void)E;
    (void)R;
    return N <= kRouteDispatchMaxTokens && (long long)N * K <= 16384;
}

size_t route_dispatch_hist_bytes(int N, int E) {
    return (size_t)2 * route_chunks(N) * E * sizeof(int32_t);
}

cudaError_t launch_route_dispatch(const RouteDispatchArgs& a, cudaStream_t s) {
    const int ints = lay::round_up4(a.C + 1) + lay::round_up4(a.R + 1) + 32;
    const size_t smem = (size_t)ints * sizeof(int);
    const dim3 grid(a.E + 1 + a.N);
    cudaError_t err;
    if (a.dtype == 0) err = launch(route_dispatch_bf16_kernel<128, 8>, grid, dim3(128), smem, s, a);
    else err = launch(route_dispatch_fp8_kernel<256, 2>, grid, dim3(256), smem, s, a);
    note_launch();
    return err;
}

}  // namespace ep
