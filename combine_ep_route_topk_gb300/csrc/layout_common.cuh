// Layout building blocks shared by the three layout kernels and the fused
// route + layout kernel: chunk table, block scans, and the stable per-chunk
// scatter of positions.  "Anatomy of a High-Performance EP Kernel", "High
// throughput: ask first, then send" and "Dispatch".
//
// Reads of data another block may have written earlier in the same kernel
// (topk_idx, chunk histograms, totals, rank offsets) use ld.global.cg, which
// is served by L2 and never by a stale L1 line.
#pragma once

#include <climits>

#include "ep_kernels.cuh"

namespace ep {
namespace lay {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kNT = 256;  // threads of the hist / scatter / fused blocks
constexpr int kWarps = kNT / 32;

// In-place inclusive scan (sum, or running max) of s[0..n) by all NT threads
// of the block; s_tmp holds NT/32 ints.
template <int NT, bool MAX>
__device__ void block_scan_inplace(int* s, int n, int* s_tmp) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + NT - 1) / NT;
    const int lo = tid * per, hi = min(n, lo + per);
    int acc = MAX ? INT_MIN : 0;
    for (int i = lo; i < hi; ++i) {
        acc = MAX ? max(acc, s[i]) : acc + s[i];
        s[i] = acc;
    }
    int v = acc;  // inclusive scan of the thread totals within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, v, off);
        if (lane >= off) v = MAX ? max(v, o) : v + o;
    }
    if (lane == 31) s_tmp[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = (lane < NT / 32) ? s_tmp[lane] : (MAX ? INT_MIN : 0);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, w, off);
            if (lane >= off) w = MAX ? max(w, o) : w + o;
        }
        if (lane < NT / 32) s_tmp[lane] = w;
    }
    __syncthreads();
    int excl = __shfl_up_sync(kFull, v, 1);
    if (lane == 0) excl = MAX ? INT_MIN : 0;
    if (warp > 0) excl = MAX ? max(excl, s_tmp[warp - 1]) : excl + s_tmp[warp - 1];
    for (int i = lo; i < hi; ++i) s[i] = MAX ? max(excl, s[i]) : excl + s[i];
    __syncthreads();
}

// Rank token bounds s_m[0..R] (clamped to [0,N] and made non-decreasing, so
// ranks never overlap whatever rank_offsets holds) and chunk starts
// s_tab[0..R] (s_tab[R] = number of chunks).
template <int NT>
__device__ void build_chunk_table(const int32_t* __restrict__ ro, int R, int N, int C, int* s_m,
                                  int* s_tab, int* s_tmp) {
    if (R < 32) {  // one warp: shuffle scans over the R + 1 <= 32 entries
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int b = 0;
            if (lane <= R) {
                const int v = ro[lane];
                b = v < 0 ? 0 : (v > N ? N : v);
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(kFull, b, off);
                if (lane >= off) b = max(b, o);
            }
            const int prev = __shfl_up_sync(kFull, b, 1);
            int n = (lane >= 1 && lane <= R) ? (b - prev + C - 1) / C : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(kFull, n, off);
                if (lane >= off) n += o;
            }
            if (lane <= R) {
                s_m[lane] = b;
                s_tab[lane] = n;
            }
        }
        __syncthreads();
        return;
    }
    for (int r = threadIdx.x; r <= R; r += NT) {
        const int v = ro[r];
        s_m[r] = v < 0 ? 0 : (v > N ? N : v);
    }
    __syncthreads();
    block_scan_inplace<NT, true>(s_m, R + 1, s_tmp);
    for (int r = threadIdx.x; r <= R; r += NT)
        s_tab[r] = (r == 0) ? 0 : (s_m[r] - s_m[r - 1] + C - 1) / C;
    __syncthreads();
    block_scan_inplace<NT, false>(s_tab, R + 1, s_tmp);
}

// Rank of chunk c (c < s_tab[R]): the largest r < R with s_tab[r] <= c.
__device__ __forceinline__ int chunk_rank(const int* s_tab, int R, int c) {
    int lo = 0, hi = R - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_tab[mid] <= c) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__host__ __device__ __forceinline__ int round_up4(int v) { return (v + 3) & ~3; }


// Expert offsets: s_eoff[0..E] = exclusive prefix of totals[0..E-1].
template <int NT>
__device__ void load_expert_offsets(const int32_t* totals, int E, int* s_eoff, int* s_tmp) {
    for (int e = threadIdx.x; e <= E; e += NT) s_eoff[e] = (e == 0) ? 0 : __ldcg(totals + e - 1);
    __syncthreads();
    block_scan_inplace<NT, false>(s_eoff, E + 1, s_tmp);
}

// Outputs that depend only on the expert offsets, spread over the grid (this
// is block b of nb): expert_offsets, masked_m and overflow (block 0), the
// expert base added to rank_expert_offsets, and -1 in row_src past the valid
// rows.  Every thread of the block must call it.
template <int NT>
__device__ void side_outputs(const LayoutArgs& a, const int* s_eoff, int* s_tmp, int b, int nb) {
    const int E = a.E;
    const int NK = a.N * a.K;
    if (b == 0) {
        for (int e = threadIdx.x; e <= E; e += NT) a.expert_offsets[e] = s_eoff[e];
        if (a.cap > 0) {
            int drop = 0;
            for (int e = threadIdx.x; e < E; e += NT) {
                const int tot = s_eoff[e + 1] - s_eoff[e];
                if (a.masked_m) a.masked_m[e] = min(tot, a.cap);
                drop += max(0, tot - a.cap);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) drop += __shfl_xor_sync(kFull, drop, off);
            __syncthreads();
            if ((threadIdx.x & 31) == 0) s_tmp[threadIdx.x >> 5] = drop;
            __syncthreads();
            if (threadIdx.x == 0 && a.overflow) {
                int d = 0;
                for (int w = 0; w < NT / 32; ++w) d += s_tmp[w];
                *a.overflow = d;
            }
            __syncthreads();
        }
    }
    for (int idx = b * NT + threadIdx.x; idx < a.R * E; idx += nb * NT)
        a.rank_expert_offsets[idx] = __ldcg(a.rank_expert_offsets + idx) + s_eoff[idx % E];
    for (int p = s_eoff[E] + b * NT + threadIdx.x; p < NK; p += nb * NT) a.row_src[p] = -1;
}

// Positions of chunk c's picks, in (t, k) order within each expert, starting
// at s_eoff[e] + the chunk's exclusive prefix (row c of ws_hist).  s_w holds
// NT/32 rows of E ints.  Every thread must call it.
template <int NT>
__device__ void scatter_chunk(const LayoutArgs& a, int c, int C, const int* s_m, const int* s_tab,
                              const int* s_eoff, int* s_w) {
    constexpr int kW = NT / 32;
    const int E = a.E, K = a.K;
    const int r = chunk_rank(s_tab, a.R, c);
    const int tok0 = s_m[r] + (c - s_tab[r]) * C;
    const int tok1 = min(tok0 + C, s_m[r + 1]);
    const int i0 = tok0 * K, i1 = tok1 * K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slice = ((i1 - i0 + NT - 1) / NT) * 32;  // items per warp, a multiple of 32
    const int w0 = min(i1, i0 + warp * slice), w1 = min(i1, w0 + slice);
    int* my = s_w + warp * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    // per-warp histograms of the warp's slice
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        int e = (i < w1) ? __ldcg(a.topk_idx + i) : -1;
        if (e < 0 || e >= E) e = -1;
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // warp bases = expert offset + chunk prefix + earlier warps
    const int* pre = a.ws_hist + (size_t)c * E;
    for (int e = threadIdx.x; e < E; e += NT) {
        int run = s_eoff[e] + __ldcg(pre + e);
        for (int w = 0; w < kW; ++w) {
            const int v = s_w[w * E + e];
            s_w[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    // positions in (t, k) order
    const unsigned lt = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        int e = (i < w1) ? __ldcg(a.topk_idx + i) : -1;
        if (e < 0 || e >= E) e = -1;
        const unsigned peers = __match_any_sync(kFull, e);
        int p = -1;
        if (e >= 0) p = my[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
        if (i < w1) {
            a.pos[i] = p;
            if (p >= 0) a.row_src[p] = i / K;
        }
    }
    __syncthreads();
}

}  // namespace lay
}  // namespace ep
