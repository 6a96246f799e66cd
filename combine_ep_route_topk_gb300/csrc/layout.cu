// Dispatch layout for sm_103a: "Anatomy of a High-Performance EP Kernel",
// "High throughput: ask first, then send" and "Dispatch" -- before any row
// moves, every (rank, expert) count and every row position is known, and each
// expert's rows form one dense block of an expert-major buffer.
//
// A stable counting sort of the N*K picks by expert id, in three kernels:
//   1. hist    one block per chunk of C tokens (chunks never straddle a rank)
//              builds the chunk's expert histogram in shared memory with
//              warp-aggregated increments (__match_any_sync leaders).
//   2. scan    E/32 blocks; each scans 32 expert columns of the chunk
//              histograms down the chunks (32 row groups per column), leaving
//              per-chunk exclusive prefixes, expert totals, per-(rank, expert)
//              counts and each rank's offset within an expert segment.
//   3. scatter one block per chunk again: expert offsets = exclusive scan of
//              the totals; the chunk's picks get positions in (t, k) order via
//              per-warp bases and __match_any_sync ranks, so the result never
//              depends on atomic ordering.
// Everything stays on the device (no host read of a count), so the masked
// decode path can be captured in a CUDA graph.
#include <climits>

#include "ep_kernels.cuh"

namespace ep {

int layout_chunk_tokens(int N) {
    int C = (N + 255) / 256;  // about 256 chunks at most, each a multiple of 32 tokens
    C = ((C + 31) / 32) * 32;
    return C < 32 ? 32 : C;
}

int layout_chunk_slots(int N, int R) {
    const int C = layout_chunk_tokens(N);
    return (N + C - 1) / C + R;
}

size_t layout_workspace_bytes(int N, int E, int /*K*/, int R) {
    const size_t slots = (size_t)layout_chunk_slots(N, R);
    const size_t b = (slots * (size_t)E + (size_t)E) * sizeof(int32_t);
    return ((b + 255) / 256) * 256;
}

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kNT = 256;  // threads of the hist / scatter blocks
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

__device__ __forceinline__ int round_up4(int v) { return (v + 3) & ~3; }

// ---- 1. chunk histograms --------------------------------------------------
__global__ void __launch_bounds__(kNT) layout_hist_kernel(LayoutArgs a, int C) {
    extern __shared__ int smem[];
    int* s_m = smem;
    int* s_tab = s_m + round_up4(a.R + 1);
    int* s_tmp = s_tab + round_up4(a.R + 1);
    int* s_hist = s_tmp + 32;
    build_chunk_table<kNT>(a.rank_offsets, a.R, a.N, C, s_m, s_tab, s_tmp);
    const int c = blockIdx.x;
    if (c >= s_tab[a.R]) return;
    for (int e = threadIdx.x; e < a.E; e += kNT) s_hist[e] = 0;
    __syncthreads();
    const int r = chunk_rank(s_tab, a.R, c);
    const int tok0 = s_m[r] + (c - s_tab[r]) * C;
    const int tok1 = min(tok0 + C, s_m[r + 1]);
    const int i0 = tok0 * a.K, i1 = tok1 * a.K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int base = i0 + warp * 32; base < i1; base += kNT) {
        const int i = base + lane;
        int e = (i < i1) ? __ldg(a.topk_idx + i) : -1;
        if (e < 0 || e >= a.E) e = -1;
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0 && lane == __ffs(peers) - 1) atomicAdd(&s_hist[e], __popc(peers));
    }
    __syncthreads();
    int* row = a.ws_hist + (size_t)c * a.E;
    for (int e = threadIdx.x; e < a.E; e += kNT) row[e] = s_hist[e];
}

// ---- 2. column scans --------------------------------------------------------
__global__ void __launch_bounds__(1024) layout_scan_kernel(LayoutArgs a, int C) {
    extern __shared__ int smem[];
    int* s_m = smem;
    int* s_tab = s_m + round_up4(a.R + 1);
    int* s_tmp = s_tab + round_up4(a.R + 1);
    int* s_part = s_tmp + 32;    // [32 groups][32 columns]
    int* s_total = s_part + 1024;  // [32 columns]
    build_chunk_table<1024>(a.rank_offsets, a.R, a.N, C, s_m, s_tab, s_tmp);
    const int S = s_tab[a.R];
    const int col = threadIdx.x & 31, g = threadIdx.x >> 5;
    const int e = blockIdx.x * 32 + col;
    const bool live = e < a.E;
    const int rpg = (S + 31) / 32;
    const int r0 = min(S, g * rpg), r1 = min(S, r0 + rpg);
    int* hist = a.ws_hist;
    int sum = 0;
    if (live)
        for (int c = r0; c < r1; ++c) sum += hist[(size_t)c * a.E + e];
    s_part[g * 32 + col] = sum;
    __syncthreads();
    int run = 0, total = 0;
    for (int gg = 0; gg < 32; ++gg) {
        const int v = s_part[gg * 32 + col];
        if (gg < g) run += v;
        total += v;
    }
    if (live)
        for (int c = r0; c < r1; ++c) {
            const size_t at = (size_t)c * a.E + e;
            const int v = hist[at];
            hist[at] = run;
            run += v;
        }
    if (g == 0) {
        s_total[col] = total;
        if (live) a.ws_totals[e] = total;
    }
    __syncthreads();
    // per-(rank, expert) counts and the rank's start within the expert segment
    // (without the expert's own offset, which the scatter kernel adds)
    for (int idx = threadIdx.x; idx < a.R * 32; idx += 1024) {
        const int r = idx >> 5, cc = idx & 31;
        const int ee = blockIdx.x * 32 + cc;
        if (ee >= a.E) continue;
        const int lo = s_tab[r], hi = s_tab[r + 1];
        const int pre_lo = (lo < S) ? hist[(size_t)lo * a.E + ee] : s_total[cc];
        const int pre_hi = (hi < S) ? hist[(size_t)hi * a.E + ee] : s_total[cc];
        a.counts[(size_t)r * a.E + ee] = pre_hi - pre_lo;
        a.rank_expert_offsets[(size_t)r * a.E + ee] = pre_lo;
    }
}

// ---- 3. stable scatter of positions ----------------------------------------
__global__ void __launch_bounds__(kNT) layout_scatter_kernel(LayoutArgs a, int C) {
    extern __shared__ int smem[];
    int* s_m = smem;
    int* s_tab = s_m + round_up4(a.R + 1);
    int* s_tmp = s_tab + round_up4(a.R + 1);
    int* s_eoff = s_tmp + 32;               // [E+1]
    int* s_w = s_eoff + round_up4(a.E + 1);  // [warps][E]
    build_chunk_table<kNT>(a.rank_offsets, a.R, a.N, C, s_m, s_tab, s_tmp);
    const int E = a.E, K = a.K;
    for (int e = threadIdx.x; e <= E; e += kNT) s_eoff[e] = (e == 0) ? 0 : a.ws_totals[e - 1];
    __syncthreads();
    block_scan_inplace<kNT, false>(s_eoff, E + 1, s_tmp);  // s_eoff[e] = exclusive prefix

    // side outputs, spread over all blocks
    const int b = blockIdx.x, nb = gridDim.x;
    const int NK = a.N * K;
    if (b == 0) {
        for (int e = threadIdx.x; e <= E; e += kNT) a.expert_offsets[e] = s_eoff[e];
        if (a.cap > 0) {
            int drop = 0;
            for (int e = threadIdx.x; e < E; e += kNT) {
                const int tot = s_eoff[e + 1] - s_eoff[e];
                if (a.masked_m) a.masked_m[e] = min(tot, a.cap);
                drop += max(0, tot - a.cap);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) drop += __shfl_xor_sync(kFull, drop, off);
            if ((threadIdx.x & 31) == 0) s_tmp[threadIdx.x >> 5] = drop;
            __syncthreads();
            if (threadIdx.x == 0 && a.overflow) {
                int d = 0;
                for (int w = 0; w < kWarps; ++w) d += s_tmp[w];
                *a.overflow = d;
            }
        }
    }
    for (int idx = b * kNT + threadIdx.x; idx < a.R * E; idx += nb * kNT)
        a.rank_expert_offsets[idx] += s_eoff[idx % E];
    for (int p = s_eoff[E] + b * kNT + threadIdx.x; p < NK; p += nb * kNT) a.row_src[p] = -1;

    const int c = blockIdx.x;
    if (c >= s_tab[a.R]) return;
    const int r = chunk_rank(s_tab, a.R, c);
    const int tok0 = s_m[r] + (c - s_tab[r]) * C;
    const int tok1 = min(tok0 + C, s_m[r + 1]);
    const int i0 = tok0 * K, i1 = tok1 * K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slice = ((i1 - i0 + kNT - 1) / kNT) * 32;  // items per warp, a multiple of 32
    const int w0 = min(i1, i0 + warp * slice), w1 = min(i1, w0 + slice);
    int* my = s_w + warp * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
    // phase 1: per-warp histograms of the warp's slice
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        int e = (i < w1) ? __ldg(a.topk_idx + i) : -1;
        if (e < 0 || e >= E) e = -1;
        const unsigned peers = __match_any_sync(kFull, e);
        if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // phase 2: warp bases = expert offset + chunk prefix + earlier warps
    const int* pre = a.ws_hist + (size_t)c * E;
    for (int e = threadIdx.x; e < E; e += kNT) {
        int run = s_eoff[e] + pre[e];
        for (int w = 0; w < kWarps; ++w) {
            const int v = s_w[w * E + e];
            s_w[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    // phase 3: positions in (t, k) order
    const unsigned lt = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        int e = (i < w1) ? __ldg(a.topk_idx + i) : -1;
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
}

}  // namespace

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t s) {
    const int C = layout_chunk_tokens(a.N);
    const int slots = layout_chunk_slots(a.N, a.R);
    const int tab = 2 * ((a.R + 1 + 3) & ~3) + 32;
    const size_t sh_hist = (size_t)(tab + a.E) * sizeof(int);
    const size_t sh_scan = (size_t)(tab + 1024 + 32) * sizeof(int);
    const size_t sh_scat = (size_t)(tab + ((a.E + 1 + 3) & ~3) + kWarps * a.E) * sizeof(int);
    layout_hist_kernel<<<slots, kNT, sh_hist, s>>>(a, C);
    layout_scan_kernel<<<(a.E + 31) / 32, 1024, sh_scan, s>>>(a, C);
    layout_scatter_kernel<<<slots, kNT, sh_scat, s>>>(a, C);
    note_launch(3);
    return cudaGetLastError();
}

}  // namespace ep
