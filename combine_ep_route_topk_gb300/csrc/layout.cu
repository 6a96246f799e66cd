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
// decode path can be captured in a CUDA graph.  Problems of at most 16384
// picks take the one-launch, one-block-per-expert variant in layout_small.cu;
// layout_cluster.cu holds a one-cluster variant for the same sizes, used when
// the first is switched off.
#include "layout_common.cuh"

namespace ep {

int layout_chunk_tokens(int N) {
    int C = (N + 255) / 256;  // about 256 chunks at most, each a multiple of 8 tokens
    C = ((C + 7) / 8) * 8;
    return C < 8 ? 8 : C;
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

using namespace lay;

// ---- 1. chunk histograms --------------------------------------------------
__global__ void __launch_bounds__(kNT) layout_hist_kernel(LayoutArgs a, int C) {
    pdl_prologue();
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
    pdl_prologue();
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
    pdl_prologue();
    extern __shared__ int smem[];
    int* s_m = smem;
    int* s_tab = s_m + round_up4(a.R + 1);
    int* s_tmp = s_tab + round_up4(a.R + 1);
    int* s_eoff = s_tmp + 32;               // [E+1]
    int* s_w = s_eoff + round_up4(a.E + 1);  // [warps][E]
    build_chunk_table<kNT>(a.rank_offsets, a.R, a.N, C, s_m, s_tab, s_tmp);
    load_expert_offsets<kNT>(a.ws_totals, a.E, s_eoff, s_tmp);
    side_outputs<kNT>(a, s_eoff, s_tmp, blockIdx.x, gridDim.x);
    if ((int)blockIdx.x >= s_tab[a.R]) return;
    scatter_chunk<kNT>(a, blockIdx.x, C, s_m, s_tab, s_eoff, s_w);
}

}  // namespace

cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t s) {
    if (layout_small_fits(a.N, a.E, a.K, a.R)) {  // layout_small.cu
        note_launch(1);
        return launch_layout_small(a, s);
    }
    if (layout_cluster_fits(a.N, a.E, a.K, a.R)) {  // layout_cluster.cu
        note_launch(1);
        return launch_layout_cluster(a, s);
    }
    const int C = layout_chunk_tokens(a.N);
    const int slots = layout_chunk_slots(a.N, a.R);
    const int tab = 2 * ((a.R + 1 + 3) & ~3) + 32;
    const size_t sh_hist = (size_t)(tab + a.E) * sizeof(int);
    const size_t sh_scan = (size_t)(tab + 1024 + 32) * sizeof(int);
    const size_t sh_scat = (size_t)(tab + ((a.E + 1 + 3) & ~3) + kWarps * a.E) * sizeof(int);
    cudaError_t err = launch(layout_hist_kernel, dim3(slots), dim3(kNT), sh_hist, s, a, C);
    if (err == cudaSuccess)
        err = launch(layout_scan_kernel, dim3((a.E + 31) / 32), dim3(1024), sh_scan, s, a, C);
    if (err == cudaSuccess)
        err = launch(layout_scatter_kernel, dim3(slots), dim3(kNT), sh_scat, s, a, C);
    note_launch(3);
    return err;
}

}  // namespace ep
