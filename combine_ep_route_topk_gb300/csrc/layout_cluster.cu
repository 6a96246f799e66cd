// Dispatch layout of a small problem in one launch: "Anatomy of a High-
// Performance EP Kernel", "High throughput: ask first, then send" and
// "Dispatch" (the counts and every row position, before any row moves).
//
// The same stable counting sort as the three layout kernels, run by one
// thread-block cluster of kCS CTAs with one full cluster barrier.  Chunks of
// C tokens (never straddling a rank) are owned Q per CTA, at most about one
// per warp:
//   1. each warp builds its chunk's expert histogram in shared memory (one
//      warp per chunk row, so no atomics) and keeps the chunk's expert ids in
//      registers when they fit;
//   2. each CTA turns its rows into local exclusive column prefixes and its
//      column totals, then pushes through distributed shared memory
//      (a) its column totals to every CTA and (b) the local prefix row at
//      every rank boundary it owns to the CTA that writes that rank's counts;
//   3. a full cluster barrier.  (An earlier, split one -- arrival at kernel
//      entry, wait just before the first push -- makes sure that no push
//      reaches a CTA that has not started.)  Every later read is local;
//   4. each CTA derives the base of its rows (the totals of earlier CTAs),
//      the expert totals and offsets, writes the counts and rank offsets of
//      its ranks (r = j mod kCS) and gives its chunks' picks their positions
//      in (t, k) order.
// No CTA touches another's shared memory after the barrier, so each may leave
// when done.  Every thread of every CTA reaches both barriers, whatever the
// sizes (no return before them).
#include <cooperative_groups.h>

#include <cstdlib>

#include "layout_common.cuh"

namespace ep {
namespace {

namespace cg = cooperative_groups;
using namespace lay;

constexpr int kCS = 8;         // CTAs of the cluster (portable cluster size)
constexpr int kCT = 512;       // threads of a CTA
constexpr int kCW = kCT / 32;  // warps of a CTA
#ifndef EP_LAYOUT_CLUSTER_U
#define EP_LAYOUT_CLUSTER_U 4
#endif
#ifndef EP_LAYOUT_CLUSTER_MAX_PICKS
#define EP_LAYOUT_CLUSTER_MAX_PICKS (1 << 14)
#endif
constexpr int kU = EP_LAYOUT_CLUSTER_U;  // 32-pick passes whose loads are issued together
constexpr size_t kMaxSmem = 160 * 1024;
// Larger problems take the three kernels: measured on GB300 (E = 256, K = 8,
// 8 ranks), the cluster takes 13.0 / 15.0 / 21.2 us at 8192 / 16384 / 32768
// picks against 15.1 / 17.1 / 18.0 us; at 64 ranks and 32768 picks, 31.4
// against 20.1 us.
constexpr long long kMaxPicks = EP_LAYOUT_CLUSTER_MAX_PICKS;
constexpr int kMaxRanks = 64;

struct ClusterPlan {
    int C;        // tokens per chunk
    int Q;        // chunk rows per CTA
    int RS;       // rank slots per CTA: ranks r = j, j + kCS, ...
    size_t smem;  // dynamic shared memory per CTA, bytes
};

// Chunks: at most kCS*kCW (one per warp) when the ranks leave room, at least
// 8 tokens each.
ClusterPlan cluster_plan(int N, int E, int R) {
    const int room = kCS * kCW - R;
    const int parts = room >= 32 ? room : kCS * kCW;
    int C = (N + parts - 1) / parts;
    C = ((C + 7) / 8) * 8;
    if (C < 8) C = 8;
    const int slots = (N + C - 1) / C + R;
    const int Q = (slots + kCS - 1) / kCS;
    const int RS = (R + kCS - 1) / kCS;
    const size_t ints = 2 * (size_t)round_up4(R + 1) + 32 + (size_t)round_up4(E + 1) +
                        2 * (size_t)round_up4(E) + (size_t)kCS * E + (size_t)Q * E +
                        2 * (size_t)RS * E;
    return {C, Q, RS, ints * sizeof(int)};
}

// Picks [i0, i1) of chunk c (c < s_tab[R]).
__device__ __forceinline__ void chunk_picks(const int* s_m, const int* s_tab, int R, int C, int K,
                                            int c, int& i0, int& i1) {
    const int r = chunk_rank(s_tab, R, c);
    const int tok0 = s_m[r] + (c - s_tab[r]) * C;
    const int tok1 = min(tok0 + C, s_m[r + 1]);
    i0 = tok0 * K;
    i1 = tok1 * K;
}

// Expert ids of kU consecutive 32-pick passes from `base` (-1: none).
__device__ __forceinline__ void load_passes(const LayoutArgs& a, int base, int i1, int lane,
                                            int (&ev)[kU]) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int i = base + u * 32 + lane;
        int e = (i < i1) ? __ldg(a.topk_idx + i) : -1;
        ev[u] = (e < 0 || e >= a.E) ? -1 : e;
    }
}

__device__ __forceinline__ void hist_passes(int* row, const int (&ev)[kU], int lane) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const unsigned peers = __match_any_sync(kFull, ev[u]);
        if (ev[u] >= 0 && lane == __ffs(peers) - 1) row[ev[u]] += __popc(peers);
        __syncwarp();
    }
}

// Positions of kU passes from `base`; `run` holds each expert's next row.
__device__ __forceinline__ void scatter_passes(const LayoutArgs& a, int* run, const int (&ev)[kU],
                                               int base, int i1, int lane) {
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        const int e = ev[u];
        const int i = base + u * 32 + lane;
        const unsigned peers = __match_any_sync(kFull, e);
        int p = -1;
        if (e >= 0) p = run[e] + __popc(peers & lt);
        __syncwarp();
        if (e >= 0 && lane == __ffs(peers) - 1) run[e] += __popc(peers);
        __syncwarp();
        if (i < i1) {
            a.pos[i] = p;
            if (p >= 0) a.row_src[p] = i / a.K;
        }
    }
}

__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kCT)
    layout_cluster_kernel(LayoutArgs a, int C, int Q, int RS) {
    // Announce this CTA to the cluster at once (no memory ordering needed):
    // the matching wait below, before the first store into another CTA's
    // shared memory, guarantees that every CTA of the cluster is running.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
    pdl_prologue();
    cg::cluster_group cl = cg::this_cluster();
    const int j = (int)cl.block_rank();
    const int R = a.R, E = a.E, K = a.K;
    extern __shared__ int smem[];
    int* s_m = smem;
    int* s_tab = s_m + round_up4(R + 1);
    int* s_tmp = s_tab + round_up4(R + 1);
    int* s_eoff = s_tmp + 32;                 // [E+1] expert offsets
    int* s_tot = s_eoff + round_up4(E + 1);   // [E] expert totals
    int* s_base = s_tot + round_up4(E);       // [E] rows of earlier CTAs, per expert
    int* s_ct = s_base + round_up4(E);        // [kCS][E] column totals of every CTA
    int* s_hist = s_ct + (size_t)kCS * E;     // [Q][E] chunk rows: histograms, then prefixes
    int* s_lo = s_hist + (size_t)Q * E;       // [RS][E] local prefix at rank r's first chunk
    int* s_hi = s_lo + (size_t)RS * E;        // [RS][E] ... at the chunk after rank r
    for (int i = threadIdx.x; i < Q * E; i += kCT) s_hist[i] = 0;
    build_chunk_table<kCT>(a.rank_offsets, R, a.N, C, s_m, s_tab, s_tmp);  // syncs
    const int S = s_tab[R];  // chunks of the problem
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // 1. histograms of this CTA's chunks j*Q + q, one warp per chunk row; the
    //    first chunk of each warp keeps its ids when they fit in kU passes
    int keep[kU];
    bool kept = false;
    for (int q = warp; q < Q && j * Q + q < S; q += kCW) {
        int i0, i1;
        chunk_picks(s_m, s_tab, R, C, K, j * Q + q, i0, i1);
        int* row = s_hist + (size_t)q * E;
        for (int base = i0; base < i1; base += 32 * kU) {
            int ev[kU];
            load_passes(a, base, i1, lane, ev);
            hist_passes(row, ev, lane);
            if (q == warp && i1 - i0 <= 32 * kU) {
#pragma unroll
                for (int u = 0; u < kU; ++u) keep[u] = ev[u];
                kept = true;
            }
        }
    }
    __syncthreads();

    // 2. local exclusive prefixes down this CTA's rows, column totals to
    //    every CTA, and the prefix rows at the rank boundaries this CTA owns
    //    to the CTAs that write those ranks.  First wait until every CTA of
    //    the cluster has arrived at the entry barrier, i.e. is running and
    //    owns its shared memory (the pushed arrays are not touched locally
    //    before the cluster barrier below, so a running target is enough).
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    for (int e = threadIdx.x; e < E; e += kCT) {
        int run = 0;
        for (int q = 0; q < Q; ++q) {
            const int v = s_hist[(size_t)q * E + e];
            s_hist[(size_t)q * E + e] = run;
            run += v;
        }
        for (int d = 0; d < kCS; ++d) cl.map_shared_rank(s_ct, (unsigned)d)[(size_t)j * E + e] = run;
    }
    __syncthreads();
    const int cq0 = j * Q, cq1 = min(S, cq0 + Q);  // this CTA's chunks
    for (int r = warp; r < R; r += kCW) {  // a warp per rank, lanes over experts
        const int lo = s_tab[r], hi = s_tab[r + 1];
        const unsigned h = (unsigned)(r % kCS);
        const size_t slot = (size_t)(r / kCS) * E;
        if (lo >= cq0 && lo < cq1) {
            int* dst = cl.map_shared_rank(s_lo, h) + slot;
            for (int e = lane; e < E; e += 32) dst[e] = s_hist[(size_t)(lo - cq0) * E + e];
        }
        if (hi >= cq0 && hi < cq1) {
            int* dst = cl.map_shared_rank(s_hi, h) + slot;
            for (int e = lane; e < E; e += 32) dst[e] = s_hist[(size_t)(hi - cq0) * E + e];
        }
    }
    cl.sync();  // the one full cluster barrier: every later access is local

    // 3. bases, totals and expert offsets
    for (int e = threadIdx.x; e < E; e += kCT) {
        int b = 0, t = 0;
        for (int d = 0; d < kCS; ++d) {
            const int v = s_ct[(size_t)d * E + e];
            if (d < j) b += v;
            t += v;
        }
        s_base[e] = b;
        s_tot[e] = t;
    }
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += kCT) s_eoff[e] = (e == 0) ? 0 : s_tot[e - 1];
    __syncthreads();
    block_scan_inplace<kCT, false>(s_eoff, E + 1, s_tmp);

    // 4a. counts and rank offsets of ranks r = j, j + kCS, ...: the prefix
    //     of chunk c is the base of its CTA plus its local prefix (the total
    //     past the last chunk)
    for (int r = j, rs = 0; r < R; r += kCS, ++rs) {
        const int lo = s_tab[r], hi = s_tab[r + 1];
        const int olo = lo / Q, ohi = hi / Q;
        for (int e = threadIdx.x; e < E; e += kCT) {
            int blo = 0, bhi = 0;
            for (int d = 0; d < kCS; ++d) {
                const int v = s_ct[(size_t)d * E + e];
                if (d < olo) blo += v;
                if (d < ohi) bhi += v;
            }
            const int plo = (lo < S) ? blo + s_lo[(size_t)rs * E + e] : s_tot[e];
            const int phi = (hi < S) ? bhi + s_hi[(size_t)rs * E + e] : s_tot[e];
            a.counts[(size_t)r * E + e] = phi - plo;
            a.rank_expert_offsets[(size_t)r * E + e] = s_eoff[e] + plo;
        }
    }
    // 4b. outputs that depend only on the expert offsets
    const int NK = a.N * K;
    if (j == 0) {
        for (int e = threadIdx.x; e <= E; e += kCT) a.expert_offsets[e] = s_eoff[e];
        if (a.cap > 0) {
            int drop = 0;
            for (int e = threadIdx.x; e < E; e += kCT) {
                const int tot = s_eoff[e + 1] - s_eoff[e];
                if (a.masked_m) a.masked_m[e] = min(tot, a.cap);
                drop += max(0, tot - a.cap);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) drop += __shfl_xor_sync(kFull, drop, off);
            if (lane == 0) s_tmp[warp] = drop;
            __syncthreads();
            if (threadIdx.x == 0 && a.overflow) {
                int d = 0;
                for (int w = 0; w < kCW; ++w) d += s_tmp[w];
                *a.overflow = d;
            }
        }
    }
    for (int p = s_eoff[E] + j * kCT + threadIdx.x; p < NK; p += kCS * kCT) a.row_src[p] = -1;

    // 4c. positions of this CTA's picks, one warp per chunk, in (t, k) order;
    //     the chunk's row becomes its running next-row counter
    for (int q = warp; q < Q && j * Q + q < S; q += kCW) {
        int i0, i1;
        chunk_picks(s_m, s_tab, R, C, K, j * Q + q, i0, i1);
        int* run = s_hist + (size_t)q * E;
        for (int e = lane; e < E; e += 32) run[e] += s_eoff[e] + s_base[e];
        __syncwarp();
        if (q == warp && kept) {
            scatter_passes(a, run, keep, i0, i1, lane);
        } else {
            for (int base = i0; base < i1; base += 32 * kU) {
                int ev[kU];
                load_passes(a, base, i1, lane, ev);
                scatter_passes(a, run, ev, base, i1, lane);
            }
        }
    }
}

}  // namespace

// The one-cluster path serves problems of at most kMaxPicks picks and
// kMaxRanks ranks whose chunk rows fit in shared memory.  EP_LAYOUT_CLUSTER=0 in the environment
// (read at every call) selects the three-kernel path for every size.
bool layout_kernels_forced() {
    const char* v = std::getenv("EP_LAYOUT_CLUSTER");
    return v && v[0] == '0';
}

bool layout_cluster_fits(int N, int E, int K, int R) {
    if (layout_kernels_forced()) return false;
    if ((long long)N * K > kMaxPicks || R > kMaxRanks) return false;
    return cluster_plan(N, E, R).smem <= kMaxSmem;
}

cudaError_t launch_layout_cluster(const LayoutArgs& a, cudaStream_t s) {
    const ClusterPlan p = cluster_plan(a.N, a.E, a.R);
    if (p.smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(
            layout_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        if (e != cudaSuccess) return e;
    }
    return launch(layout_cluster_kernel, dim3(kCS), dim3(kCT), p.smem, s, a, p.C, p.Q, p.RS);
}

}  // namespace ep
