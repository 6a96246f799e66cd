// Fused route + layout for sm_103a: one cooperative, persistent kernel that
// computes exactly what ep_route_topk followed by ep_dispatch_layout compute
// ("Anatomy of a High-Performance EP Kernel": route locally, then "ask first,
// then send"), without the launches and ramp-ups in between.
//
//   phase 1  tokens go round-robin to every warp of the grid (balanced to
//            one token per warp); each warp routes its tokens
//            (route::route_token) and adds each pick to its chunk's
//            histogram row with an L2 atomic (chunks of C tokens never
//            straddle a rank; the rows are zeroed before the launch).
//   barrier
//   phase 2  blocks take tiles of 32 expert columns; each warp scans a group
//            of chunk rows (coalesced 128-byte reads) and the block combines
//            the groups: exclusive prefixes, expert totals, per-rank counts
//            and offsets.
//   barrier
//   phase 3  expert offsets from the totals, side outputs, and the stable
//            per-chunk scatter of positions (lay::scatter_chunk).
//
// The grid never exceeds the blocks that can be resident at once (the launch
// is cooperative), so every block reaches each barrier.  A barrier is a
// counter in the workspace, zeroed (with the chunk histograms) by one memset
// before the launch; each wait is bounded (kSpinLimit polls with a back-off)
// and, if it ever ran out, the block would record 1 in `status` and return
// instead of waiting on.  Block 0 stores 0 in `status` before it arrives at
// the first barrier, so a 1 recorded by any timeout is never overwritten.
#include <algorithm>

#include "ep.h"
#include "ep_kernels.cuh"
#include "layout_common.cuh"
#include "route_common.cuh"

namespace ep {

int route_layout_chunk_tokens(int N) {
    // About 256 chunks, as in the layout kernels: routing goes round-robin over
    // all warps whatever the chunk size, and fewer chunk rows keep the column
    // scans short.
    int C = (N + 255) / 256;
    C = ((C + 7) / 8) * 8;
    return C < 8 ? 8 : C;
}

int route_layout_chunk_slots(int N, int R) {
    const int C = route_layout_chunk_tokens(N);
    return (N + C - 1) / C + R;
}

size_t route_layout_workspace_bytes(int N, int E, int K, int R) {
    const size_t slots = (size_t)route_layout_chunk_slots(N, R);
    size_t b = (slots * (size_t)E + (size_t)E + 64) * sizeof(int32_t);
    b = ((b + 255) / 256) * 256;
    const size_t sep = layout_workspace_bytes(N, E, K, R);  // fallback path
    return b > sep ? b : sep;
}

namespace {

using namespace lay;

constexpr unsigned kSpinLimit = 1u << 22;

struct FusedArgs {
    LayoutArgs a;            // a.topk_idx aliases topk_idx below
    const float* logits;
    const int32_t* emap;
    int32_t* topk_idx;
    float* topk_w;
    unsigned* bar;           // two barrier counters, zero at launch
    int32_t* status;         // may be null
};

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Grid-wide barrier over a co-resident grid: every block adds one to *ctr,
// then waits until it reaches `target` (the grid size).  The wait is bounded
// by `limit` polls; if it runs out the block records 1 in *status and the
// barrier returns false, which a cooperative launch rules out.
__device__ bool grid_barrier(unsigned* ctr, unsigned target, unsigned limit, int32_t* status) {
    __syncthreads();
    int ok = 1;
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(ctr, 1u);
        unsigned polls = 0;
        while (ld_acquire_gpu(ctr) < target) {
            if (++polls > limit) {
                ok = 0;
                if (status) atomicExch(status, 1);
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
    }
    return __syncthreads_and(ok) != 0;
}

// Self-test of the bounded wait: a barrier that waits for one block more
// than the grid has, so the wait runs out after `limit` polls, records 1 in
// *status, and every block returns.
__global__ void __launch_bounds__(32) barrier_timeout_kernel(unsigned* ctr, unsigned limit,
                                                             int32_t* status) {
    pdl_prologue();
    grid_barrier(ctr, gridDim.x + 1, limit, status);
}

// Rank of token t, s_m[0] <= t < s_m[R]: the r with s_m[r] <= t < s_m[r+1]
// (s_m non-decreasing; empty ranks never match).
__device__ __forceinline__ int token_rank(const int* s_m, int R, int t) {
    int lo = 0, hi = R - 1;
    while (lo < hi) {  // largest r < R with s_m[r] <= t
        const int mid = (lo + hi + 1) >> 1;
        if (s_m[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int VPL, bool VEC, int KT>
__global__ void __launch_bounds__(kNT) route_layout_kernel(FusedArgs f, int C) {
    extern __shared__ int smem[];
    const LayoutArgs& a = f.a;
    int* s_m = smem;
    int* s_tab = s_m + round_up4(a.R + 1);
    int* s_tmp = s_tab + round_up4(a.R + 1);
    int* s_eoff = s_tmp + 32;                // [E+1]
    int* s_w = s_eoff + round_up4(a.E + 1);   // [warps][E]; phase 1: one histogram
    build_chunk_table<kNT>(a.rank_offsets, a.R, a.N, C, s_m, s_tab, s_tmp);
    const int S = s_tab[a.R];
    const int E = a.E;
    const int K = KT > 0 ? KT : a.K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

    // ---- phase 1: tokens round-robin over every warp of the grid (balanced
    // to one token); each pick counts into its chunk's histogram row, zeroed
    // before the launch, with an L2 atomic
    const int gw = blockIdx.x * kWarps + warp, nw = gridDim.x * kWarps;
    const int t_lo = s_m[0], t_hi = s_m[a.R];  // tokens that belong to a rank
    for (int t = gw; t < a.N; t += nw) {
        int id;
        float w;
        route::route_token<VPL, VEC, KT>(f.logits + (size_t)t * E, E, a.K, f.emap, lane, id, w);
        if (lane < K) {
            f.topk_idx[(size_t)t * K + lane] = id;
            f.topk_w[(size_t)t * K + lane] = w;
            if (id >= 0 && t >= t_lo && t < t_hi) {
                const int r = token_rank(s_m, a.R, t);
                const int c = s_tab[r] + (t - s_m[r]) / C;
                atomicAdd(a.ws_hist + (size_t)c * E + id, 1);
            }
        }
    }
    // Block 0 clears the status word before it arrives at the first barrier.
    // Any timeout is recorded after this store: one at the second barrier
    // comes from a block that passed the first, hence after block 0 arrived
    // (the barrier's fence and acquire order the two); one at the first
    // barrier keeps its block from ever arriving at the second, so block 0's
    // own wait there runs out and records 1 after its 0.
    if (blockIdx.x == 0 && threadIdx.x == 0 && f.status) *f.status = 0;
    if (!grid_barrier(f.bar + 0, gridDim.x, kSpinLimit, f.status)) return;

    // ---- phase 2: tiles of 32 expert columns; warp w scans row group w, so
    // every row read is one coalesced 128-byte line per warp
    for (int tile = blockIdx.x; tile * 32 < E; tile += gridDim.x) {
        int* hist = a.ws_hist;
        const int e = tile * 32 + lane;
        const bool live = e < E;
        const int rpg = (S + kWarps - 1) / kWarps;
        const int r0 = min(S, warp * rpg), r1 = min(S, r0 + rpg);
        constexpr int kB = 8;  // rows whose loads are in flight together
        int sum = 0;
        if (live)
            for (int c0 = r0; c0 < r1; c0 += kB) {
                int v[kB];
#pragma unroll
                for (int b = 0; b < kB; ++b)
                    v[b] = (c0 + b < r1) ? __ldcg(hist + (size_t)(c0 + b) * E + e) : 0;
#pragma unroll
                for (int b = 0; b < kB; ++b) sum += v[b];
            }
        s_w[warp * 32 + lane] = sum;
        __syncthreads();
        int run = 0, total = 0;
        for (int w = 0; w < kWarps; ++w) {
            const int v = s_w[w * 32 + lane];
            if (w < warp) run += v;
            total += v;
        }
        if (live)
            for (int c0 = r0; c0 < r1; c0 += kB) {
                int v[kB];
#pragma unroll
                for (int b = 0; b < kB; ++b)
                    v[b] = (c0 + b < r1) ? __ldcg(hist + (size_t)(c0 + b) * E + e) : 0;
#pragma unroll
                for (int b = 0; b < kB; ++b)
                    if (c0 + b < r1) {
                        hist[(size_t)(c0 + b) * E + e] = run;
                        run += v[b];
                    }
            }
        if (warp == 0) {
            s_w[kWarps * 32 + lane] = total;
            if (live) a.ws_totals[e] = total;
        }
        __syncthreads();
        for (int idx = threadIdx.x; idx < a.R * 32; idx += kNT) {
            const int r = idx >> 5, cc = idx & 31;
            const int ee = tile * 32 + cc;
            if (ee >= E) continue;
            const int tot = s_w[kWarps * 32 + cc];
            const int lo = s_tab[r], hi = s_tab[r + 1];
            const int pre_lo = (lo < S) ? __ldcg(hist + (size_t)lo * E + ee) : tot;
            const int pre_hi = (hi < S) ? __ldcg(hist + (size_t)hi * E + ee) : tot;
            a.counts[(size_t)r * E + ee] = pre_hi - pre_lo;
            a.rank_expert_offsets[(size_t)r * E + ee] = pre_lo;
        }
        __syncthreads();
    }
    if (!grid_barrier(f.bar + 1, gridDim.x, kSpinLimit, f.status)) return;

    // ---- phase 3: offsets, side outputs, stable positions
    load_expert_offsets<kNT>(a.ws_totals, E, s_eoff, s_tmp);
    side_outputs<kNT>(a, s_eoff, s_tmp, blockIdx.x, gridDim.x);
    for (int c = blockIdx.x; c < S; c += gridDim.x)
        scatter_chunk<kNT>(a, c, C, s_m, s_tab, s_eoff, s_w);
}

template <int VPL, bool VEC, int KT>
cudaError_t launch_fused_t(FusedArgs& f, int C, int slots, size_t smem, cudaStream_t s,
                           bool* launched) {
    const int N = f.a.N;
    auto* fn = route_layout_kernel<VPL, VEC, KT>;
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kNT, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaSuccess;  // not launched: caller falls back
    // Enough blocks for about 4 tokens per warp in phase 1 and one block per
    // chunk in phase 3, but no more (a larger grid only slows the barriers
    // and repeats the per-block offset work), and never more than can be
    // resident at once.
    const int want = std::max(slots, (N + kWarps * 4 - 1) / (kWarps * 4));
    int grid = std::min(per_sm * sm_count(), want);
    if (grid < 1) grid = 1;
    void* args[] = {&f, &C};
    err = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fn), dim3(grid), dim3(kNT),
                                      args, smem, s);
    if (err == cudaSuccess) {
        *launched = true;
        note_launch();
    }
    return err;
}

}  // namespace

cudaError_t launch_barrier_selftest(unsigned* ctr, int32_t* status, cudaStream_t s) {
    cudaError_t err = cudaMemsetAsync(ctr, 0, sizeof(unsigned), s);
    if (err == cudaSuccess) err = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
    if (err == cudaSuccess)
        err = launch(barrier_timeout_kernel, dim3(2), dim3(32), 0, s, ctr, 1u << 20, status);
    note_launch();
    return err;
}

cudaError_t launch_route_layout(const RouteLayoutArgs& r, cudaStream_t s, bool* launched) {
    *launched = false;
    const LayoutArgs& a = r.lay;
    const int C = route_layout_chunk_tokens(a.N);
    const int slots = route_layout_chunk_slots(a.N, a.R);
    // workspace: chunk histograms [slots][E], barrier counters (64 ints, so
    // one memset zeroes both), expert totals [E]
    FusedArgs f;
    f.a = a;
    f.a.ws_hist = r.workspace;
    f.bar = reinterpret_cast<unsigned*>(r.workspace + (size_t)slots * a.E);
    f.a.ws_totals = r.workspace + (size_t)slots * a.E + 64;
    f.logits = r.logits;
    f.emap = r.emap;
    f.topk_idx = r.topk_idx;
    f.topk_w = r.topk_w;
    f.status = r.status;
    const bool vec = (a.E % 128 == 0) && ((reinterpret_cast<uintptr_t>(r.logits) & 15u) == 0);
    const size_t smem = (size_t)(2 * ((a.R + 1 + 3) & ~3) + 32 + ((a.E + 1 + 3) & ~3) +
                                 kWarps * (a.E > kNT ? a.E : kNT)) * sizeof(int);
    // phase 1 counts into the chunk histograms with atomics; the status word
    // is written by the kernel (0 by block 0 before the first barrier, 1 by
    // any block whose wait runs out)
    const cudaError_t err =
        cudaMemsetAsync(r.workspace, 0, ((size_t)slots * a.E + 64) * sizeof(int32_t), s);
    if (err != cudaSuccess) return err;
    const int K = a.K;
    if (vec && a.E == 256) {
        if (K == 8) return launch_fused_t<8, true, 8>(f, C, slots, smem, s, launched);
        if (K == 4) return launch_fused_t<8, true, 4>(f, C, slots, smem, s, launched);
        return launch_fused_t<8, true, 0>(f, C, slots, smem, s, launched);
    }
    if (vec && a.E == 128) {
        if (K == 8) return launch_fused_t<4, true, 8>(f, C, slots, smem, s, launched);
        if (K == 4) return launch_fused_t<4, true, 4>(f, C, slots, smem, s, launched);
        return launch_fused_t<4, true, 0>(f, C, slots, smem, s, launched);
    }
    if (vec && a.E == 512) return launch_fused_t<16, true, 0>(f, C, slots, smem, s, launched);
    if (vec && a.E == 1024) return launch_fused_t<32, true, 0>(f, C, slots, smem, s, launched);
    if (a.E <= 32) {
        if (K == 2) return launch_fused_t<1, false, 2>(f, C, slots, smem, s, launched);
        return launch_fused_t<1, false, 0>(f, C, slots, smem, s, launched);
    }
    if (a.E <= 64) return launch_fused_t<2, false, 0>(f, C, slots, smem, s, launched);
    if (a.E <= 128) return launch_fused_t<4, false, 0>(f, C, slots, smem, s, launched);
    if (a.E <= 256) return launch_fused_t<8, false, 0>(f, C, slots, smem, s, launched);
    return cudaSuccess;  // other sizes: not launched, the caller runs the two-step path
}

}  // namespace ep
