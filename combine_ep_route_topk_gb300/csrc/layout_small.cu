// Dispatch layout of a small (decode-sized) problem, one block per expert:
// "Anatomy of a High-Performance EP Kernel", "High throughput: ask first,
// then send" and "Dispatch" (every count and row position before any row
// moves); "Expert Parallelism" (SGLang docs), "Supported backends" (the
// low-latency mode, where the layout's latency is on the critical path).
//
// The stable counting sort of the picks by expert, split by expert instead
// of by token: block e (of E) reads all N*K ids once into registers (16 per
// lane up to 8192 picks, so that two blocks fit an SM, 32 up to 16384) and
// finds its own expert's picks with warp ballots, which keep (t, k) order:
//   1. per warp, over a contiguous range of ids: the number of valid ids
//      below e (summed over warps: expert_offsets[e]) and the ballot masks of
//      the ids equal to e, kept in registers;
//   2. lane r of each warp counts, from those masks, e's picks below rank r's
//      first token (r = 0..R); their sums over warps give counts[r][e] (the
//      difference of neighbours) and rank_expert_offsets[r][e];
//   3. the warps' exclusive prefix of e's picks gives each warp's first slot;
//      every pick then gets slot = warp base + running count + its rank within
//      the ballot, pos = expert_offsets[e] + slot and row_src[pos] = token.
// Block E handles what belongs to no expert: pos = -1 for invalid ids, the
// valid total expert_offsets[E], the -1 tail of row_src and the overflow
// (a shared histogram of all ids).  No block waits for another, nothing is
// counted with global atomics, and the result never depends on timing; two
// block barriers per block.
#include <cstdlib>

#include "layout_common.cuh"

namespace ep {
namespace {

using namespace lay;

constexpr int kST = 512;         // threads per block
constexpr int kSW = kST / 32;    // warps per block
constexpr long long kSmallMaxPicks = (long long)kSW * 32 * 32;  // 16384: 32 ids per lane

__device__ __forceinline__ int clamp_tok(int v, int N) { return v < 0 ? 0 : (v > N ? N : v); }

// Picks among the 32 of ballot mask m (ids first .. first + 31) whose index is
// below b.
__device__ __forceinline__ int picks_below(unsigned m, int first, int b) {
    const int n = b - first;
    if (n <= 0) return 0;
    if (n >= 32) return __popc(m);
    return __popc(m & ((1u << n) - 1u));
}

// Sum of v over the first `n` (<= 32) lanes of the warp; every lane gets it.
__device__ __forceinline__ int warp_sum_first(int v, int n, int lane) {
    int x = lane < n ? v : 0;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(kFull, x, off);
    return x;
}

// SC ids per lane (16 up to 8192 picks: two blocks fit an SM; else 32).
template <int SC>
__global__ void __launch_bounds__(kST, SC <= 16 ? 2 : 1) layout_small_kernel(LayoutArgs a) {
    pdl_prologue();
    extern __shared__ int smem[];
    const int R = a.R, E = a.E, K = a.K, N = a.N, NK = N * K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int e = blockIdx.x;
    // every block holds all ids: warp w a contiguous range, a multiple of 32
    // long, loaded before any store (stores to pos could alias the ids)
    const int span = ((NK + kSW * 32 - 1) / (kSW * 32)) * 32;
    const int base = warp * span;
    int v[SC];
#pragma unroll
    for (int s = 0; s < SC; ++s) {
        const int i = base + s * 32 + lane;
        v[s] = (s * 32 < span && i < NK) ? __ldg(a.topk_idx + i) : -1;
    }
    // the first 32 rank offsets, read now so their latency overlaps the ids'
    const int ro0 = (lane <= R) ? __ldg(a.rank_offsets + lane) : 0;

    if (e == E) {  // ---- what belongs to no expert
        int* s_hist = smem;                  // [E]
        int* s_cnt = smem + round_up4(E);    // [kSW] valid ids, then [kSW] drops
        const bool want_drop = a.cap > 0 && a.overflow != nullptr;
        if (want_drop)
            for (int j = threadIdx.x; j < E; j += kST) s_hist[j] = 0;
        __syncthreads();
        int valid = 0;
#pragma unroll
        for (int s = 0; s < SC; ++s) {
            const int x = v[s];
            const bool ok = x >= 0 && x < E;
            valid += __popc(__ballot_sync(kFull, ok));
            if (ok) {
                if (want_drop) atomicAdd(s_hist + x, 1);
            } else {
                const int i = base + s * 32 + lane;
                if (s * 32 < span && i < NK) a.pos[i] = -1;
            }
        }
        if (lane == 0) s_cnt[warp] = valid;
        __syncthreads();
        const int total = warp_sum_first(s_cnt[lane & (kSW - 1)], kSW, lane);
        if (threadIdx.x == 0) a.expert_offsets[E] = total;
        for (int p = total + threadIdx.x; p < NK; p += kST) a.row_src[p] = -1;
        if (want_drop) {
            int drop = 0;
            for (int j = threadIdx.x; j < E; j += kST) drop += max(0, s_hist[j] - a.cap);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) drop += __shfl_xor_sync(kFull, drop, off);
            if (lane == 0) s_cnt[kSW + warp] = drop;
            __syncthreads();
            if (warp == 0) {
                const int d = warp_sum_first(s_cnt[kSW + (lane & (kSW - 1))], kSW, lane);
                if (lane == 0) *a.overflow = d;
            }
        }
        return;
    }

    // ---- expert e
    int* s_bc = smem;                       // [R+1] picks of e below each rank start
    int* s_wb = s_bc + round_up4(R + 1);    // [kSW] ids below e, then [kSW] ids equal to e
    for (int r = threadIdx.x; r <= R; r += kST) s_bc[r] = 0;

    // 1. ballots: ids below e (the expert's offset) and e's picks, per warp
    unsigned m[SC];
    int below = 0, eq = 0;
#pragma unroll
    for (int s = 0; s < SC; ++s) {
        const int x = v[s];
        below += __popc(__ballot_sync(kFull, x >= 0 && x < e));
        m[s] = __ballot_sync(kFull, x == e);
        eq += __popc(m[s]);
    }
    __syncthreads();  // s_bc zeroed
    // 2. e's picks below each rank start o_r (r = 0..R), counted by lane r of
    //    every warp over the warp's range.  The rank starts are the rank
    //    offsets clamped to [0, N] and made non-decreasing (a running
    //    maximum, scanned 32 at a time with the previous chunk's carry).
    int carry = 0;
    for (int r0 = 0; r0 <= R; r0 += 32) {
        const int r = r0 + lane;
        int o = (r <= R) ? clamp_tok(r0 == 0 ? ro0 : __ldg(a.rank_offsets + r), N) : 0;
        o = max(o, carry);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(kFull, o, off);
            if (lane >= off) o = max(o, u);
        }
        carry = __shfl_sync(kFull, o, 31);
        if (r <= R && eq > 0) {
            const int b = o * K;
            int c = 0;
#pragma unroll
            for (int s = 0; s < SC; ++s) c += picks_below(m[s], base + s * 32, b);
            if (c) atomicAdd(s_bc + r, c);
        }
    }
    if (lane == 0) {
        s_wb[warp] = below;
        s_wb[kSW + warp] = eq;
    }
    __syncthreads();
    const int eoff = warp_sum_first(s_wb[lane & (kSW - 1)], kSW, lane);
    const int wbase = warp_sum_first(s_wb[kSW + (lane & (kSW - 1))], warp, lane);
    const int total = warp_sum_first(s_wb[kSW + (lane & (kSW - 1))], kSW, lane);

    // 3. positions of e's picks, in (t, k) order
    const unsigned lt = (1u << lane) - 1u;
    int run = wbase;
#pragma unroll
    for (int s = 0; s < SC; ++s) {
        if (m[s] != 0u) {  // warp-uniform
            if (m[s] >> lane & 1u) {
                const int i = base + s * 32 + lane;
                const int p = eoff + run + __popc(m[s] & lt);
                a.pos[i] = p;
                a.row_src[p] = i / K;
            }
            run += __popc(m[s]);
        }
    }

    // 4. the expert's column of counts and rank offsets
    for (int r = threadIdx.x; r < R; r += kST) {
        const int lo = s_bc[r], hi = s_bc[r + 1];
        a.counts[(size_t)r * E + e] = hi - lo;
        a.rank_expert_offsets[(size_t)r * E + e] = eoff + lo;
    }
    if (threadIdx.x == 0) {
        a.expert_offsets[e] = eoff;
        if (a.cap > 0 && a.masked_m) a.masked_m[e] = min(total, a.cap);
    }
}

}  // namespace

// Problems of at most 16384 picks.  EP_LAYOUT_SMALL=0 in the environment (read
// at every call) turns this path off, as EP_LAYOUT_CLUSTER=0 does (which
// forces the three kernels).
bool layout_small_fits(int N, int /*E*/, int K, int /*R*/) {
    const char* v = std::getenv("EP_LAYOUT_SMALL");
    if ((v && v[0] == '0') || layout_kernels_forced()) return false;
    return (long long)N * K <= kSmallMaxPicks;
}

cudaError_t launch_layout_small(const LayoutArgs& a, cudaStream_t s) {
    const int ints = round_up4(a.R + 1) + 2 * kSW;
    const int ints_e = round_up4(a.E) + 2 * kSW;
    const size_t smem = (size_t)(ints > ints_e ? ints : ints_e) * sizeof(int);
    if ((long long)a.N * a.K <= (long long)kSW * 32 * 16)
        return launch(layout_small_kernel<16>, dim3(a.E + 1), dim3(kST), smem, s, a);
    return launch(layout_small_kernel<32>, dim3(a.E + 1), dim3(kST), smem, s, a);
}

}  // namespace ep
