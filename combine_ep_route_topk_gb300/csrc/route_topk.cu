// Route top-K and balanced expert renumbering for sm_103a.
//
// route_topk: one warp per token runs route::route_token (route_common.cuh);
// HBM-bound on the N*E*4 logit bytes, issue-bound at small E.  route_hist:
// the same, plus each block's expert histogram and its prefix, for
// ep_route_dispatch.
//
// balance_map: "21K output tokens/s DeepSeek inference on AMD Instinct MI300X
// GPUs with Expert Parallelism", "Load balancing across GPUs" -- renumber
// experts so R contiguous sets of E/R have balanced activation frequency;
// a bitonic sort of (frequency desc, id asc) in shared memory, then one warp
// runs the greedy set assignment with a warp arg-min per expert.
#include <climits>

#include "ep_kernels.cuh"
#include "route_common.cuh"

namespace ep {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// One warp per token; KT > 0: K == KT known at compile time (rounds unrolled).
template <int VPL, bool VEC, int KT>
__global__ void __launch_bounds__(256)
route_topk_kernel(const float* __restrict__ logits, int N, int E, int Kr,
                  const int32_t* __restrict__ emap, int32_t* __restrict__ topk_idx,
                  float* __restrict__ topk_w) {
    pdl_prologue();
    const int K = KT > 0 ? KT : Kr;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= N) return;  // warp-uniform
    int id;
    float w;
    route::route_token<VPL, VEC, KT>(logits + (size_t)t * E, E, Kr, emap, lane, id, w);
    if (lane < K) {
        topk_idx[(size_t)t * K + lane] = id;
        topk_w[(size_t)t * K + lane] = w;
    }
}

// Route + the block's expert histogram, for ep_route_dispatch: block b routes
// tokens 8b .. 8b+7 (one warp each, as route_topk_kernel does) and writes
// H[e][b] (its picks of expert e) and P[e][b] (their exclusive prefix over
// experts) for every e, so that a later kernel can place any pick from these
// columns alone.  Block 0 zeroes *zero_me (the overflow counter that kernel
// accumulates into).
template <int VPL, bool VEC, int KT>
__global__ void __launch_bounds__(256)
route_hist_kernel(const float* __restrict__ logits, int N, int E, int Kr,
                  const int32_t* __restrict__ emap, int32_t* __restrict__ topk_idx,
                  float* __restrict__ topk_w, int32_t* __restrict__ hist, int C,
                  int32_t* zero_me) {
    __shared__ int s_h[kMaxE];
    __shared__ int s_tmp[32];
    pdl_prologue();
    const int K = KT > 0 ? KT : Kr;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kRouteTokensPerBlock + (threadIdx.x >> 5);
    for (int e = threadIdx.x; e < E; e += 256) s_h[e] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0 && zero_me) *zero_me = 0;
    __syncthreads();
    if (t < N) {  // warp-uniform
        int id;
        float w;
        route::route_token<VPL, VEC, KT>(logits + (size_t)t * E, E, Kr, emap, lane, id, w);
        if (lane < K) {
            topk_idx[(size_t)t * K + lane] = id;
            topk_w[(size_t)t * K + lane] = w;
            if (id >= 0) atomicAdd(s_h + id, 1);  // route_token returns -1 or an id < E
        }
    }
    __syncthreads();
    // expert-major: H[e][b] at hist[e * C + b], P[e][b] at hist[(E + e) * C + b],
    // so that a reader of one expert's column over all blocks loads it whole.
    // Thread j owns experts 4j .. 4j+3: their exclusive prefix is its local
    // prefix plus a warp scan of the threads' sums plus the earlier warps'.
    constexpr int kPer = kMaxE / 256;
    int h[kPer], sum = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = threadIdx.x * kPer + j;
        h[j] = (e < E) ? s_h[e] : 0;
        if (e < E) hist[(size_t)e * C + blockIdx.x] = h[j];
        sum += h[j];
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    const int warp = threadIdx.x >> 5;
    if (lane == 31) s_tmp[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += s_tmp[w];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int e = threadIdx.x * kPer + j;
        if (e < E) hist[((size_t)E + e) * C + blockIdx.x] = run;
        run += h[j];
    }
}

template <int VPL, bool VEC>
cudaError_t launch_hist(const float* logits, int N, int E, int K, const int32_t* emap,
                        int32_t* idx, float* w, int32_t* hist, int32_t* zero_me,
                        cudaStream_t s) {
    const int C = route_chunks(N);
    const dim3 grid(C > 0 ? C : 1), block(256);
    switch (K) {
        case 2: return launch(route_hist_kernel<VPL, VEC, 2>, grid, block, 0, s, logits, N, E, K, emap, idx, w, hist, C, zero_me);
        case 4: return launch(route_hist_kernel<VPL, VEC, 4>, grid, block, 0, s, logits, N, E, K, emap, idx, w, hist, C, zero_me);
        case 8: return launch(route_hist_kernel<VPL, VEC, 8>, grid, block, 0, s, logits, N, E, K, emap, idx, w, hist, C, zero_me);
        default: return launch(route_hist_kernel<VPL, VEC, 0>, grid, block, 0, s, logits, N, E, K, emap, idx, w, hist, C, zero_me);
    }
}

template <int VPL, bool VEC>
cudaError_t launch_route(const float* logits, int N, int E, int K, const int32_t* emap,
                         int32_t* idx, float* w, cudaStream_t s) {
    const dim3 grid((N + 7) / 8), block(256);
    switch (K) {
        case 2: return launch(route_topk_kernel<VPL, VEC, 2>, grid, block, 0, s, logits, N, E, K, emap, idx, w);
        case 4: return launch(route_topk_kernel<VPL, VEC, 4>, grid, block, 0, s, logits, N, E, K, emap, idx, w);
        case 8: return launch(route_topk_kernel<VPL, VEC, 8>, grid, block, 0, s, logits, N, E, K, emap, idx, w);
        default: return launch(route_topk_kernel<VPL, VEC, 0>, grid, block, 0, s, logits, N, E, K, emap, idx, w);
    }
}

// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(1024)
balance_map_kernel(const int32_t* __restrict__ counts, int R, int E, int32_t* __restrict__ emap) {
    pdl_prologue();
    __shared__ unsigned long long s_key[kMaxE];
    __shared__ long long s_load[kMaxR];
    __shared__ int s_size[kMaxR];
    const int tid = threadIdx.x;
    int P = 1;
    while (P < E) P <<= 1;
    // key ascending = (frequency descending, id ascending): 10 id bits under
    // 41 frequency bits (R <= 1024 counts below 2^31 sum to less than 2^41,
    // so every frequency is exact)
    constexpr long long kFreqTop = (1ll << 41) - 1;
    for (int e = tid; e < P; e += blockDim.x) {
        unsigned long long key = ~0ull;
        if (e < E) {
            long long f = 0;
            for (int r = 0; r < R; ++r) {
                const int c = counts[(size_t)r * E + e];
                f += c > 0 ? c : 0;
            }
            key = ((unsigned long long)(kFreqTop - f) << 10) | (unsigned long long)e;
        }
        s_key[e] = key;
    }
    for (int r = tid; r < R; r += blockDim.x) {
        s_load[r] = 0;
        s_size[r] = 0;
    }
    __syncthreads();
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < P; i += blockDim.x) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long a = s_key[i], b = s_key[ixj];
                    const bool up = (i & k) == 0;
                    if ((a > b) == up) {
                        s_key[i] = b;
                        s_key[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    if (tid >= 32) return;
    const int per = E / R;
    for (int i = 0; i < E; ++i) {
        const unsigned long long key = s_key[i];
        const int e = (int)(key & 1023ull);
        const long long f = kFreqTop - (long long)(key >> 10);
        long long bl = LLONG_MAX;
        int bs = INT_MAX;
        for (int s = tid; s < R; s += 32) {
            if (s_size[s] < per) {
                const long long l = s_load[s];
                if (l < bl || (l == bl && s < bs)) {
                    bl = l;
                    bs = s;
                }
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const long long ol = __shfl_xor_sync(kFull, bl, off);
            const int os = __shfl_xor_sync(kFull, bs, off);
            if (ol < bl || (ol == bl && os < bs)) {
                bl = ol;
                bs = os;
            }
        }
        if (tid == 0) {
            emap[e] = bs * per + s_size[bs];
            s_size[bs] += 1;
            s_load[bs] += f;
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int N, int E, int K, const int32_t* emap,
                              int32_t* idx, float* w, cudaStream_t s) {
    if (N == 0) return cudaSuccess;
    const bool vec = (E % 128 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
    cudaError_t err;
    if (vec && E == 128) err = launch_route<4, true>(logits, N, E, K, emap, idx, w, s);
    else if (vec && E == 256) err = launch_route<8, true>(logits, N, E, K, emap, idx, w, s);
    else if (vec && E == 512) err = launch_route<16, true>(logits, N, E, K, emap, idx, w, s);
    else if (vec && E == 1024) err = launch_route<32, true>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 32) err = launch_route<1, false>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 64) err = launch_route<2, false>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 128) err = launch_route<4, false>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 256) err = launch_route<8, false>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 512) err = launch_route<16, false>(logits, N, E, K, emap, idx, w, s);
    else err = launch_route<32, false>(logits, N, E, K, emap, idx, w, s);
    note_launch();
    return err;
}

cudaError_t launch_route_hist(const float* logits, int N, int E, int K, const int32_t* emap,
                              int32_t* idx, float* w, int32_t* hist, int32_t* zero_me,
                              cudaStream_t s) {
    const bool vec = (E % 128 == 0) && ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0);
    cudaError_t err;
    if (vec && E == 128) err = launch_hist<4, true>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else if (vec && E == 256) err = launch_hist<8, true>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else if (vec && E == 512) err = launch_hist<16, true>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else if (vec && E == 1024) err = launch_hist<32, true>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else if (E <= 32) err = launch_hist<1, false>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else if (E <= 64) err = launch_hist<2, false>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else if (E <= 128) err = launch_hist<4, false>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else if (E <= 256) err = launch_hist<8, false>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else if (E <= 512) err = launch_hist<16, false>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    else err = launch_hist<32, false>(logits, N, E, K, emap, idx, w, hist, zero_me, s);
    note_launch();
    return err;
}

cudaError_t launch_balance_map(const int32_t* counts, int R, int E, int32_t* emap,
                               cudaStream_t s) {
    const cudaError_t err = launch(balance_map_kernel, dim3(1), dim3(1024), 0, s, counts, R, E,
                                   emap);
    note_launch();
    return err;
}

}  // namespace ep
