// Route top-K and balanced expert renumbering for sm_103a.
//
// route_topk: "Anatomy of a High-Performance EP Kernel", "What we have to do"
// -- each token's length-E router logits select its K experts (the routing
// table's t0 row goes to experts [3, 13]); weights are a softmax over the K
// picked logits.  One warp per token: the E logits are read once with
// coalesced (16-byte when E is a multiple of 128) loads and held in
// registers as order-preserving 32-bit keys; each lane caches its two best
// keys, and each of the K rounds is two warp reductions (redux.sync max of
// the head keys, then min of the expert id among lanes holding that key, so
// ties go to the lower id); the winning lane advances its cache and rescans
// its registers only when both cached keys are used.  HBM-bound on the N*E*4
// logit bytes.
//
// balance_map: "21K output tokens/s DeepSeek inference on AMD Instinct MI300X
// GPUs with Expert Parallelism", "Load balancing across GPUs" -- renumber
// experts so R contiguous sets of E/R have balanced activation frequency;
// a bitonic sort of (frequency desc, id asc) in shared memory, then one warp
// runs the greedy set assignment with a warp arg-min per expert.
#include <climits>

#include "ep_kernels.cuh"

namespace ep {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Larger float -> larger key.  -0 folds onto +0 so equal logits tie; key 0 is
// reserved for "taken" (only the NaN pattern 0xffffffff would map there).
__device__ __forceinline__ uint32_t order_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
    return __uint_as_float(u);
}

// VPL logits per lane.  VEC: lane holds 4 consecutive experts of each
// 128-wide slab (16-byte loads); else expert lane + 32 j.  Slot j's expert id
// increases with j, so "lower slot" means "lower id" within a lane.
template <int VPL, bool VEC>
__device__ __forceinline__ uint32_t expert_of(int lane, int j) {
    return VEC ? (uint32_t)((j >> 2) * 128 + lane * 4 + (j & 3)) : (uint32_t)(lane + 32 * j);
}

template <int VPL, bool VEC>
__global__ void __launch_bounds__(256)
route_topk_kernel(const float* __restrict__ logits, int N, int E, int K,
                  const int32_t* __restrict__ emap, int32_t* __restrict__ topk_idx,
                  float* __restrict__ topk_w) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= N) return;  // warp-uniform
    const float* row = logits + (size_t)t * E;

    float v[VPL];
    if (VEC) {
#pragma unroll
        for (int s = 0; s < VPL / 4; ++s) {
            const float4 q = __ldcs(reinterpret_cast<const float4*>(row + s * 128 + lane * 4));
            v[4 * s + 0] = q.x;
            v[4 * s + 1] = q.y;
            v[4 * s + 2] = q.z;
            v[4 * s + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            v[j] = (e < E) ? __ldcs(row + e) : -INFINITY;
        }
    }
    // Present slots: all but the padding past E.
    uint32_t live = 0u;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
        if (VEC || lane + 32 * j < E) live |= 1u << j;

    // This lane's two best live slots in (value desc, slot asc) order, found
    // on the floats (-0 == +0 there); b1/b2 are their values.  A lane
    // rescans its registers only after its second win (for 8 of 256 picks,
    // under once per token on average); otherwise a round is two warp
    // reductions and a few selects.
    int s1 = -1, s2 = -1;
    float b1 = 0.0f, b2 = 0.0f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
        if (!(live >> j & 1u)) continue;
        if (s1 < 0 || v[j] > b1) {
            s2 = s1; b2 = b1;
            s1 = j;  b1 = v[j];
        } else if (s2 < 0 || v[j] > b2) {
            s2 = j;  b2 = v[j];
        }
    }
    uint32_t k1 = s1 >= 0 ? order_key(b1) : 0u;
    uint32_t k2 = s2 >= 0 ? order_key(b2) : 0u;
    uint32_t id1 = s1 >= 0 ? expert_of<VPL, VEC>(lane, s1) : 0xffffffffu;
    uint32_t id2 = s2 >= 0 ? expert_of<VPL, VEC>(lane, s2) : 0xffffffffu;

    uint32_t my_key = 0u, top_key = 0u;
    int my_id = -1;
    for (int k = 0; k < K; ++k) {
        const uint32_t wmax = __reduce_max_sync(kFull, k1);
        const uint32_t cand = (k1 == wmax && k1 != 0u) ? id1 : 0xffffffffu;
        const uint32_t wid = __reduce_min_sync(kFull, cand);
        if (k == 0) top_key = wmax;
        if (lane == k) {
            my_key = wmax;
            my_id = (wid == 0xffffffffu) ? -1 : (int)wid;
        }
        if (cand == wid && cand != 0xffffffffu) {  // this lane's head was taken
            const int ls = s1;
            const float lv = b1;
            k1 = k2; id1 = id2; s1 = s2; b1 = b2;
            k2 = 0u; id2 = 0xffffffffu; s2 = -1;
            if (s1 < 0) {  // both cached slots used: the next two after (lv, ls)
#pragma unroll
                for (int j = 0; j < VPL; ++j) {
                    const bool after = (live >> j & 1u) && (v[j] < lv || (v[j] == lv && j > ls));
                    if (!after) continue;
                    if (s1 < 0 || v[j] > b1) {
                        s2 = s1; b2 = b1;
                        s1 = j;  b1 = v[j];
                    } else if (s2 < 0 || v[j] > b2) {
                        s2 = j;  b2 = v[j];
                    }
                }
                k1 = s1 >= 0 ? order_key(b1) : 0u;
                k2 = s2 >= 0 ? order_key(b2) : 0u;
                id1 = s1 >= 0 ? expert_of<VPL, VEC>(lane, s1) : 0xffffffffu;
                id2 = s2 >= 0 ? expert_of<VPL, VEC>(lane, s2) : 0xffffffffu;
            }
        }
    }

    float ex = 0.0f;
    if (lane < K && my_id >= 0) ex = expf(key_value(my_key) - key_value(top_key));
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    if (lane < K) {
        int id = my_id;
        if (id >= 0 && emap != nullptr) {
            id = __ldg(emap + id);
            if (id < 0 || id >= E) id = -1;
        }
        topk_idx[(size_t)t * K + lane] = id;
        topk_w[(size_t)t * K + lane] = ex / sum;
    }
}

template <int VPL, bool VEC>
void launch_route(const float* logits, int N, int E, int K, const int32_t* emap,
                  int32_t* idx, float* w, cudaStream_t s) {
    const int blocks = (N + 7) / 8;
    route_topk_kernel<VPL, VEC><<<blocks, 256, 0, s>>>(logits, N, E, K, emap, idx, w);
}

// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(1024)
balance_map_kernel(const int32_t* __restrict__ counts, int R, int E, int32_t* __restrict__ emap) {
    __shared__ unsigned long long s_key[kMaxE];
    __shared__ long long s_load[kMaxR];
    __shared__ int s_size[kMaxR];
    const int tid = threadIdx.x;
    int P = 1;
    while (P < E) P <<= 1;
    // key ascending = (frequency descending, id ascending); 10 id bits
    for (int e = tid; e < P; e += blockDim.x) {
        unsigned long long key = ~0ull;
        if (e < E) {
            long long f = 0;
            for (int r = 0; r < R; ++r) {
                const int c = counts[(size_t)r * E + e];
                f += c > 0 ? c : 0;
            }
            if (f > 0xffffffffll) f = 0xffffffffll;
            key = ((unsigned long long)(0xffffffffll - f) << 10) | (unsigned long long)e;
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
        const long long f = 0xffffffffll - (long long)(key >> 10);
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
    if (vec) {
        switch (E) {
            case 128: launch_route<4, true>(logits, N, E, K, emap, idx, w, s); break;
            case 256: launch_route<8, true>(logits, N, E, K, emap, idx, w, s); break;
            case 512: launch_route<16, true>(logits, N, E, K, emap, idx, w, s); break;
            case 1024: launch_route<32, true>(logits, N, E, K, emap, idx, w, s); break;
            default: goto scalar;
        }
        note_launch();
        return cudaGetLastError();
    }
scalar:
    if (E <= 32) launch_route<1, false>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 64) launch_route<2, false>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 128) launch_route<4, false>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 256) launch_route<8, false>(logits, N, E, K, emap, idx, w, s);
    else if (E <= 512) launch_route<16, false>(logits, N, E, K, emap, idx, w, s);
    else launch_route<32, false>(logits, N, E, K, emap, idx, w, s);
    note_launch();
    return cudaGetLastError();
}

cudaError_t launch_balance_map(const int32_t* counts, int R, int E, int32_t* emap,
                               cudaStream_t s) {
    balance_map_kernel<<<1, 1024, 0, s>>>(counts, R, E, emap);
    note_launch();
    return cudaGetLastError();
}

}  // namespace ep
