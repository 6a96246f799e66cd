// Routing of one token by one warp, shared by the route kernel and the fused
// route + layout kernel.  "Anatomy of a High-Performance EP Kernel", "What we
// have to do": the token's length-E router logits select its K experts
// (descending logit, ties to the lower id); the weights are a softmax over
// the K picked logits.
//
// The E logits are read once with coalesced (16-byte when E is a multiple of
// 128) loads and held in registers; each lane caches its three best slots, and
// each of the K rounds is two warp reductions (redux.sync max of the lanes'
// head keys -- order-preserving 32-bit images of the logits -- then min of the
// expert id among lanes holding that key); the winning lane shifts its cache
// and rescans its registers only after a third win.
#pragma once

#include <cstdint>

namespace ep {
namespace route {

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

// Insert slot j (value x) into the sorted triple (s0,b0) >= (s1,b1) >= (s2,b2);
// later slots lose ties, so the order is (value desc, slot asc).
__device__ __forceinline__ void insert3(int j, float x, int& s0, float& b0, int& s1, float& b1,
                                        int& s2, float& b2) {
    if (s0 < 0 || x > b0) {
        s2 = s1; b2 = b1;
        s1 = s0; b1 = b0;
        s0 = j;  b0 = x;
    } else if (s1 < 0 || x > b1) {
        s2 = s1; b2 = b1;
        s1 = j;  b1 = x;
    } else if (s2 < 0 || x > b2) {
        s2 = j;  b2 = x;
    }
}


// Route the token whose logits start at `row`.  Every lane of the warp must
// call it.  Lanes k < K return pick k (expert id, -1 for none; after
// expert_map when given) and its weight; other lanes return -1 and 0.
template <int VPL, bool VEC, int KT>
__device__ __forceinline__ void route_token(const float* __restrict__ row, int E, int Kr,
                                            const int32_t* __restrict__ emap, int lane,
                                            int& out_id, float& out_w) {
    const int K = KT > 0 ? KT : Kr;

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

    // This lane's three best live slots in (value desc, slot asc) order,
    // found on the floats (-0 == +0 there).  A round is two warp reductions
    // and a shift of the winner's cache; a lane rescans its registers only
    // after its third win (for 8 of 256 picks about once in 20 tokens).
    int s0 = -1, s1 = -1, s2 = -1;
    float b0 = 0.0f, b1 = 0.0f, b2 = 0.0f;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
        if (live >> j & 1u) insert3(j, v[j], s0, b0, s1, b1, s2, b2);
    uint32_t head = s0 >= 0 ? order_key(b0) : 0u;
    uint32_t hid = s0 >= 0 ? expert_of<VPL, VEC>(lane, s0) : 0xffffffffu;

    uint32_t my_key = 0u, top_key = 0u;
    int my_id = -1;
#pragma unroll(KT > 0 ? KT : 1)
    for (int k = 0; k < K; ++k) {
        const uint32_t wmax = __reduce_max_sync(kFull, head);
        const uint32_t cand = (head == wmax && head != 0u) ? hid : 0xffffffffu;
        const uint32_t wid = __reduce_min_sync(kFull, cand);
        if (k == 0) top_key = wmax;
        if (lane == k) {
            my_key = wmax;
            my_id = (wid == 0xffffffffu) ? -1 : (int)wid;
        }
        const bool won = (cand == wid && cand != 0xffffffffu);  // this lane's head was taken
        const int ls = s0;
        const float lv = b0;
        if (won) {
            s0 = s1; b0 = b1;
            s1 = s2; b1 = b2;
            s2 = -1;
            head = s0 >= 0 ? order_key(b0) : 0u;
            hid = s0 >= 0 ? expert_of<VPL, VEC>(lane, s0) : 0xffffffffu;
        }
        // Rare: the winner used all three cached slots.  The vote keeps this a
        // real, warp-uniform branch instead of predicated code in every round.
        if (__any_sync(kFull, won && s0 < 0)) {
            if (won && s0 < 0) {  // the next three after (lv, ls)
#pragma unroll
                for (int j = 0; j < VPL; ++j) {
                    const bool after = (live >> j & 1u) && (v[j] < lv || (v[j] == lv && j > ls));
                    if (after) insert3(j, v[j], s0, b0, s1, b1, s2, b2);
                }
                head = s0 >= 0 ? order_key(b0) : 0u;
                hid = s0 >= 0 ? expert_of<VPL, VEC>(lane, s0) : 0xffffffffu;
            }
        }
    }

    float ex = 0.0f;
    if (lane < K && my_id >= 0) ex = expf(key_value(my_key) - key_value(top_key));
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
    out_id = -1;
    out_w = 0.0f;
    if (lane < K) {
        int id = my_id;
        if (id >= 0 && emap != nullptr) {
            id = __ldg(emap + id);
            if (id < 0 || id >= E) id = -1;
        }
        out_id = id;
        out_w = ex / sum;
    }
}

}  // namespace route
}  // namespace ep
