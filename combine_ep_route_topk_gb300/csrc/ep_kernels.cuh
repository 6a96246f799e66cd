// Internal declarations shared by the CUDA translation units of libep_gb300.
// Launchers enqueue kernels on a stream; argument checking happens in
// ep_api.cu before any of them is called.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace ep {

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
constexpr int kMaxR = 1024;

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Counts one kernel launch (ep_kernel_launch_count).
void note_launch(int n = 1);

// ---- routing -------------------------------------------------------------
cudaError_t launch_route_topk(const float* logits, int N, int E, int K, const int32_t* emap,
                              int32_t* topk_idx, float* topk_w, cudaStream_t s);

cudaError_t launch_balance_map(const int32_t* counts, int R, int E, int32_t* emap,
                               cudaStream_t s);

// ---- layout --------------------------------------------------------------
// Tokens per layout chunk; chunks never straddle a rank boundary.
int layout_chunk_tokens(int N);
// Upper bound on chunk slots: ceil(N / C) + R.
int layout_chunk_slots(int N, int R);
size_t layout_workspace_bytes(int N, int E, int K, int R);

struct LayoutArgs {
    const int32_t* topk_idx;
    const int32_t* rank_offsets;
    int R, N, E, K, cap;
    int32_t* counts;
    int32_t* expert_offsets;
    int32_t* rank_expert_offsets;
    int32_t* pos;
    int32_t* row_src;
    int32_t* masked_m;
    int32_t* overflow;
    int32_t* ws_hist;    // [slots, E] chunk histograms, then chunk prefixes
    int32_t* ws_totals;  // [E] expert totals
};
cudaError_t launch_layout(const LayoutArgs& a, cudaStream_t s);

// ---- fused route + layout (one cooperative kernel) ------------------------
int route_layout_chunk_tokens(int N);
int route_layout_chunk_slots(int N, int R);
// Workspace for the fused kernel and for the two-step fallback.
size_t route_layout_workspace_bytes(int N, int E, int K, int R);

struct RouteLayoutArgs {
    LayoutArgs lay;          // lay.topk_idx aliases topk_idx; lay.ws_* unused
    const float* logits;
    const int32_t* emap;
    int32_t* topk_idx;
    float* topk_w;
    int32_t* status;         // device int32 or nullptr
    int32_t* workspace;
};
// *launched is false when the sizes have no fused instance or the device
// cannot hold a block of it; the caller then runs route and layout kernels.
cudaError_t launch_route_layout(const RouteLayoutArgs& r, cudaStream_t s, bool* launched);

// ---- dispatch / combine --------------------------------------------------
struct MoveArgs {
    const void* src;            // x (dispatch) or y (combine)
    void* dst;                  // out
    float* scales;              // FP8 scales (dispatch) or nullptr
    const int32_t* topk_idx;
    const float* topk_w;        // combine only
    const int32_t* pos;
    const int32_t* expert_offsets;
    int N, H, E, K, cap;
    int layout;                 // 0 contiguous, 1 masked
    int dtype;                  // 0 bf16, 1 fp8 e4m3 1x128
};
cudaError_t launch_dispatch(const MoveArgs& a, cudaStream_t s);
cudaError_t launch_combine(const MoveArgs& a, cudaStream_t s);

}  // namespace ep
