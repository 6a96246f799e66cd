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

// ---- programmatic dependent launch -----------------------------------------
// Every kernel of the library starts with pdl_prologue(): it waits until the
// grids it depends on in the stream have completed and their writes are
// visible (griddepcontrol.wait, before any global load or store), then allows
// the next kernel of the stream to be launched (griddepcontrol.launch_
// dependents).  Kernels are launched with programmatic stream serialisation,
// so the next kernel's blocks are scheduled while this kernel's last wave
// runs and start their work the moment it ends, instead of after a launch
// gap.  Stream order and results are unchanged.  EP_DISABLE_PDL=1 in the
// environment turns the launch attribute off (plain stream order).
__device__ __forceinline__ void pdl_prologue() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

bool pdl_enabled();

template <typename... Params, typename... Args>
cudaError_t launch(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// Counts one kernel launch (ep_kernel_launch_count).
void note_launch(int n = 1);

// ---- routing -------------------------------------------------------------
cudaError_t launch_route_topk(const float* logits, int N, int E, int K, const int32_t* emap,
                              int32_t* topk_idx, float* topk_w, cudaStream_t s);

// Tokens routed per block of the route kernels (one warp each).
constexpr int kRouteTokensPerBlock = 8;
__host__ __device__ inline int route_chunks(int N) {
    return (N + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
}
// Route, plus per-block expert histograms H [E][C] and their exclusive
// prefixes over experts P [E][C] in hist (C = route_chunks(N); expert-major,
// so one expert's values over all blocks are contiguous); zeroes *zero_me
// (may be null).
cudaError_t launch_route_hist(const float* logits, int N, int E, int K, const int32_t* emap,
                              int32_t* topk_idx, float* topk_w, int32_t* hist,
                              int32_t* zero_me, cudaStream_t s);

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
// Small problems: the whole layout in one launch of one block per expert (no
// workspace), or in one thread-block cluster.
bool layout_small_fits(int N, int E, int K, int R);
cudaError_t launch_layout_small(const LayoutArgs& a, cudaStream_t s);
bool layout_cluster_fits(int N, int E, int K, int R);
cudaError_t launch_layout_cluster(const LayoutArgs& a, cudaStream_t s);
// EP_LAYOUT_CLUSTER=0 in the environment: the three layout kernels for every
// size (read at every call).
bool layout_kernels_forced();

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
// Self-test of the fused kernel's bounded grid-barrier wait (route_layout.cu).
cudaError_t launch_barrier_selftest(unsigned* ctr, int32_t* status, cudaStream_t s);

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

// ---- layout + dispatch after route_hist (ep_route_dispatch) ---------------
constexpr int kRouteDispatchMaxTokens = 2048;
struct RouteDispatchArgs {
    const int32_t* topk_idx;
    const int32_t* rank_offsets;
    const int32_t* hist;        // H [E][C], then P [E][C], from launch_route_hist
    int R, N, E, K, H, cap, C;
    int layout;                 // 0 contiguous, 1 masked
    int dtype;                  // 0 bf16, 1 fp8 e4m3 1x128
    int32_t* counts;
    int32_t* expert_offsets;
    int32_t* rank_expert_offsets;
    int32_t* pos;
    int32_t* row_src;
    int32_t* masked_m;
    int32_t* overflow;          // zeroed by launch_route_hist
    const void* x;
    void* out;
    float* scales;
};
// Sizes served by the two launches (at most 2048 tokens and 16384 picks).
bool route_dispatch_fits(int N, int E, int K, int R);
size_t route_dispatch_hist_bytes(int N, int E);
cudaError_t launch_route_dispatch(const RouteDispatchArgs& a, cudaStream_t s);

}  // namespace ep
