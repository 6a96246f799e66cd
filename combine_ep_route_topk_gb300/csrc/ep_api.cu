// C ABI of libep_gb300 (declared in include/ep.h): host-side argument checks,
// then kernel launches on the caller's stream.  Nothing here allocates,
// synchronises or reads device memory.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include "ep.h"
#include "ep_kernels.cuh"

namespace ep {

namespace {
std::atomic<uint64_t> g_launches{0};
thread_local char g_last_error[256] = {0};
std::atomic<int> g_sm_count[64];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

ep_status_t cuda_status(cudaError_t err) {
    if (err == cudaSuccess) return EP_OK;
    std::strncpy(g_last_error, cudaGetErrorString(err), sizeof(g_last_error) - 1);
    g_last_error[sizeof(g_last_error) - 1] = 0;
    return EP_ERR_CUDA;
}

// Shared limits of every entry point.
ep_status_t check_sizes(int32_t N, int32_t E, int32_t K) {
    if (N < 0 || E < 1 || K < 1) return EP_ERR_INVALID_ARG;
    if (K > E) return EP_ERR_INVALID_ARG;
    if (E > kMaxE || K > kMaxK) return EP_ERR_UNSUPPORTED;
    if ((int64_t)N * K > INT32_MAX) return EP_ERR_UNSUPPORTED;
    return EP_OK;
}
}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;  // GB300
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

void note_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("EP_DISABLE_PDL");
        return !(v && v[0] == '1');
    }();
    return on;
}

}  // namespace ep

using namespace ep;

extern "C" {

ep_status_t ep_route_topk(const float* logits, int32_t N, int32_t E, int32_t K,
                          const int32_t* expert_map, int32_t* topk_idx, float* topk_w,
                          void* stream) {
    ep_status_t st = check_sizes(N, E, K);
    if (st != EP_OK) return st;
    if (N > 0 && (!logits || !topk_idx || !topk_w)) return EP_ERR_INVALID_ARG;
    if (!aligned4(logits) || !aligned4(topk_idx) || !aligned4(topk_w) || !aligned4(expert_map))
        return EP_ERR_INVALID_ARG;
    return cuda_status(launch_route_topk(logits, N, E, K, expert_map, topk_idx, topk_w,
                                         static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_expert_balance_map(const int32_t* counts, int32_t R, int32_t E,
                                  int32_t* expert_map, void* stream) {
    if (R < 1 || E < 1 || !counts || !expert_map) return EP_ERR_INVALID_ARG;
    if (R > kMaxR || E > kMaxE) return EP_ERR_UNSUPPORTED;
    if (E % R != 0) return EP_ERR_INVALID_ARG;
    if (!aligned4(counts) || !aligned4(expert_map)) return EP_ERR_INVALID_ARG;
    return cuda_status(launch_balance_map(counts, R, E, expert_map,
                                          static_cast<cudaStream_t>(stream)));
}

size_t ep_dispatch_layout_workspace_size(int32_t N, int32_t E, int32_t K, int32_t R) {
    if (N < 0) N = 0;
    if (E < 1) E = 1;
    if (R < 1) R = 1;
    return layout_workspace_bytes(N, E, K, R);
}

ep_status_t ep_dispatch_layout(const int32_t* topk_idx, const int32_t* rank_offsets,
                               int32_t R, int32_t N, int32_t E, int32_t K, int32_t cap,
                               int32_t* counts, int32_t* expert_offsets,
                               int32_t* rank_expert_offsets, int32_t* pos, int32_t* row_src,
                               int32_t* masked_m, int32_t* overflow_count,
                               void* workspace, size_t ws_bytes, void* stream) {
    ep_status_t st = check_sizes(N, E, K);
    if (st != EP_OK) return st;
    if (R < 1) return EP_ERR_INVALID_ARG;
    if (R > kMaxR) return EP_ERR_UNSUPPORTED;
    if (cap < 0) return EP_ERR_INVALID_ARG;
    if ((masked_m || overflow_count) && cap == 0) return EP_ERR_INVALID_ARG;
    if (!rank_offsets || !counts || !expert_offsets || !rank_expert_offsets)
        return EP_ERR_INVALID_ARG;
    if (N > 0 && (!topk_idx || !pos || !row_src)) return EP_ERR_INVALID_ARG;
    const void* ptrs[] = {topk_idx, rank_offsets, counts, expert_offsets, rank_expert_offsets,
                          pos, row_src, masked_m, overflow_count};
    for (const void* p : ptrs)
        if (!aligned4(p)) return EP_ERR_INVALID_ARG;
    const size_t need = layout_workspace_bytes(N, E, K, R);
    if (!workspace || ws_bytes < need || !aligned16(workspace)) return EP_ERR_WORKSPACE;
    LayoutArgs a;
    a.topk_idx = topk_idx;
    a.rank_offsets = rank_offsets;
    a.R = R;
    a.N = N;
    a.E = E;
    a.K = K;
    a.cap = cap;
    a.counts = counts;
    a.expert_offsets = expert_offsets;
    a.rank_expert_offsets = rank_expert_offsets;
    a.pos = pos;
    a.row_src = row_src;
    a.masked_m = masked_m;
    a.overflow = overflow_count;
    a.ws_hist = static_cast<int32_t*>(workspace);
    a.ws_totals = a.ws_hist + (size_t)layout_chunk_slots(N, R) * E;
    return cuda_status(launch_layout(a, static_cast<cudaStream_t>(stream)));
}

size_t ep_route_layout_workspace_size(int32_t N, int32_t E, int32_t K, int32_t R) {
    if (N < 0) N = 0;
    if (E < 1) E = 1;
    if (R < 1) R = 1;
    return route_layout_workspace_bytes(N, E, K, R);
}

ep_status_t ep_route_layout(const float* logits, const int32_t* rank_offsets, int32_t R,
                            int32_t N, int32_t E, int32_t K, const int32_t* expert_map,
                            int32_t cap, int32_t* topk_idx, float* topk_w, int32_t* counts,
                            int32_t* expert_offsets, int32_t* rank_expert_offsets, int32_t* pos,
                            int32_t* row_src, int32_t* masked_m, int32_t* overflow_count,
                            int32_t* status, void* workspace, size_t ws_bytes, void* stream) {
    ep_status_t st = check_sizes(N, E, K);
    if (st != EP_OK) return st;
    if (R < 1) return EP_ERR_INVALID_ARG;
    if (R > kMaxR) return EP_ERR_UNSUPPORTED;
    if (cap < 0) return EP_ERR_INVALID_ARG;
    if ((masked_m || overflow_count) && cap == 0) return EP_ERR_INVALID_ARG;
    if (!rank_offsets || !counts || !expert_offsets || !rank_expert_offsets)
        return EP_ERR_INVALID_ARG;
    if (N > 0 && (!logits || !topk_idx || !topk_w || !pos || !row_src)) return EP_ERR_INVALID_ARG;
    const void* ptrs[] = {logits, rank_offsets, expert_map, topk_idx, topk_w, counts,
                          expert_offsets, rank_expert_offsets, pos, row_src, masked_m,
                          overflow_count, status};
    for (const void* p : ptrs)
        if (!aligned4(p)) return EP_ERR_INVALID_ARG;
    const size_t need = route_layout_workspace_bytes(N, E, K, R);
    if (!workspace || ws_bytes < need || !aligned16(workspace)) return EP_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    LayoutArgs a;
    a.topk_idx = topk_idx;
    a.rank_offsets = rank_offsets;
    a.R = R;
    a.N = N;
    a.E = E;
    a.K = K;
    a.cap = cap;
    a.counts = counts;
    a.expert_offsets = expert_offsets;
    a.rank_expert_offsets = rank_expert_offsets;
    a.pos = pos;
    a.row_src = row_src;
    a.masked_m = masked_m;
    a.overflow = overflow_count;
    a.ws_hist = nullptr;
    a.ws_totals = nullptr;
    RouteLayoutArgs r;
    r.lay = a;
    r.logits = logits;
    r.emap = expert_map;
    r.topk_idx = topk_idx;
    r.topk_w = topk_w;
    r.status = status;
    r.workspace = static_cast<int32_t*>(workspace);
    bool launched = false;
    cudaError_t err = launch_route_layout(r, s, &launched);
    if (err != cudaSuccess) return cuda_status(err);
    if (launched) return EP_OK;
    // no fused instance for these sizes: the same results from the two kernels
    if (status) err = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
    if (err != cudaSuccess) return cuda_status(err);
    err = launch_route_topk(logits, N, E, K, expert_map, topk_idx, topk_w, s);
    if (err != cudaSuccess) return cuda_status(err);
    a.ws_hist = static_cast<int32_t*>(workspace);
    a.ws_totals = a.ws_hist + (size_t)layout_chunk_slots(N, R) * E;
    return cuda_status(launch_layout(a, s));
}

static ep_status_t check_move(const void* src, int32_t N, int32_t H, int32_t E, int32_t K,
                              const int32_t* topk_idx, const int32_t* pos,
                              const int32_t* expert_offsets, ep_layout_t layout, int32_t cap,
                              const void* dst) {
    ep_status_t st = check_sizes(N, E, K);
    if (st != EP_OK) return st;
    if (H < 8 || H % 8 != 0) return EP_ERR_INVALID_ARG;
    if (layout != EP_LAYOUT_CONTIG && layout != EP_LAYOUT_MASKED) return EP_ERR_INVALID_ARG;
    if (layout == EP_LAYOUT_MASKED && cap < 1) return EP_ERR_INVALID_ARG;
    if (N > 0 && (!src || !topk_idx || !pos || !dst)) return EP_ERR_INVALID_ARG;
    if (N > 0 && layout == EP_LAYOUT_MASKED && !expert_offsets) return EP_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return EP_ERR_INVALID_ARG;
    if (!aligned4(topk_idx) || !aligned4(pos) || !aligned4(expert_offsets))
        return EP_ERR_INVALID_ARG;
    return EP_OK;
}

ep_status_t ep_dispatch(const void* x, int32_t N, int32_t H, int32_t E, int32_t K,
                        const int32_t* topk_idx, const int32_t* pos,
                        const int32_t* expert_offsets, ep_layout_t layout, int32_t cap,
                        ep_dtype_t dtype, void* out, float* out_scales, void* stream) {
    ep_status_t st = check_move(x, N, H, E, K, topk_idx, pos, expert_offsets, layout, cap, out);
    if (st != EP_OK) return st;
    if (dtype != EP_DTYPE_BF16 && dtype != EP_DTYPE_FP8_E4M3_B128) return EP_ERR_INVALID_ARG;
    if (dtype == EP_DTYPE_FP8_E4M3_B128) {
        if (H % 128 != 0) return EP_ERR_INVALID_ARG;
        if (N > 0 && !out_scales) return EP_ERR_INVALID_ARG;
        if (!aligned4(out_scales)) return EP_ERR_INVALID_ARG;
    }
    MoveArgs a;
    a.src = x;
    a.dst = out;
    a.scales = out_scales;
    a.topk_idx = topk_idx;
    a.topk_w = nullptr;
    a.pos = pos;
    a.expert_offsets = expert_offsets;
    a.N = N;
    a.H = H;
    a.E = E;
    a.K = K;
    a.cap = cap;
    a.layout = (int)layout;
    a.dtype = (int)dtype;
    return cuda_status(launch_dispatch(a, static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_combine(const void* y, int32_t N, int32_t H, int32_t E, int32_t K,
                       const int32_t* topk_idx, const float* topk_w, const int32_t* pos,
                       const int32_t* expert_offsets, ep_layout_t layout, int32_t cap,
                       void* out, void* stream) {
    ep_status_t st = check_move(y, N, H, E, K, topk_idx, pos, expert_offsets, layout, cap, out);
    if (st != EP_OK) return st;
    if (N > 0 && !topk_w) return EP_ERR_INVALID_ARG;
    if (!aligned4(topk_w)) return EP_ERR_INVALID_ARG;
    MoveArgs a;
    a.src = y;
    a.dst = out;
    a.scales = nullptr;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.pos = pos;
    a.expert_offsets = expert_offsets;
    a.N = N;
    a.H = H;
    a.E = E;
    a.K = K;
    a.cap = cap;
    a.layout = (int)layout;
    a.dtype = 0;
    return cuda_status(launch_combine(a, static_cast<cudaStream_t>(stream)));
}

size_t ep_route_dispatch_workspace_size(int32_t N, int32_t E, int32_t K, int32_t R) {
    if (N < 0) N = 0;
    if (E < 1) E = 1;
    if (R < 1) R = 1;
    if (K < 1) K = 1;
    size_t b = route_dispatch_fits(N, E, K, R) ? route_dispatch_hist_bytes(N, E)
                                               : layout_workspace_bytes(N, E, K, R);
    b = ((b + 255) / 256) * 256;
    return b > 0 ? b : 256;
}

ep_status_t ep_route_dispatch(const float* logits, const int32_t* rank_offsets, const void* x,
                              int32_t R, int32_t N, int32_t H, int32_t E, int32_t K,
                              const int32_t* expert_map, ep_layout_t layout, int32_t cap,
                              ep_dtype_t dtype, int32_t* topk_idx, float* topk_w,
                              int32_t* counts, int32_t* expert_offsets,
                              int32_t* rank_expert_offsets, int32_t* pos, int32_t* row_src,
                              int32_t* masked_m, int32_t* overflow_count, void* out,
                              float* out_scales, void* workspace, size_t ws_bytes,
                              void* stream) {
    ep_status_t st = check_sizes(N, E, K);
    if (st != EP_OK) return st;
    if (R < 1) return EP_ERR_INVALID_ARG;
    if (R > kMaxR) return EP_ERR_UNSUPPORTED;
    if (cap < 0) return EP_ERR_INVALID_ARG;
    if ((masked_m || overflow_count) && cap == 0) return EP_ERR_INVALID_ARG;
    if (layout != EP_LAYOUT_CONTIG && layout != EP_LAYOUT_MASKED) return EP_ERR_INVALID_ARG;
    if (layout == EP_LAYOUT_MASKED && cap < 1) return EP_ERR_INVALID_ARG;
    if (H < 8 || H % 8 != 0) return EP_ERR_INVALID_ARG;
    if (dtype != EP_DTYPE_BF16 && dtype != EP_DTYPE_FP8_E4M3_B128) return EP_ERR_INVALID_ARG;
    if (dtype == EP_DTYPE_FP8_E4M3_B128 && H % 128 != 0) return EP_ERR_INVALID_ARG;
    if (!rank_offsets || !counts || !expert_offsets || !rank_expert_offsets)
        return EP_ERR_INVALID_ARG;
    if (N > 0 && (!logits || !x || !topk_idx || !topk_w || !pos || !row_src || !out))
        return EP_ERR_INVALID_ARG;
    if (N > 0 && dtype == EP_DTYPE_FP8_E4M3_B128 && !out_scales) return EP_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out)) return EP_ERR_INVALID_ARG;
    const void* ptrs[] = {logits, rank_offsets, expert_map, topk_idx, topk_w, counts,
                          expert_offsets, rank_expert_offsets, pos, row_src, masked_m,
                          overflow_count, out_scales};
    for (const void* p : ptrs)
        if (!aligned4(p)) return EP_ERR_INVALID_ARG;
    const size_t need = ep_route_dispatch_workspace_size(N, E, K, R);
    if (!workspace || ws_bytes < need || !aligned16(workspace)) return EP_ERR_WORKSPACE;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (route_dispatch_fits(N, E, K, R)) {
        int32_t* hist = static_cast<int32_t*>(workspace);
        cudaError_t err = cudaSuccess;
        if (N > 0)
            err = launch_route_hist(logits, N, E, K, expert_map, topk_idx, topk_w, hist,
                                    cap > 0 ? overflow_count : nullptr, s);
        else if (overflow_count)
            err = cudaMemsetAsync(overflow_count, 0, sizeof(int32_t), s);
        if (err != cudaSuccess) return cuda_status(err);
        RouteDispatchArgs a;
        a.topk_idx = topk_idx;
        a.rank_offsets = rank_offsets;
        a.hist = hist;
        a.R = R;
        a.N = N;
        a.E = E;
        a.K = K;
        a.H = H;
        a.cap = cap;
        a.C = route_chunks(N);
        a.layout = (int)layout;
        a.dtype = (int)dtype;
        a.counts = counts;
        a.expert_offsets = expert_offsets;
        a.rank_expert_offsets = rank_expert_offsets;
        a.pos = pos;
        a.row_src = row_src;
        a.masked_m = masked_m;
        a.overflow = overflow_count;
        a.x = x;
        a.out = out;
        a.scales = out_scales;
        return cuda_status(launch_route_dispatch(a, s));
    }
    // larger problems: the route kernel, the layout kernels, the dispatch kernel
    cudaError_t err = launch_route_topk(logits, N, E, K, expert_map, topk_idx, topk_w, s);
    if (err != cudaSuccess) return cuda_status(err);
    LayoutArgs l;
    l.topk_idx = topk_idx;
    l.rank_offsets = rank_offsets;
    l.R = R;
    l.N = N;
    l.E = E;
    l.K = K;
    l.cap = cap;
    l.counts = counts;
    l.expert_offsets = expert_offsets;
    l.rank_expert_offsets = rank_expert_offsets;
    l.pos = pos;
    l.row_src = row_src;
    l.masked_m = masked_m;
    l.overflow = overflow_count;
    l.ws_hist = static_cast<int32_t*>(workspace);
    l.ws_totals = l.ws_hist + (size_t)layout_chunk_slots(N, R) * E;
    err = launch_layout(l, s);
    if (err != cudaSuccess) return cuda_status(err);
    MoveArgs m;
    m.src = x;
    m.dst = out;
    m.scales = out_scales;
    m.topk_idx = topk_idx;
    m.topk_w = nullptr;
    m.pos = pos;
    m.expert_offsets = expert_offsets;
    m.N = N;
    m.H = H;
    m.E = E;
    m.K = K;
    m.cap = cap;
    m.layout = (int)layout;
    m.dtype = (int)dtype;
    return cuda_status(launch_dispatch(m, s));
}

ep_status_t ep_selftest_wait_timeout(int32_t* status, void* workspace, size_t ws_bytes,
                                     void* stream) {
    if (!status || !workspace || ws_bytes < sizeof(unsigned)) return EP_ERR_INVALID_ARG;
    if (!aligned4(status) || !aligned4(workspace)) return EP_ERR_INVALID_ARG;
    return cuda_status(launch_barrier_selftest(static_cast<unsigned*>(workspace), status,
                                               static_cast<cudaStream_t>(stream)));
}

const char* ep_status_string(ep_status_t status) {
    switch (status) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
        case EP_ERR_WORKSPACE: return "EP_ERR_WORKSPACE";
        case EP_ERR_CUDA: return "EP_ERR_CUDA";
        case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED";
    }
    return "EP_ERR_UNKNOWN";
}

const char* ep_last_cuda_error(void) { return g_last_error; }

uint64_t ep_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t ep_abi_version(void) { return 1; }

}  // extern "C"
