// ep_dispatch_layout_static: the dispatch layout with its scratch memory held
// inside the library, for callers that cannot allocate device memory.
//
// ep_dispatch_layout needs a workspace of chunk histograms and expert totals
// that the caller allocates.  Some callers cannot do that: an embedder whose
// device memory is all reserved up front by another allocator, a plain C
// host with no device allocator of its own, or code running where a call to
// cudaMalloc is not permitted.  This variant takes the same inputs and
// outputs but no workspace: its scratch is the fixed array below, which
// every GPU that loads the library holds until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  The layout kernels write every scratch entry they later read
// (each live chunk writes its whole histogram row, the column scan writes
// every total), so nothing has to start at zero and nothing is cleared.
// Calls whose work overlaps on the GPU (two streams, or two host threads)
// race on the array; order them on one stream.
#include <mutex>

#include "ep.h"
#include "ep_kernels.cuh"

namespace {

constexpr size_t kScratchBytes = EP_LAYOUT_STATIC_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) unsigned char g_layout_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The symbol's
// host-side name is only a stand-in, so its address is asked for once per
// device, with that device current, and cached.
cudaError_t scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" ep_status_t ep_dispatch_layout_static(
    const int32_t* topk_idx, const int32_t* rank_offsets, int32_t R, int32_t N, int32_t E,
    int32_t K, int32_t cap, int32_t* counts, int32_t* expert_offsets,
    int32_t* rank_expert_offsets, int32_t* pos, int32_t* row_src, int32_t* masked_m,
    int32_t* overflow_count, void* stream) {
    if (N < 0 || E < 1 || K < 1 || K > E || R < 1 || cap < 0) return EP_ERR_INVALID_ARG;
    if (E > ep::kMaxE || K > ep::kMaxK || R > ep::kMaxR) return EP_ERR_UNSUPPORTED;
    if ((int64_t)N * K > INT32_MAX) return EP_ERR_UNSUPPORTED;
    if ((masked_m || overflow_count) && cap == 0) return EP_ERR_INVALID_ARG;
    if (!rank_offsets || !counts || !expert_offsets || !rank_expert_offsets)
        return EP_ERR_INVALID_ARG;
    if (N > 0 && (!topk_idx || !pos || !row_src)) return EP_ERR_INVALID_ARG;
    const void* ptrs[] = {topk_idx, rank_offsets, counts, expert_offsets, rank_expert_offsets,
                          pos, row_src, masked_m, overflow_count};
    for (const void* p : ptrs)
        if (!aligned4(p)) return EP_ERR_INVALID_ARG;
    // sizes whose scratch would not fit the fixed array are refused
    if (ep::layout_workspace_bytes(N, E, K, R) > kScratchBytes) return EP_ERR_UNSUPPORTED;

    void* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return EP_ERR_CUDA;

    ep::LayoutArgs a;
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
    a.ws_hist = static_cast<int32_t*>(scratch);
    a.ws_totals = a.ws_hist + (size_t)ep::layout_chunk_slots(N, R) * E;
    return ep::launch_layout(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? EP_OK
                                                                                   : EP_ERR_CUDA;
}
