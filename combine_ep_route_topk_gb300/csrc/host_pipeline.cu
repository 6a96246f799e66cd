// Steps over host buffers (include/ep.h, ep_host_pipeline_*): route -> layout
// -> dispatch -> combine whose inputs and result live in host memory.  Copies
// in, kernels and copies out run on three streams; `depth` sets of device
// input and result buffers rotate, so step i + 1's copies in run under step
// i's kernels and copy out.  A set is reused only after the kernels and the
// copy out of the step that last used it are done (events).  Every device
// buffer is carved from the caller's workspace; the object holds only its
// streams and events.  The host link, not HBM, bounds such a step.
//
// ep_host_alloc / ep_host_free give the host side page-locked memory backed by
// transparent huge pages: on 64 KB base pages the kernel periodically
// reactivates the pages of ordinary pinned buffers, and every copy that
// overlapped such an event was measured at a quarter or less of the link's
// 211 GB/s; copies from huge-page buffers did not slow.
#include <sys/mman.h>
#include <unistd.h>

#include <cstddef>
#include <cstdio>
#include <cstdint>
#include <map>
#include <mutex>
#include <new>

#include "ep.h"
#include "ep_kernels.cuh"

namespace {

constexpr int kMaxDepth = 4;

// Buffers of the workspace, in carve order; the per-set ones repeat.
enum Piece {
    P_IDX, P_W, P_COUNTS, P_EOFF, P_REOFF, P_POS, P_ROWSRC, P_MASKEDM, P_OVERFLOW, P_LAYWS,
    P_OUT, P_SCALES, P_SHARED,  // then per set: logits, rank offsets, x, y, result
};
enum SetPiece { S_LOGITS, S_RO, S_X, S_Y, S_COMB, S_PIECES };

struct Dims {
    int N, E, K, H, R, cap, depth;
    ep_dtype_t dtype;
};

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

size_t rows_of(const Dims& d) {
    return d.cap > 0 ? (size_t)d.E * d.cap : (size_t)d.N * d.K;
}

// Byte size of piece p (set pieces: p = P_SHARED + s * S_PIECES + q).
size_t piece_bytes(const Dims& d, int p) {
    const size_t N = d.N, E = d.E, K = d.K, H = d.H, R = d.R;
    const bool fp8 = d.dtype == EP_DTYPE_FP8_E4M3_B128;
    switch (p) {
        case P_IDX: return N * K * 4;
        case P_W: return N * K * 4;
        case P_COUNTS: return R * E * 4;
        case P_EOFF: return (E + 1) * 4;
        case P_REOFF: return R * E * 4;
        case P_POS: return N * K * 4;
        case P_ROWSRC: return N * K * 4;
        case P_MASKEDM: return d.cap > 0 ? E * 4 : 0;
        case P_OVERFLOW: return d.cap > 0 ? 4 : 0;
        case P_LAYWS: return ep_dispatch_layout_workspace_size(d.N, d.E, d.K, d.R);
        case P_OUT: return rows_of(d) * H * (fp8 ? 1 : 2);
        case P_SCALES: return fp8 ? rows_of(d) * (H / 128) * 4 : 0;
        default: break;
    }
    switch ((p - P_SHARED) % S_PIECES) {
        case S_LOGITS: return N * E * 4;
        case S_RO: return (R + 1) * 4;
        case S_X: return N * H * 2;
        case S_Y: return rows_of(d) * H * 2;
        default: return N * H * 2;  // S_COMB
    }
}

int piece_count(const Dims& d) { return P_SHARED + d.depth * S_PIECES; }

// Offset of piece p; every piece starts on a 256-byte boundary.
size_t piece_offset(const Dims& d, int p) {
    size_t off = 0;
    for (int i = 0; i < p; ++i) off += round256(piece_bytes(d, i));
    return off;
}

ep_status_t check_dims(const Dims& d) {
    if (d.N < 1 || d.E < 1 || d.K < 1 || d.H < 8 || d.R < 1) return EP_ERR_INVALID_ARG;
    if (d.K > d.E || d.H % 8 != 0 || d.cap < 0) return EP_ERR_INVALID_ARG;
    if (d.depth < 1) return EP_ERR_INVALID_ARG;
    if (d.dtype != EP_DTYPE_BF16 && d.dtype != EP_DTYPE_FP8_E4M3_B128) return EP_ERR_INVALID_ARG;
    if (d.dtype == EP_DTYPE_FP8_E4M3_B128 && d.H % 128 != 0) return EP_ERR_INVALID_ARG;
    if (d.depth > kMaxDepth || d.E > ep::kMaxE || d.K > ep::kMaxK || d.R > ep::kMaxR)
        return EP_ERR_UNSUPPORTED;
    if ((int64_t)d.N * d.K > INT32_MAX) return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

ep_status_t cuda_st(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

// Huge-page size of transparent huge pages (PMD size), or 2 MiB if unknown.
size_t huge_page_bytes() {
    size_t v = 0;
    if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
        unsigned long long u = 0;
        if (std::fscanf(f, "%llu", &u) == 1) v = (size_t)u;
        std::fclose(f);
    }
    const size_t page = (size_t)sysconf(_SC_PAGESIZE);
    if (v < page || (v & (v - 1)) != 0) v = (size_t)2 << 20;
    return v;
}

// Live ep_host_alloc mappings: returned pointer -> (mapping start, length).
struct HostMapping {
    void* base;
    size_t len;
};
std::mutex g_host_mutex;
std::map<void*, HostMapping>& host_mappings() {
    static std::map<void*, HostMapping> m;
    return m;
}

}  // namespace

struct ep_host_pipeline {
    Dims d;
    const int32_t* emap;
    char* ws;
    int device;
    cudaStream_t h2d, comp, d2h;
    cudaEvent_t caller;  // the caller's stream at the start of a step
    struct Set {
        cudaEvent_t routed_in, x_in, y_in, inputs_free, result_free;
        // timing: the start of the copies in (their end is y_in) and of the
        // copy out (its end is result_free)
        cudaEvent_t in_start, out_start;
        bool used;
    } set[kMaxDepth];
    uint64_t steps;

    template <typename T>
    T* at(int p) { return reinterpret_cast<T*>(ws + piece_offset(d, p)); }
    template <typename T>
    T* set_at(int s, int q) { return at<T>(P_SHARED + s * S_PIECES + q); }
};

namespace {

void destroy_handles(ep_host_pipeline* p) {
    for (int s = 0; s < kMaxDepth; ++s) {
        ep_host_pipeline::Set& S = p->set[s];
        cudaEvent_t* evs[] = {&S.routed_in, &S.x_in,      &S.y_in,     &S.inputs_free,
                              &S.result_free, &S.in_start, &S.out_start};
        for (cudaEvent_t* e : evs)
            if (*e) cudaEventDestroy(*e);
    }
    if (p->caller) cudaEventDestroy(p->caller);
    cudaStream_t* sts[] = {&p->h2d, &p->comp, &p->d2h};
    for (cudaStream_t* s : sts)
        if (*s) cudaStreamDestroy(*s);
}

}  // namespace

extern "C" {

ep_status_t ep_host_alloc(size_t bytes, void** out) {
    if (!out) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    if (bytes == 0) return EP_ERR_INVALID_ARG;
    const size_t hp = huge_page_bytes();
    if (bytes > SIZE_MAX - 2 * hp) return EP_ERR_INVALID_ARG;
    const size_t len = (bytes + hp - 1) / hp * hp;
    // map one huge page more, so an aligned start exists inside the mapping
    const size_t map_len = len + hp;
    void* base = mmap(nullptr, map_len, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (base == MAP_FAILED) return EP_ERR_CUDA;
    const uintptr_t b = reinterpret_cast<uintptr_t>(base);
    char* p = reinterpret_cast<char*>((b + hp - 1) / hp * hp);
    madvise(p, len, MADV_HUGEPAGE);  // best effort: base pages if refused
    // touch every base page so the memory exists (as huge pages where
    // granted) before it is locked
    const size_t page = (size_t)sysconf(_SC_PAGESIZE);
    for (size_t off = 0; off < len; off += page) p[off] = 0;
    if (cudaHostRegister(p, len, cudaHostRegisterPortable) != cudaSuccess) {
        cudaGetLastError();
        munmap(base, map_len);
        return EP_ERR_CUDA;
    }
    {
        std::lock_guard<std::mutex> lock(g_host_mutex);
        host_mappings()[p] = HostMapping{base, map_len};
    }
    *out = p;
    return EP_OK;
}

ep_status_t ep_host_free(void* ptr) {
    if (!ptr) return EP_OK;
    HostMapping m;
    {
        std::lock_guard<std::mutex> lock(g_host_mutex);
        auto it = host_mappings().find(ptr);
        if (it == host_mappings().end()) return EP_ERR_INVALID_ARG;
        m = it->second;
        host_mappings().erase(it);
    }
    const cudaError_t e = cudaHostUnregister(ptr);
    munmap(m.base, m.len);
    return cuda_st(e);
}

size_t ep_host_pipeline_workspace_size(int32_t N, int32_t E, int32_t K, int32_t H, int32_t R,
                                       int32_t cap, ep_dtype_t dtype, int32_t depth) {
    const Dims d{N, E, K, H, R, cap, depth, dtype};
    if (check_dims(d) != EP_OK) return 0;
    return piece_offset(d, piece_count(d));
}

ep_status_t ep_host_pipeline_create(int32_t N, int32_t E, int32_t K, int32_t H, int32_t R,
                                    int32_t cap, ep_dtype_t dtype, int32_t depth,
                                    const int32_t* expert_map, void* workspace, size_t ws_bytes,
                                    ep_host_pipeline_t** out) {
    if (!out) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    const Dims d{N, E, K, H, R, cap, depth, dtype};
    const ep_status_t st = check_dims(d);
    if (st != EP_OK) return st;
    if ((reinterpret_cast<uintptr_t>(expert_map) & 3u) != 0) return EP_ERR_INVALID_ARG;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
        ws_bytes < piece_offset(d, piece_count(d)))
        return EP_ERR_WORKSPACE;
    ep_host_pipeline* p = new (std::nothrow) ep_host_pipeline();
    if (!p) return EP_ERR_UNSUPPORTED;
    p->d = d;
    p->emap = expert_map;
    p->ws = static_cast<char*>(workspace);
    p->steps = 0;
    cudaError_t e = cudaGetDevice(&p->device);
    const unsigned ev_flags = cudaEventDisableTiming;
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->comp, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->caller, ev_flags);
    for (int s = 0; s < depth && e == cudaSuccess; ++s) {
        ep_host_pipeline::Set& S = p->set[s];
        S.used = false;
        cudaEvent_t* evs[] = {&S.routed_in, &S.x_in, &S.inputs_free};
        for (cudaEvent_t* ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, ev_flags);
        cudaEvent_t* timed[] = {&S.y_in, &S.result_free, &S.in_start, &S.out_start};
        for (cudaEvent_t* ev : timed)
            if (e == cudaSuccess) e = cudaEventCreate(ev);
    }
    if (e != cudaSuccess) {
        destroy_handles(p);
        delete p;
        return EP_ERR_CUDA;
    }
    *out = p;
    return EP_OK;
}

ep_status_t ep_host_pipeline_step(ep_host_pipeline_t* p, const float* logits_h,
                                  const int32_t* rank_offsets_h, const void* x_h,
                                  const void* y_h, void* out_h, void* stream) {
    if (!p || !logits_h || !rank_offsets_h || !x_h || !y_h || !out_h) return EP_ERR_INVALID_ARG;
    const Dims& d = p->d;
    const int j = (int)(p->steps % (uint64_t)d.depth);
    ep_host_pipeline::Set& S = p->set[j];
    float* logits = p->set_at<float>(j, S_LOGITS);
    int32_t* ro = p->set_at<int32_t>(j, S_RO);
    void* x = p->set_at<char>(j, S_X);
    void* y = p->set_at<char>(j, S_Y);
    void* comb = p->set_at<char>(j, S_COMB);
    const int PS = P_SHARED + j * S_PIECES;
    const cudaStream_t caller = static_cast<cudaStream_t>(stream);

    // every stream starts after what the caller enqueued before this step
    ep_status_t st = cuda_st(cudaEventRecord(p->caller, caller));
    cudaStream_t sts[] = {p->h2d, p->comp, p->d2h};
    for (cudaStream_t s : sts)
        if (st == EP_OK) st = cuda_st(cudaStreamWaitEvent(s, p->caller, 0));
    // copies in, once the kernels of this set's last step are done with it
    if (st == EP_OK && S.used) st = cuda_st(cudaStreamWaitEvent(p->h2d, S.inputs_free, 0));
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice;
    if (st == EP_OK) st = cuda_st(cudaEventRecord(S.in_start, p->h2d));
    if (st == EP_OK)
        st = cuda_st(cudaMemcpyAsync(logits, logits_h, piece_bytes(d, PS + S_LOGITS), h2d, p->h2d));
    if (st == EP_OK)
        st = cuda_st(cudaMemcpyAsync(ro, rank_offsets_h, piece_bytes(d, PS + S_RO), h2d, p->h2d));
    if (st == EP_OK) st = cuda_st(cudaEventRecord(S.routed_in, p->h2d));
    if (st == EP_OK) st = cuda_st(cudaMemcpyAsync(x, x_h, piece_bytes(d, PS + S_X), h2d, p->h2d));
    if (st == EP_OK) st = cuda_st(cudaEventRecord(S.x_in, p->h2d));
    if (st == EP_OK) st = cuda_st(cudaMemcpyAsync(y, y_h, piece_bytes(d, PS + S_Y), h2d, p->h2d));
    if (st == EP_OK) st = cuda_st(cudaEventRecord(S.y_in, p->h2d));
    if (st != EP_OK) return st;

    // kernels
    const ep_layout_t layout = d.cap > 0 ? EP_LAYOUT_MASKED : EP_LAYOUT_CONTIG;
    int32_t* idx = p->at<int32_t>(P_IDX);
    float* w = p->at<float>(P_W);
    int32_t* pos = p->at<int32_t>(P_POS);
    int32_t* eoff = p->at<int32_t>(P_EOFF);
    st = cuda_st(cudaStreamWaitEvent(p->comp, S.routed_in, 0));
    if (st == EP_OK) st = ep_route_topk(logits, d.N, d.E, d.K, p->emap, idx, w, p->comp);
    if (st == EP_OK)
        st = ep_dispatch_layout(idx, ro, d.R, d.N, d.E, d.K, d.cap, p->at<int32_t>(P_COUNTS), eoff,
                                p->at<int32_t>(P_REOFF), pos, p->at<int32_t>(P_ROWSRC),
                                d.cap > 0 ? p->at<int32_t>(P_MASKEDM) : nullptr,
                                d.cap > 0 ? p->at<int32_t>(P_OVERFLOW) : nullptr,
                                p->at<char>(P_LAYWS), piece_bytes(d, P_LAYWS), p->comp);
    if (st == EP_OK) st = cuda_st(cudaStreamWaitEvent(p->comp, S.x_in, 0));
    if (st == EP_OK)
        st = ep_dispatch(x, d.N, d.H, d.E, d.K, idx, pos, eoff, layout, d.cap, d.dtype,
                         p->at<char>(P_OUT),
                         d.dtype == EP_DTYPE_FP8_E4M3_B128 ? p->at<float>(P_SCALES) : nullptr,
                         p->comp);
    if (st == EP_OK) st = cuda_st(cudaStreamWaitEvent(p->comp, S.y_in, 0));
    // the result buffer is rewritten only after its last copy out is done
    if (st == EP_OK && S.used) st = cuda_st(cudaStreamWaitEvent(p->comp, S.result_free, 0));
    if (st == EP_OK)
        st = ep_combine(y, d.N, d.H, d.E, d.K, idx, w, pos, eoff, layout, d.cap, comb, p->comp);
    if (st == EP_OK) st = cuda_st(cudaEventRecord(S.inputs_free, p->comp));
    if (st != EP_OK) return st;

    // copy out
    st = cuda_st(cudaStreamWaitEvent(p->d2h, S.inputs_free, 0));
    if (st == EP_OK) st = cuda_st(cudaEventRecord(S.out_start, p->d2h));
    if (st == EP_OK)
        st = cuda_st(cudaMemcpyAsync(out_h, comb, piece_bytes(d, PS + S_COMB),
                                     cudaMemcpyDeviceToHost, p->d2h));
    if (st == EP_OK) st = cuda_st(cudaEventRecord(S.result_free, p->d2h));
    if (st != EP_OK) return st;
    S.used = true;
    p->steps += 1;
    return EP_OK;
}

ep_status_t ep_host_pipeline_copy_ms(const ep_host_pipeline_t* p, float* h2d_ms,
                                     float* d2h_ms) {
    if (!p || !h2d_ms || !d2h_ms) return EP_ERR_INVALID_ARG;
    *h2d_ms = *d2h_ms = 0.0f;
    if (p->steps == 0) return EP_ERR_INVALID_ARG;
    const ep_host_pipeline::Set& S = p->set[(int)((p->steps - 1) % (uint64_t)p->d.depth)];
    cudaError_t e = cudaEventElapsedTime(h2d_ms, S.in_start, S.y_in);
    if (e == cudaSuccess) e = cudaEventElapsedTime(d2h_ms, S.out_start, S.result_free);
    if (e != cudaSuccess) {
        cudaGetLastError();  // not ready: leave no sticky error behind
        *h2d_ms = *d2h_ms = 0.0f;
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

ep_status_t ep_host_pipeline_join(ep_host_pipeline_t* p, void* stream) {
    if (!p) return EP_ERR_INVALID_ARG;
    const cudaStream_t caller = static_cast<cudaStream_t>(stream);
    cudaStream_t sts[] = {p->h2d, p->comp, p->d2h};
    ep_status_t st = EP_OK;
    for (cudaStream_t s : sts) {
        if (st == EP_OK) st = cuda_st(cudaEventRecord(p->caller, s));
        if (st == EP_OK) st = cuda_st(cudaStreamWaitEvent(caller, p->caller, 0));
    }
    return st;
}

ep_status_t ep_host_pipeline_buffer(const ep_host_pipeline_t* p, ep_host_buffer_t which,
                                    void** device_ptr, size_t* bytes) {
    if (!p || !device_ptr || !bytes) return EP_ERR_INVALID_ARG;
    int piece;
    switch (which) {
        case EP_HOST_BUF_TOPK_IDX: piece = P_IDX; break;
        case EP_HOST_BUF_TOPK_W: piece = P_W; break;
        case EP_HOST_BUF_COUNTS: piece = P_COUNTS; break;
        case EP_HOST_BUF_EXPERT_OFFSETS: piece = P_EOFF; break;
        case EP_HOST_BUF_RANK_EXPERT_OFFSETS: piece = P_REOFF; break;
        case EP_HOST_BUF_POS: piece = P_POS; break;
        case EP_HOST_BUF_ROW_SRC: piece = P_ROWSRC; break;
        case EP_HOST_BUF_MASKED_M: piece = P_MASKEDM; break;
        case EP_HOST_BUF_OVERFLOW: piece = P_OVERFLOW; break;
        case EP_HOST_BUF_OUT: piece = P_OUT; break;
        case EP_HOST_BUF_OUT_SCALES: piece = P_SCALES; break;
        default: return EP_ERR_INVALID_ARG;
    }
    *device_ptr = p->ws + piece_offset(p->d, piece);
    *bytes = piece_bytes(p->d, piece);
    return EP_OK;
}

ep_status_t ep_host_pipeline_destroy(ep_host_pipeline_t* p) {
    if (!p) return EP_OK;
    cudaStream_t sts[] = {p->h2d, p->comp, p->d2h};
    ep_status_t st = EP_OK;
    for (cudaStream_t s : sts)
        if (s && st == EP_OK) st = cuda_st(cudaStreamSynchronize(s));
    destroy_handles(p);
    delete p;
    return st;
}

}  // extern "C"
