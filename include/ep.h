/*
 * ep.h -- C ABI of libep_gb300: the MoE expert-parallel hot path
 * (route top-K -> layout -> dispatch -> combine) on one GB300 (sm_103a).
 *
 * Expert parallelism with data-parallel attention is emulated on one GPU: R
 * logical data-parallel ranks hold B_i tokens each, packed rank-major in one
 * buffer (token t of rank r is row rank_offsets[r] + i).  Experts are split
 * into R contiguous sets of E/R; the all-to-all of a multi-GPU system becomes
 * the HBM scatter (dispatch) and gather (combine) below.
 *
 * Sources, by page title and section:
 *   [Anatomy]  "Anatomy of a High-Performance EP Kernel" (Korean and Chinese
 *              renderings): "What we have to do" (shapes (B_i,H), (B_i,E),
 *              (B_i,K); routing table t0..t3), "High throughput: ask first,
 *              then send", "Dispatch" (dense per-expert buffer for the
 *              grouped GEMM; irregular per-expert counts).
 *   [Moreh]    "21K output tokens/s DeepSeek inference on AMD Instinct MI300X
 *              GPUs with Expert Parallelism": "Parallelization method"
 *              (DP8/EP8, 32 of 256 experts per GPU), "Load balancing across
 *              GPUs" (balanced expert renumbering), "Using HIP Graphs"
 *              (static tensor sizes for graph capture).
 *   [SGLang]   "Expert Parallelism" (SGLang docs): "Backends for MoE
 *              computation" (deep_gemm: contiguous layout for prefill, masked
 *              layout for decode, FP8 block-wise quantisation), "Supported
 *              backends" (normal vs low_latency / CUDA-graph-compatible
 *              modes), "Framework overview" (TopK -> dispatch -> runner ->
 *              combine -> final_hidden_states).
 *
 * Conventions for every entry point:
 *   - Pointers are device pointers owned by the caller unless stated; the
 *     library allocates and frees no device memory, and keeps no pointer
 *     after return (except a host pipeline, which keeps its workspace and
 *     expert map, and holds streams and events until destroyed).
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream) and returns without synchronising
 *     (ep_host_pipeline_destroy alone waits, for its own streams); no call
 *     reads device memory on the host, so the four calls and the layout
 *     variants can be captured in a CUDA graph.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns EP_ERR_INVALID_ARG (or EP_ERR_WORKSPACE /
 *     EP_ERR_UNSUPPORTED) and launches nothing.  A failed launch returns
 *     EP_ERR_CUDA.  No kernel traps or asserts.  Besides the stream-order wait
 *     of programmatic launch (below), the only waits are the bounded grid
 *     barriers inside ep_route_layout.
 *   - Device-side data that break a precondition (an expert id outside
 *     [0,E), rank_offsets that are not a non-decreasing 0..N sequence, pos
 *     values that do not come from ep_dispatch_layout) never cause an access
 *     outside the buffers described here: such picks are skipped.
 *   - Kernels are launched with programmatic dependent launch (all but the
 *     cooperative kernel of ep_route_layout, which is a plain cooperative
 *     launch): each one waits for the preceding grids of the stream to
 *     complete (griddepcontrol.wait) before touching memory, then lets the
 *     next kernel launch early.  A
 *     caller kernel that follows ours and is itself launched with the
 *     programmatic-serialisation attribute must wait for its grid dependency
 *     (cudaGridDependencySynchronize) before reading our outputs; kernels
 *     launched without it see plain stream order.  EP_DISABLE_PDL=1 in the
 *     environment launches ours without the attribute.
 *   - bf16 is IEEE binary16-brain (1-8-7); FP8 is OCP E4M3FN.
 *   - Limits: 1 <= E <= 1024, 1 <= K <= min(E, 32), 1 <= R <= 1024,
 *     0 <= N, N*K <= 2^31 - 1; beyond them EP_ERR_UNSUPPORTED.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,  /* null pointer, bad size or alignment */
    EP_ERR_WORKSPACE = 2,    /* workspace missing or smaller than required */
    EP_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
    EP_ERR_UNSUPPORTED = 4   /* sizes beyond the documented limits */
} ep_status_t;

typedef enum {
    EP_LAYOUT_CONTIG = 0,    /* [N*K, H] rows grouped by expert (prefill) */
    EP_LAYOUT_MASKED = 1     /* [E, cap, H] fixed capacity per expert (decode) */
} ep_layout_t;

typedef enum {
    EP_DTYPE_BF16 = 0,          /* rows copied as bf16 */
    EP_DTYPE_FP8_E4M3_B128 = 1  /* E4M3 codes + one float scale per 128 columns */
} ep_dtype_t;

/*
 * ep_route_topk -- [Anatomy] "What we have to do": each token's router
 * logits (length E) select the K experts with the largest logits, giving the
 * (B_i, K) assignment (the table's t0 row routes to [3, 13]).
 *   logits     float32 [N, E] row-major, finite values (NaN is not ordered).
 *   expert_map int32 [E] or NULL; when given, output ids are expert_map[id]
 *              ([Moreh] "Load balancing across GPUs": the gate must emit the
 *              renumbered ids).  Entries outside [0,E) become "no pick".
 *   topk_idx   int32 [N, K] out: picks in descending logit order; equal
 *              logits go to the lower expert id; -0.0 equals +0.0.
 *   topk_w     float32 [N, K] out: softmax over the K picked logits,
 *              w_k = exp(l_k - l_0) / sum_j exp(l_j - l_0), in float (the
 *              pages print no gate formula; softmax renormalised over the
 *              top K is the reading used).
 */
ep_status_t ep_route_topk(const float* logits, int32_t N, int32_t E, int32_t K,
                          const int32_t* expert_map, int32_t* topk_idx, float* topk_w,
                          void* stream);

/*
 * ep_expert_balance_map -- [Moreh] "Load balancing across GPUs": group the E
 * experts into R sets of E/R with balanced activation frequency and renumber
 * each set contiguously.  The page names the problem (a balanced number
 * partitioning variant) but no algorithm; this computes the greedy one:
 * frequency[e] = sum_r counts[r][e]; experts in descending frequency (ties:
 * lower id) each join the set with the least load among sets with room
 * (ties: lower set id); new id = set * (E/R) + arrival order in the set.
 *   counts     int32 [R, E] per-(rank, expert) counts (ep_dispatch_layout's
 *              output for a calibration batch), non-negative.
 *   expert_map int32 [E] out: old id -> new id, a permutation of [0, E).
 * Requires E % R == 0.  One small single-block kernel.
 */
ep_status_t ep_expert_balance_map(const int32_t* counts, int32_t R, int32_t E,
                                  int32_t* expert_map, void* stream);

/*
 * Bytes of device workspace ep_dispatch_layout needs for these sizes (a
 * multiple of 256; 0 never occurs).  Pure host function.
 */
size_t ep_dispatch_layout_workspace_size(int32_t N, int32_t E, int32_t K, int32_t R);

/*
 * ep_dispatch_layout -- [Anatomy] "High throughput: ask first, then send":
 * every (rank, expert) count is known before any row moves, and each expert's
 * rows form one dense block for the grouped GEMM ("Dispatch").  A stable
 * counting sort of the N*K picks by expert id:
 *   topk_idx            int32 [N, K]; ids outside [0,E) are "no pick".
 *   rank_offsets        int32 [R+1] device: 0 = o_0 <= o_1 <= ... <= o_R = N;
 *                       tokens [o_r, o_{r+1}) belong to rank r.
 *   cap                 0, or the masked capacity per expert (> 0).
 *   counts              int32 [R, E] out: picks of expert e by rank r.
 *   expert_offsets      int32 [E+1] out: exclusive prefix of expert totals;
 *                       expert_offsets[E] = number of valid picks.
 *   rank_expert_offsets int32 [R, E] out: expert_offsets[e] +
 *                       sum_{r'<r} counts[r'][e] (where rank r's rows for
 *                       expert e start).
 *   pos                 int32 [N, K] out: row of pick (t,k) in the expert-
 *                       major buffer; within an expert, picks keep (t, k)
 *                       order (hence source-rank order); -1 for no pick.
 *   row_src             int32 [N*K] out: token of row p; -1 past the valid
 *                       rows.
 *   masked_m            int32 [E] or NULL out (needs cap > 0): min(total, cap)
 *                       ([SGLang] masked layout's per-expert valid count).
 *   overflow_count      int32 [1] or NULL out (needs cap > 0): picks beyond
 *                       cap, which the masked layout drops.
 *   workspace           device scratch of ws_bytes >= the size above; its
 *                       contents need no initialisation and are clobbered.
 * R need not divide E.  The layout uses a rank only as a range of tokens
 * (its counts row and where its rows start in each expert segment); which
 * experts a rank hosts (E/R contiguous ones, [Moreh] "Parallelization
 * method") matters only to ep_expert_balance_map, which requires E % R == 0.
 * A micro-batch of a subset of the ranks (one rank of eight, say, with all
 * 256 experts) is therefore a valid layout problem.
 * Problems of at most 16384 picks (N*K) run as one launch of one block per
 * expert (no workspace is touched); larger ones as three kernels.  In the
 * environment (read at every call) EP_LAYOUT_SMALL=0 switches the first path
 * off, so that problems of at most 16384 picks and 64 ranks whose chunk rows
 * fit in shared memory run as one thread-block cluster, and
 * EP_LAYOUT_CLUSTER=0 selects the three kernels for every size.  All give the
 * same results, which are deterministic (no order depends on atomics).
 */
ep_status_t ep_dispatch_layout(const int32_t* topk_idx, const int32_t* rank_offsets,
                               int32_t R, int32_t N, int32_t E, int32_t K, int32_t cap,
                               int32_t* counts, int32_t* expert_offsets,
                               int32_t* rank_expert_offsets, int32_t* pos, int32_t* row_src,
                               int32_t* masked_m, int32_t* overflow_count,
                               void* workspace, size_t ws_bytes, void* stream);

/* Bytes of device workspace ep_route_layout needs (a multiple of 256). */
size_t ep_route_layout_workspace_size(int32_t N, int32_t E, int32_t K, int32_t R);

/*
 * ep_route_layout -- ep_route_topk followed by ep_dispatch_layout in one
 * cooperative persistent kernel (no launches or ramp-ups in between); same
 * arguments and bit-identical outputs as the two calls.  [Anatomy] "What we
 * have to do" (route locally) and "High throughput: ask first, then send".
 *   status    int32 [1] device, or NULL: 0 when the call completed, 1 if a
 *             block's bounded wait at an internal grid barrier ran out
 *             (results then incomplete; the co-resident launch rules it out).
 *             Written on every call (need not be cleared): the kernel stores
 *             0 before its first barrier and any timeout stores 1 after
 *             that, so a 1 is never overwritten; the two-kernel fallback
 *             clears it with a memset.
 *   workspace ep_route_layout_workspace_size bytes, no initialisation needed.
 * Sizes without a fused instance (E not a multiple of 128 above 256 experts)
 * or a device that cannot hold one block run the two kernels instead, with
 * the same results.  Launches one memset before the kernel (the chunk
 * histograms that the routing phase counts into, and the barrier counters);
 * the kernel writes the status word.
 */
ep_status_t ep_route_layout(const float* logits, const int32_t* rank_offsets, int32_t R,
                            int32_t N, int32_t E, int32_t K, const int32_t* expert_map,
                            int32_t cap, int32_t* topk_idx, float* topk_w, int32_t* counts,
                            int32_t* expert_offsets, int32_t* rank_expert_offsets, int32_t* pos,
                            int32_t* row_src, int32_t* masked_m, int32_t* overflow_count,
                            int32_t* status, void* workspace, size_t ws_bytes, void* stream);

/* Bytes of the fixed scratch array that ep_dispatch_layout_static keeps
 * inside the library on every GPU that loads it (4 MiB). */
#define EP_LAYOUT_STATIC_SCRATCH_BYTES (4u * 1024u * 1024u)

/*
 * ep_dispatch_layout_static -- no counterpart in the source pages; an
 * addition of this library for callers that cannot allocate device memory
 * (an embedder whose device memory is reserved up front by another
 * allocator, a plain C host without a device allocator, code running where
 * cudaMalloc is not permitted).  Same inputs, outputs and results as
 * ep_dispatch_layout, but no workspace argument: the scratch is a fixed
 * array of EP_LAYOUT_STATIC_SCRATCH_BYTES inside the library, held by every
 * GPU that loads the library until the process exits.
 *   - Sizes whose scratch (ep_dispatch_layout_workspace_size) exceeds
 *     EP_LAYOUT_STATIC_SCRATCH_BYTES return EP_ERR_UNSUPPORTED and launch
 *     nothing; other argument errors as for ep_dispatch_layout.
 *   - The first call on a device looks up the array's device address (with
 *     that device current) and caches it; make that first call before any
 *     stream capture.  A failed lookup returns EP_ERR_CUDA.  The cached
 *     address belongs to the device's current context: after
 *     cudaDeviceReset (or anything else that destroys and recreates the
 *     primary context) the library reloads and the array may move, so do
 *     not call this entry point again in a process that has reset a device
 *     it was used on.
 *   - Allocates nothing (no cudaMalloc/cudaFree, no allocating library call).
 *   - All calls share the array and it keeps the last call's contents; the
 *     kernels write every entry they read, so nothing needs clearing.  Calls
 *     that overlap on the GPU (different streams or host threads) race on
 *     the array: order them on one stream.
 */
ep_status_t ep_dispatch_layout_static(const int32_t* topk_idx, const int32_t* rank_offsets,
                                      int32_t R, int32_t N, int32_t E, int32_t K, int32_t cap,
                                      int32_t* counts, int32_t* expert_offsets,
                                      int32_t* rank_expert_offsets, int32_t* pos,
                                      int32_t* row_src, int32_t* masked_m,
                                      int32_t* overflow_count, void* stream);

/*
 * ep_dispatch -- [Anatomy] "Dispatch" and [SGLang] deep_gemm row: scatter each
 * token's activation row to the rows of its K picks.  Each source row is read
 * once and written K times.
 *   x              bf16 [N, H], 16-byte aligned; H % 8 == 0.
 *   topk_idx, pos, expert_offsets: as produced by ep_dispatch_layout.
 *   layout CONTIG: out rows = N*K, row of pick (t,k) = pos[t,k].  When
 *                  some picks are "no pick", the rows from expert_offsets[E]
 *                  on receive nothing and are not written.
 *   layout MASKED: out is [E, cap, H]; slot = pos[t,k] - expert_offsets[e];
 *                  delivered to (e, slot) when slot < cap, else dropped.
 *                  Rows at or past masked_m[e] are not written.
 *   dtype BF16:    out bf16 rows, bit copies of x; out_scales unused (NULL ok).
 *   dtype FP8_E4M3_B128 ([SGLang] "FP8 block-wise quantisation"; block size
 *                  1x128 and E4M3 are the reading used): H % 128 == 0; per
 *                  token and 128-column block b, amax = max|x|, scale =
 *                  amax / 448 (IEEE float division; 1 when amax == 0), code =
 *                  E4M3(x / scale) rounded to nearest even with saturation to
 *                  +-448; out uint8 codes [rows, H], out_scales float32
 *                  [rows, H/128].  The codes are computed once per token and
 *                  written to all K rows.
 *   out            16-byte aligned.
 * From 4096 tokens on (rows of at most 32 KB), each destination row is written
 * by one bulk shared-to-global copy; EP_DISPATCH_BULK=0 in the environment
 * (read at every call) keeps the per-thread stores at every size.  The
 * results are the same either way.
 */
ep_status_t ep_dispatch(const void* x, int32_t N, int32_t H, int32_t E, int32_t K,
                        const int32_t* topk_idx, const int32_t* pos,
                        const int32_t* expert_offsets, ep_layout_t layout, int32_t cap,
                        ep_dtype_t dtype, void* out, float* out_scales, void* stream);

/*
 * ep_combine -- [Anatomy] "bring the results home" after the expert GEMM, and
 * [SGLang] "Framework overview" (Dispatcher.combine -> final_hidden_states):
 *   out[t] = bf16_rn( sum_{k=0..K-1} topk_w[t,k] * y[row(t,k)] )
 * accumulated in float, one fused multiply-add per pick in the order k = 0..
 * K-1; picks that were not delivered (no pick, masked overflow) add nothing.
 *   y      bf16 expert outputs, 16-byte aligned: [N*K, H] (CONTIG) or
 *          [E, cap, H] (MASKED); row(t,k) as in ep_dispatch.
 *   topk_w float32 [N, K].
 *   out    bf16 [N, H], 16-byte aligned; must not overlap y.
 */
ep_status_t ep_combine(const void* y, int32_t N, int32_t H, int32_t E, int32_t K,
                       const int32_t* topk_idx, const float* topk_w, const int32_t* pos,
                       const int32_t* expert_offsets, ep_layout_t layout, int32_t cap,
                       void* out, void* stream);

/*
 * ep_route_dispatch -- ep_route_topk, ep_dispatch_layout and ep_dispatch in
 * one call, with the same arguments and bit-identical outputs; problems of at
 * most 2048 tokens and 16384 picks (the decode-sized ones) take two launches.
 * [Anatomy] "What we have to do", "High throughput: ask first, then send"
 * and "Dispatch"; [SGLang] "Supported backends" (the low-latency mode).  The
 * routing kernel also writes, for each block of 8 tokens, its expert
 * histogram and the histogram's prefix over experts (into the workspace);
 * from those rows alone one more kernel places every pick, writes every
 * layout output and stores the rows, with no layout launch in between.
 * Larger problems run the route kernel, the layout kernels and the dispatch
 * kernel, with the same results.
 *   logits, expert_map, topk_idx, topk_w   as for ep_route_topk.
 *   rank_offsets, R, cap, counts ... overflow_count   as for
 *              ep_dispatch_layout (overflow_count is zeroed by the call).
 *   x, H, layout, dtype, out, out_scales   as for ep_dispatch (cap > 0 for
 *              MASKED).
 *   workspace  ep_route_dispatch_workspace_size bytes, 16-byte aligned, no
 *              initialisation needed (EP_ERR_WORKSPACE otherwise).
 */
size_t ep_route_dispatch_workspace_size(int32_t N, int32_t E, int32_t K, int32_t R);

ep_status_t ep_route_dispatch(const float* logits, const int32_t* rank_offsets, const void* x,
                              int32_t R, int32_t N, int32_t H, int32_t E, int32_t K,
                              const int32_t* expert_map, ep_layout_t layout, int32_t cap,
                              ep_dtype_t dtype, int32_t* topk_idx, float* topk_w,
                              int32_t* counts, int32_t* expert_offsets,
                              int32_t* rank_expert_offsets, int32_t* pos, int32_t* row_src,
                              int32_t* masked_m, int32_t* overflow_count, void* out,
                              float* out_scales, void* workspace, size_t ws_bytes,
                              void* stream);

/*
 * ep_host_pipeline_* -- no counterpart in the source pages: the path for
 * callers whose inputs and results live in host memory.  Each step copies the
 * step's logits, rank offsets, tokens x and expert outputs y in, runs
 * ep_route_topk, ep_dispatch_layout, ep_dispatch and ep_combine, and copies
 * the combined [N, H] bf16 result out.  Copies in, kernels and the copy out
 * run on three streams of the pipeline.  `depth` device buffer sets rotate,
 * so a step's copies in overlap the previous step's kernels and copy out.
 * A set is reused only after the kernels and the copy out of the step that
 * last used it are done.
 *   N, E, K, H, R, cap, dtype  as for the four calls (cap > 0: masked layout,
 *              y is [E, cap, H]; cap == 0: contiguous, y is [N*K, H]);
 *              N >= 1; depth 1..4 (1: each step waits for the previous).
 *   expert_map device int32 [E] or NULL, the same for every step; it must
 *              stay valid while the pipeline exists.
 *   workspace  device memory of at least ep_host_pipeline_workspace_size
 *              bytes, 256-byte aligned, owned by the caller and kept alive
 *              (and untouched) until ep_host_pipeline_destroy returns.  Every
 *              device buffer of the pipeline lives in it.
 * The object itself holds three streams and 7*depth + 1 events on the device
 * that was current at creation; call its functions with that device
 * current.
 */
typedef struct ep_host_pipeline ep_host_pipeline_t;

/* Bytes of workspace a pipeline needs; 0 for invalid or unsupported sizes. */
size_t ep_host_pipeline_workspace_size(int32_t N, int32_t E, int32_t K, int32_t H, int32_t R,
                                       int32_t cap, ep_dtype_t dtype, int32_t depth);

/* Creates a pipeline in *out.  EP_ERR_INVALID_ARG / EP_ERR_UNSUPPORTED for
 * sizes outside the four calls' limits (or depth outside 1..4),
 * EP_ERR_WORKSPACE for a missing, small or misaligned workspace, EP_ERR_CUDA
 * if a stream or event cannot be created (*out is then NULL). */
ep_status_t ep_host_pipeline_create(int32_t N, int32_t E, int32_t K, int32_t H, int32_t R,
                                    int32_t cap, ep_dtype_t dtype, int32_t depth,
                                    const int32_t* expert_map, void* workspace, size_t ws_bytes,
                                    ep_host_pipeline_t** out);

/* Enqueues one step.  Host buffers (page-locked for the copies to overlap;
 * pageable memory works but its copies do not overlap): logits_h float32
 * [N, E], rank_offsets_h int32 [R+1], x_h bf16 [N, H], y_h bf16 [N*K, H] or
 * [E, cap, H], out_h bf16 [N, H].  The step starts after the work enqueued
 * on `stream` before the call.  The inputs must stay untouched and out_h
 * unread until the step is done (ep_host_pipeline_join, then a sync of
 * `stream`).  An argument or launch failure returns its status; the
 * pipeline's streams may then hold part of the step. */
ep_status_t ep_host_pipeline_step(ep_host_pipeline_t* pipeline, const float* logits_h,
                                  const int32_t* rank_offsets_h, const void* x_h,
                                  const void* y_h, void* out_h, void* stream);

/* Makes `stream` wait for every step enqueued so far. */
ep_status_t ep_host_pipeline_join(ep_host_pipeline_t* pipeline, void* stream);

/* Device-timed durations, in milliseconds, of the last enqueued step's
 * copies in (logits, rank offsets, x and y, from the start of the first to
 * the end of the last) and of its copy out, once that step is done (after a
 * join and a sync).  EP_ERR_INVALID_ARG before the first step or for NULL
 * pointers; EP_ERR_CUDA (times 0) while the step is still running. */
ep_status_t ep_host_pipeline_copy_ms(const ep_host_pipeline_t* pipeline, float* h2d_ms,
                                     float* d2h_ms);

/* Device buffers of the last step's intermediate outputs, inside the
 * workspace (valid after a join and a sync): the routed picks and weights,
 * the layout, and the dispatched rows (and FP8 scales). */
typedef enum {
    EP_HOST_BUF_TOPK_IDX = 0,
    EP_HOST_BUF_TOPK_W = 1,
    EP_HOST_BUF_COUNTS = 2,
    EP_HOST_BUF_EXPERT_OFFSETS = 3,
    EP_HOST_BUF_RANK_EXPERT_OFFSETS = 4,
    EP_HOST_BUF_POS = 5,
    EP_HOST_BUF_ROW_SRC = 6,
    EP_HOST_BUF_MASKED_M = 7,      /* 0 bytes when cap == 0 */
    EP_HOST_BUF_OVERFLOW = 8,      /* 0 bytes when cap == 0 */
    EP_HOST_BUF_OUT = 9,
    EP_HOST_BUF_OUT_SCALES = 10    /* 0 bytes for bf16 */
} ep_host_buffer_t;

ep_status_t ep_host_pipeline_buffer(const ep_host_pipeline_t* pipeline, ep_host_buffer_t which,
                                    void** device_ptr, size_t* bytes);

/* Waits for the pipeline's streams, then releases its streams and events and
 * the object (NULL is a no-op).  The workspace is the caller's to free. */
ep_status_t ep_host_pipeline_destroy(ep_host_pipeline_t* pipeline);

/*
 * ep_host_alloc / ep_host_free -- no counterpart in the source pages: page-
 * locked host memory for the host pipeline's inputs and results.  The
 * pipeline's copies stream gigabytes per step over the host link; on a
 * GB300 machine (64 KB base pages) the kernel's periodic reactivation of the
 * pages of ordinary pinned buffers (cudaHostAlloc) was measured to cut a
 * copy that overlapped it from 211 to about 50 GB/s, while copies from
 * buffers backed by huge pages never slowed.  ep_host_alloc therefore maps
 * anonymous memory aligned to the huge-page size, asks for transparent huge
 * pages (madvise), touches it and page-locks it with cudaHostRegister.
 * Where the kernel offers no transparent huge pages the memory is still
 * page-locked, on base pages.
 *   bytes  > 0; rounded up to whole huge pages (a 1-byte buffer holds one).
 *   *out   receives the host pointer (aligned to the huge-page size), usable
 *          by the host and by copies on every device; NULL on failure.
 * Returns EP_ERR_INVALID_ARG for bytes == 0 or out == NULL, EP_ERR_CUDA if
 * the mapping or the registration fails.  Allocates host memory only.
 * ep_host_free unregisters and unmaps a pointer from ep_host_alloc (NULL is
 * a no-op; any other pointer returns EP_ERR_INVALID_ARG).  Thread-safe.
 */
ep_status_t ep_host_alloc(size_t bytes, void** out);
ep_status_t ep_host_free(void* ptr);

/*
 * ep_selftest_wait_timeout -- no counterpart in the source pages: a check of
 * the bounded wait that guards the grid barriers of ep_route_layout.  It
 * launches a 2-block kernel whose barrier waits for a third block that never
 * comes; the wait gives up after 2^20 polls (well under a second), the kernel
 * sets *status to 1 and every block returns, leaving the context usable.
 *   status     device int32, set to 0 before the kernel and 1 by it.
 *   workspace  device memory of at least 4 bytes, 4-byte aligned (the
 *              barrier counter; zeroed here).
 * Returns EP_ERR_INVALID_ARG (nothing launched) for a NULL or misaligned
 * pointer or ws_bytes < 4, EP_ERR_CUDA on a launch failure.
 */
ep_status_t ep_selftest_wait_timeout(int32_t* status, void* workspace, size_t ws_bytes,
                                     void* stream);

/* Human-readable name of a status code (static storage). */
const char* ep_status_string(ep_status_t status);

/* Text of the last CUDA error seen by this library on the calling thread
 * ("" if none); valid until the next call on that thread. */
const char* ep_last_cuda_error(void);

/* Number of kernels this library has launched in this process (all threads,
 * all devices).  Lets a caller count launches inside a timed region. */
uint64_t ep_kernel_launch_count(void);

/* ABI version of this header: 1. */
int32_t ep_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
