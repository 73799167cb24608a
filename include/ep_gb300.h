/*
 * ep_gb300.h -- C ABI of the MoE expert-parallel dispatch / combine library
 * (libep_gb300.so, CUDA, sm_103a).
 *
 * The W expert-parallel ranks are W logical partitions of one receive buffer in
 * one GPU's memory: the "send" of a row to rank r is a store into rank r's
 * region.  There is no collective and no second device.
 *
 * Conventions shared by every entry point
 *  - Every pointer argument is a DEVICE pointer owned by the caller.  Tensors
 *    are dense and row-major.  The library allocates nothing, keeps no state
 *    between calls (apart from a per-device cache of the SM count) and never
 *    synchronises: each call enqueues its kernels on `stream` and returns.
 *  - Return value: EP_OK, or an EP_ERR_* code found on the host before anything
 *    was enqueued (bad argument, misaligned pointer, unsupported shape), or
 *    EP_ERR_CUDA when a launch was refused.
 *  - Data-dependent problems are reported on the device: the kernels OR
 *    EP_STATUS_* bits into the caller's int32 `*status` (may be NULL).  The
 *    caller zeroes it and reads it whenever it likes; nothing traps.
 *  - Payload pointers (x, recv_x, y, out) must be 16-byte aligned; index,
 *    weight, count and slot pointers 4-byte aligned.
 *  - Kernels are launched with programmatic dependent launch: each one waits
 *    for the previous kernel on the stream to finish before it touches memory,
 *    so consecutive calls overlap only their launch latency.  The one
 *    exception is inside a single call: in ep_dispatch_with_layout,
 *    ep_dispatch_regions_with_layout and ep_dispatch_experts_with_layout the
 *    dispatch kernel loads its first rows of x while that call's own layout
 *    kernels run (x must be complete in stream order before the call, as for
 *    any input).
 *
 * Notation: T tokens, H hidden size, E experts, k experts per token, W ranks,
 * Er = E / W experts per rank, rank(e) = e / Er, D(t) = the distinct ranks of
 * token t's valid expert ids, R = sum over t of |D(t)| receive rows.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st* ep_stream_t;

/* Host-side return codes. */
enum {
  EP_OK = 0,
  EP_ERR_INVALID_ARG = 1,  /* a size or pointer argument is out of range / NULL */
  EP_ERR_MISALIGNED = 2,   /* a pointer violates the alignment rule above */
  EP_ERR_UNSUPPORTED = 3,  /* shape outside the supported set (see each call) */
  EP_ERR_CUDA = 4,         /* the CUDA runtime refused a launch */
  EP_ERR_WORKSPACE = 5     /* workspace smaller than ep_layout_workspace_bytes() */
};

/* Device-side status bits, OR-ed into *status. */
enum {
  EP_STATUS_BAD_EXPERT = 1, /* an expert id outside [0, E): the entry was ignored */
  EP_STATUS_CAPACITY = 2,   /* a receive row >= capacity_rows: it was not read / written */
  EP_STATUS_TIMEOUT = 4     /* a bounded on-chip wait gave up (about 1 s); outputs incomplete */
};

/* Dispatch payload formats. */
enum {
  EP_QUANT_BF16 = 0,         /* rows copied as bf16 */
  EP_QUANT_FP8_E4M3_B128 = 1 /* rows quantised to FP8 e4m3 with one fp32 scale per 1x128 block */
};

/*
 * Bytes of device workspace that ep_dispatch_layout needs for T tokens, W
 * ranks and E experts.  The contents need no initialisation.  Returns 0 for
 * invalid arguments.  Host only.  A convention of this library (the caller
 * owns all device memory); the pages define no such call.
 */
EP_API size_t ep_layout_workspace_bytes(int64_t T, int W, int E);

/*
 * Worst-case number of receive rows, T * min(k, W): a receive buffer of this
 * many rows can never overflow.  (Sizing the receive side for the worst case
 * follows the size hint of "Feature/sm free normal kernel", deepseek-ai/DeepEP
 * pull 347, section 3.3.1.)  Returns -1 for invalid arguments.
 */
EP_API int64_t ep_max_recv_rows(int64_t T, int k, int W);

/*
 * Routing layout.  Follows "perf(ep): optimize IntraNode dispatch kernel for
 * MI350X" (ROCm/mori pull 586), Technical Details 1: the destination rank of
 * expert e is e / Er, a token is sent once per destination rank, and the
 * destination of every kept (token, rank) pair is computed once and cached for
 * the copy and for combine.  The pages reserve receive slots with atomics; here
 * they come from a stable prefix scan, so the layout is deterministic.
 *
 *  topk_idx              int32 [T, k]   expert ids; ids outside [0, E) are
 *                                       ignored and set EP_STATUS_BAD_EXPERT
 *  num_tokens_per_expert int32 [E]      out: #(t, j) with topk_idx[t][j] == e
 *                                       (before deduplication)
 *  num_tokens_per_rank   int32 [W]      out: #t with r in D(t)
 *  rank_offset           int32 [W + 1]  out: exclusive prefix sum of
 *                                       num_tokens_per_rank; rank_offset[W] = R
 *  slot                  int32 [T, W]   out: receive row of (t, r):
 *                                       rank_offset[r] + #{t' < t : r in D(t')}
 *                                       if r in D(t), else -1
 *  workspace             ep_layout_workspace_bytes(T, W, E) bytes, 16-byte aligned;
 *                        it serves one call at a time (calls that overlap on
 *                        the GPU need workspaces of their own)
 * Limits: 0 <= T, T * min(k, W) < 2^31; 1 <= k; 1 <= W <= 32; E % W == 0;
 * 1 <= E <= 8192.
 */
EP_API int ep_dispatch_layout(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                       int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                       int32_t* rank_offset, int32_t* slot, void* workspace,
                       size_t workspace_bytes, int32_t* status, ep_stream_t stream);

/*
 * Dispatch: scatter each token's row to the receive row of every rank in D(t),
 * reading x[t] once, and carry the routing metadata with it.  Follows "perf(ep):
 * optimize IntraNode dispatch kernel for MI350X", Technical Details 1, 3 and 4
 * (cached destinations, warp-wide row copy, metadata copied by the whole warp)
 * and "Optimizing Distributed Inference Kernels for AMD DEVELOPER CHALLENGE
 * 2025", section 3.1 (16-byte vector copies of a token row).
 *
 *  x              bf16 [T, H]
 *  topk_idx       int32 [T, k], topk_w fp32 [T, k]
 *  slot           int32 [T, W] from ep_dispatch_layout
 *  capacity_rows  rows of every receive buffer; rows >= capacity_rows are
 *                 skipped and set EP_STATUS_CAPACITY
 *  quant          EP_QUANT_BF16: recv_x is bf16 [capacity_rows, H], a bit copy.
 *                 EP_QUANT_FP8_E4M3_B128: recv_x is uint8 [capacity_rows, H];
 *                 per row and 128-column block b: scale = amax / 448 (fp32,
 *                 IEEE division), recv_scale[s][b] = scale, code =
 *                 e4m3 round-to-nearest-even with saturation of x / scale (fp32
 *                 IEEE division); scale 0 gives all-zero codes.  The FP8 e4m3
 *                 dispatch of the same page (Test Plan) is the model; the block
 *                 scale rule is this library's.
 *  recv_scale     fp32 [capacity_rows, H / 128] for FP8, else ignored (may be NULL)
 *  recv_topk_idx  int32 [capacity_rows, k]  copy of topk_idx[t]  (NULL: skipped)
 *  recv_topk_w    fp32  [capacity_rows, k]  copy of topk_w[t]    (NULL: skipped)
 *  recv_src       int32 [capacity_rows]     source token t       (NULL: skipped)
 * Rows of the receive buffers that no (t, r) maps to are left untouched.
 * Limits: H % 8 == 0 (bf16) or H % 128 == 0 (FP8); 1 <= W <= 32; 1 <= k.
 */
EP_API int ep_dispatch(const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T, int H,
                int k, int W, const int32_t* slot, int64_t capacity_rows, int quant, void* recv_x,
                float* recv_scale, int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                int32_t* status, ep_stream_t stream);

/*
 * Layout and dispatch in one call: ep_dispatch_layout followed by ep_dispatch
 * on the same stream, with the same arguments, limits, results and errors as
 * those two calls.  The layout's counts and slots are written as by
 * ep_dispatch_layout.  What one call allows that two do not: the dispatch
 * kernel is known to follow the layout kernels directly, so it becomes resident
 * while they run and starts loading its first rows of x before the slots
 * exist (x must be complete in stream order before this call, as it must
 * before ep_dispatch).  For T > 1024 (FP8 rows, or bf16 rows of at least
 * 1 KB) the dispatch also finishes the layout: the count kernel numbers each
 * token inside its chunk of 128 and the dispatch adds the chunk's base row, so
 * the scan kernel is not launched; its bf16 warps then take tokens from a
 * counter that the count kernel zeroes in the workspace (the workspace must
 * not be shared by calls that overlap on the GPU, as for ep_dispatch_layout).
 * Which warp sends which token varies from call to call; the results do not.
 * bf16 batches of up to 512 tokens (k <= 16)
 * take the one-launch kernel of ep_dispatch_fused, the fastest there
 * (ep_dispatch_with_layout_launches).  The layout
 * is the one of "perf(ep): optimize IntraNode dispatch kernel for MI350X",
 * Technical Details 1; the dispatch follows the same page's Technical Details
 * 1, 3 and 4.
 */
EP_API int ep_dispatch_with_layout(const void* x, const int32_t* topk_idx, const float* topk_w,
                                   int64_t T, int H, int k, int E, int W,
                                   int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                   int32_t* rank_offset, int32_t* slot, void* workspace,
                                   size_t workspace_bytes, int64_t capacity_rows, int quant,
                                   void* recv_x, float* recv_scale, int32_t* recv_topk_idx,
                                   float* recv_topk_w, int32_t* recv_src, int32_t* status,
                                   ep_stream_t stream);

/*
 * Number of kernels one ep_dispatch_with_layout call with these sizes
 * launches (for callers that count launches, e.g. to size a CUDA graph):
 * 1 for bf16 batches of 1 to 512 tokens with k <= 16 (the one-launch dispatch
 * of ep_dispatch_fused); 2 when the dispatch finishes the layout itself
 * (T > 1024, FP8 rows or bf16 rows of at least 1 KB, and a chunk table
 * (ceil(T / 128) * W ints) of at most 16 KB); else the layout's kernels (1 for
 * T <= 1024, else 2) plus 1 for the dispatch when T > 0.  Returns -1 for
 * invalid arguments.  Host only.  A convention of this library; the pages
 * define no such call.
 */
EP_API int ep_dispatch_with_layout_launches(int64_t T, int H, int k, int W, int quant);

/*
 * Local expert ids, in place, after ep_dispatch on the same stream: in receive
 * row s of rank r (rank_offset[r] <= s < rank_offset[r+1], s < capacity_rows)
 * each of the k ids e in recv_topk_idx[s] becomes e - r * (E / W) when e is a
 * valid expert hosted by rank r, and -1 otherwise; rows from rank_offset[W] on
 * are untouched.  Gives each rank's expert side the local experts a row needs,
 * from the per-rank destination rule of "perf(ep): optimize IntraNode dispatch
 * kernel for MI350X", Technical Details 1 (expert e lives on rank e / (E/W)).
 *  recv_topk_idx  int32 [capacity_rows, k], rank_offset int32 [W + 1]
 * Limits: 1 <= k; 1 <= W <= 32; E % W == 0.
 */
EP_API int ep_localize_expert_ids(int32_t* recv_topk_idx, const int32_t* rank_offset,
                                  int64_t capacity_rows, int k, int E, int W, ep_stream_t stream);

/*
 * ep_dispatch_layout followed by a bf16 ep_dispatch, in one launch, for small
 * batches (decode): T <= EP_FUSED_MAX_TOKENS.  Every output is the one the two
 * calls would produce (layout outputs included: slot is needed by combine), so
 * it is a drop-in replacement for them where latency matters.  Every CTA
 * recomputes the batch's layout from topk_idx and then sends the tokens it
 * owns at once, which saves the second launch and the slot round trip.
 * Follows the single-pass routing of the low-latency kernel discussed on
 * "perf(ep): optimize IntraNode dispatch kernel for MI350X" (the IntraNodeLL
 * comparison), with the deterministic slot numbering of ep_dispatch_layout.
 *
 * Arguments: those of ep_dispatch_layout and ep_dispatch (bf16 payload only),
 * no workspace.  Limits: T <= EP_FUSED_MAX_TOKENS, 1 <= k <= 16, 1 <= W <= 32,
 * E % W == 0, E <= 8192, H % 8 == 0; EP_ERR_UNSUPPORTED otherwise.
 */
#define EP_FUSED_MAX_TOKENS 1024
EP_API int ep_dispatch_fused(const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T,
                             int H, int k, int E, int W, int32_t* num_tokens_per_expert,
                             int32_t* num_tokens_per_rank, int32_t* rank_offset, int32_t* slot,
                             int64_t capacity_rows, void* recv_x, int32_t* recv_topk_idx,
                             float* recv_topk_w, int32_t* recv_src, int32_t* status,
                             ep_stream_t stream);

/*
 * Combine: out[t] = bf16_rne( ((+0 + y[s_0]) + y[s_1]) + ... ) with the fp32
 * sum taken over the ranks r in D(t) in ascending order, s_r = slot[t][r]; a
 * token with no rows gives +0.  Follows "perf(ep): optimize IntraNode dispatch
 * kernel for MI350X", "Remaining gap" (combine reads the pre-routed rows of each
 * token and accumulates them) and "Optimizing Distributed Inference Kernels for
 * AMD DEVELOPER CHALLENGE 2025", section 3.1 (combine brings the expert outputs
 * back to token order).  The sum is unweighted: the expert side applies the
 * gate weights.
 *
 *  y              bf16 [capacity_rows, H]  expert outputs, one per receive row
 *  slot           int32 [T, W] from ep_dispatch_layout
 *  out            bf16 [T, H]
 * Rows >= capacity_rows are skipped and set EP_STATUS_CAPACITY.
 * Limits: H % 8 == 0; 1 <= W <= 32.
 */
EP_API int ep_combine(const void* y, const int32_t* slot, int64_t T, int H, int W, int64_t capacity_rows,
               void* out, int32_t* status, ep_stream_t stream);

/*
 * Receive storage of one rank when the W rank regions live in separate
 * allocations (ep_dispatch_regions, ep_combine_regions).  All pointers are
 * device pointers owned by the caller; rows are dense and row-major.
 */
typedef struct ep_rank_region {
  void* recv_x;           /* bf16 [rows, H] (EP_QUANT_BF16) or uint8 codes [rows, H] (FP8);
                             16-byte aligned */
  float* recv_scale;      /* fp32 [rows, H / 128] for FP8, else ignored (may be NULL) */
  int32_t* recv_topk_idx; /* int32 [rows, k], or NULL: not written */
  float* recv_topk_w;     /* fp32 [rows, k], or NULL: not written */
  int32_t* recv_src;      /* int32 [rows], or NULL: not written */
  int64_t rows;           /* capacity of this region, 0 <= rows < 2^31 */
} ep_rank_region_t;

/*
 * Dispatch into per-rank regions: ep_dispatch with rank r's receive rows in an
 * allocation of their own, named by a table of base pointers.  Token t's row
 * for rank r in D(t) goes to row slot[t][r] - rank_offset[r] of region r (its
 * position among rank r's tokens, ascending token order), with the same bits
 * (bf16 copy, or FP8 codes and scales) and metadata that ep_dispatch writes
 * at global row slot[t][r].  Rows at or beyond regions[r].rows are skipped and
 * set EP_STATUS_CAPACITY.  This is the push model of "perf(ep): optimize
 * IntraNode dispatch kernel for MI350X", Technical Details 1 (each rank's rows
 * are stored straight into that rank's receive buffer), on one GPU: a region
 * is any allocation of this device.  (A region on a peer GPU would need the
 * kernels' row stores to be plain peer stores; this library keeps every copy
 * on this GPU's memory.)
 *
 *  x, topk_idx, topk_w  as for ep_dispatch
 *  slot, rank_offset    int32 [T, W] and [W + 1] from ep_dispatch_layout (or any
 *                       of the layout calls), complete in stream order
 *  regions              HOST array of W ep_rank_region_t, read during the call
 *                       (the table travels with the launch; the caller may
 *                       reuse the array as soon as the call returns)
 * Limits: those of ep_dispatch.
 */
EP_API int ep_dispatch_regions(const void* x, const int32_t* topk_idx, const float* topk_w,
                               int64_t T, int H, int k, int W, const int32_t* slot,
                               const int32_t* rank_offset, const ep_rank_region_t* regions,
                               int quant, int32_t* status, ep_stream_t stream);

/*
 * Layout and dispatch into per-rank regions in one call: ep_dispatch_layout
 * followed by ep_dispatch_regions on the same stream, with their arguments,
 * limits, results and errors (every layout output is written; region r gets
 * the rows that ep_dispatch_regions would write).  As in
 * ep_dispatch_with_layout, the dispatch loads its first rows of x while the
 * layout kernels run (x must be complete in stream order before this call),
 * and beyond 1024 tokens (bf16 rows of at least 1 KB, or FP8) it finishes the
 * layout itself and its bulk-copy warps take tokens from a counter in the
 * workspace, so the workspace serves one call at a time; bf16 batches of up
 * to 512 tokens take the one-launch kernel, as in ep_dispatch_with_layout.
 * Same passages as ep_dispatch_layout and ep_dispatch_regions.
 */
EP_API int ep_dispatch_regions_with_layout(const void* x, const int32_t* topk_idx,
                                           const float* topk_w, int64_t T, int H, int k, int E,
                                           int W, int32_t* num_tokens_per_expert,
                                           int32_t* num_tokens_per_rank, int32_t* rank_offset,
                                           int32_t* slot, void* workspace, size_t workspace_bytes,
                                           const ep_rank_region_t* regions, int quant,
                                           int32_t* status, ep_stream_t stream);

/*
 * Combine from per-rank regions: ep_combine with rank r's expert outputs in an
 * allocation of their own.  The row of (t, r) is y_regions[r] row
 * slot[t][r] - rank_offset[r]; out[t] is the bf16 rounding of the fp32 sum of
 * those rows over the ranks of D(t) in ascending order from +0, as in
 * ep_combine.  Rows at or beyond y_rows[r] are skipped and set
 * EP_STATUS_CAPACITY.  Follows "perf(ep): optimize IntraNode dispatch kernel
 * for MI350X", "Remaining gap" (combine reads each token's rows where the
 * ranks hold them and accumulates them).
 *
 *  y_regions  HOST array of W device pointers, bf16 [y_rows[r], H], 16-byte aligned
 *  y_rows     HOST array of W capacities
 *  slot, rank_offset, out  as for ep_combine / ep_dispatch_regions
 * Limits: H % 8 == 0; 1 <= W <= 32.
 */
EP_API int ep_combine_regions(const void* const* y_regions, const int64_t* y_rows,
                              const int32_t* slot, const int32_t* rank_offset, int64_t T, int H,
                              int W, void* out, int32_t* status, ep_stream_t stream);

/*
 * ep_dispatch_layout without a workspace argument, for callers that cannot
 * allocate device memory: C or embedded hosts without a device allocator, and
 * latency-critical paths that must not call cudaMalloc (it blocks the host and
 * synchronises the device).  The pages have no counterpart; this is an entry
 * point of this library only.
 *
 * The workspace is a device array of EP_LAYOUT_NOALLOC_SCRATCH_BYTES built into
 * the library; every GPU that loads the library holds it until the process
 * exits.  Arguments, outputs and status bits are those of ep_dispatch_layout;
 * the call allocates nothing.
 *  - Returns EP_ERR_WORKSPACE when ep_layout_workspace_bytes(T, W, E) exceeds
 *    EP_LAYOUT_NOALLOC_SCRATCH_BYTES (up to 85504 tokens at W = 8, E = 256).
 *  - The first call in a CUDA context looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it per device, keyed by the context's
 *    unique id: a context re-created after cudaDeviceReset, or another context
 *    made current on the device, triggers a new lookup, never a stale address.
 *    Make that first call in each context before any stream capture in it.
 *  - All calls share the one array: calls whose kernels overlap on the GPU
 *    (other streams, other host threads) race and must be serialised by the
 *    caller.  The array needs no clearing: each call writes what it reads.
 */
#define EP_LAYOUT_NOALLOC_SCRATCH_BYTES (1u << 20)
EP_API int ep_dispatch_layout_noalloc(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                                      int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                      int32_t* rank_offset, int32_t* slot, int32_t* status,
                                      ep_stream_t stream);

/*
 * Expert-major layout: one receive row per valid (token, top-k column) pair,
 * grouped by expert, for an expert side that runs one grouped GEMM over its
 * experts.  Expert e owns rows [expert_offset[e], expert_offset[e+1]), the
 * exclusive prefix sum of num_tokens_per_expert, and inside them the pairs
 * come in (token, column) order; slot[t][j] is the row of pair (t, j), or -1
 * when topk_idx[t][j] is outside [0, E) (then EP_STATUS_BAD_EXPERT is set).  A
 * token that names one expert twice gets two rows.  The experts of rank r
 * are r*Er .. (r+1)*Er - 1, so rank r's rows are the range
 * [expert_offset[r*Er], expert_offset[(r+1)*Er]).  This is the per-expert
 * receive layout of the recv kernel in "Optimizing Distributed Inference
 * Kernels for AMD DEVELOPER CHALLENGE 2025", section 3.1 item 1, packed by a
 * scan of the counts instead of a fixed per-expert maximum.
 *
 * The payload moves with ep_dispatch(..., W = k, slot, ...), which copies the
 * token row to every row its slot table names (here one per valid column), and
 * comes back with ep_combine_weighted(y, slot, topk_w, T, H, k, ...).
 *
 *  topk_idx               int32 [T, k]
 *  num_tokens_per_expert  int32 [E]      valid pairs per expert
 *  expert_offset          int32 [E + 1]  expert_offset[E] = number of rows
 *  slot                   int32 [T, k]
 *  workspace              >= ep_layout_experts_workspace_bytes(T, k, E) bytes,
 *                         16-byte aligned, no initialisation; it serves one
 *                         call at a time
 * Limits: 1 <= k; 1 <= E <= 4096; T * k < 2^31.  Up to 2048 pairs and 1024
 * experts it is one kernel on one CTA; above that a count and an assign kernel
 * (and a scan kernel between them beyond 32 chunks of 1024 pairs).
 * ep_layout_experts_workspace_bytes (host only, 0 for invalid arguments) is a
 * convention of this library, like ep_layout_workspace_bytes; the pages define
 * no such call.
 */
EP_API size_t ep_layout_experts_workspace_bytes(int64_t T, int k, int E);
EP_API int ep_dispatch_layout_experts(const int32_t* topk_idx, int64_t T, int k, int E,
                                      int32_t* num_tokens_per_expert, int32_t* expert_offset,
                                      int32_t* slot, void* workspace, size_t workspace_bytes,
                                      int32_t* status, ep_stream_t stream);

/*
 * Expert-major layout and dispatch in one call: ep_dispatch_layout_experts
 * followed by ep_dispatch of its [T, k] slot table (W = k) on the same stream,
 * with the same arguments, limits (also k <= 32), results and errors.  The
 * dispatch becomes resident while the layout kernels run and loads its first
 * rows of x before the slots exist (x must be complete in stream order before
 * this call).  Above 2048 pairs or 1024 experts, its bf16 bulk-copy warps
 * then take tokens from a counter that the layout's count kernel zeroes in the
 * workspace, so the workspace must not be shared by calls that overlap on the
 * GPU; which warp sends which token varies from call to call, the results do
 * not.
 */
EP_API int ep_dispatch_experts_with_layout(const void* x, const int32_t* topk_idx,
                                           const float* topk_w, int64_t T, int H, int k, int E,
                                           int32_t* num_tokens_per_expert,
                                           int32_t* expert_offset, int32_t* slot, void* workspace,
                                           size_t workspace_bytes, int64_t capacity_rows,
                                           int quant, void* recv_x, float* recv_scale,
                                           int32_t* recv_topk_idx, float* recv_topk_w,
                                           int32_t* recv_src, int32_t* status,
                                           ep_stream_t stream);

/*
 * Weighted combine over a slot table of C columns:
 *   out[t] = bf16_rne( fma(w[t][c_n], y[s_n], ... fma(w[t][c_1], y[s_1], +0)) )
 * over the columns c with s = slot[t][c] >= 0 in ascending order, each step one
 * fp32 fused multiply-add (rounded once).  With the expert-major slot table and
 * w = topk_w it is the gate-weighted sum of the token's expert outputs; with a
 * rank-major slot table [T, W] and per-(token, rank) weights it is the weighted
 * form of ep_combine, which it equals bit for bit when every weight is 1.
 * Follows "perf(ep): optimize IntraNode dispatch kernel for MI350X", "Remaining
 * gap" (combine accumulates the pre-routed rows with FMA).
 *
 *  y     bf16 [capacity_rows, H]   expert outputs, one per receive row
 *  slot  int32 [T, C]
 *  w     fp32 [T, C]               read only where slot >= 0
 *  out   bf16 [T, H]
 * Rows >= capacity_rows are skipped and set EP_STATUS_CAPACITY.
 * Limits: H % 8 == 0; 1 <= C <= 32.
 */
EP_API int ep_combine_weighted(const void* y, const int32_t* slot, const float* w, int64_t T,
                               int H, int C, int64_t capacity_rows, void* out, int32_t* status,
                               ep_stream_t stream);

/*
 * FP8 cast and transposed cast of the expert-major rows, with the amax fused,
 * for expert GEMMs that take FP8 operands (row-major for the forward product,
 * transposed for the weight gradient).  Expert e owns rows
 * [expert_offset[e], expert_offset[e+1]) of y (n_e rows); with its scale s_e
 * every element gets code = e4m3(fl(x * s_e)) (fp32 product, then round to
 * nearest even, saturating to +-448):
 *   out_c[row][h] = code (row-major, the rows of y),
 *   out_t[H * (ld_0 + ... + ld_{e-1}) + h * ld_e + i] = code of row
 *     expert_offset[e] + i, column h, with ld_e = n_e rounded up to a multiple
 *     of 16 (the padding bytes are 0): one [H][ld_e] block per expert,
 *   amax[e] = max(amax[e], max |x| over the expert's rows) (zero amax first
 *     for a fresh maximum).
 * Follows "Optimized rocm specific multicast transpose kernel" (ROCm/
 * TransformerEngine pull 586): both casts of every expert's tensor in one
 * launch, amax fused, pad-16 rows.
 *
 *  y              bf16 [capacity_rows, H]   (from ep_dispatch into the expert-major layout)
 *  expert_offset  int32 [E + 1], nondecreasing (from ep_dispatch_layout_experts)
 *  scale          fp32 [E]
 *  out_c          uint8 [capacity_rows, H]
 *  out_t          uint8, ep_cast_transpose_t_bytes(capacity_rows, E, H) bytes
 *  amax           fp32 [E], read and written
 * Experts whose rows leave [0, capacity_rows) are skipped and set
 * EP_STATUS_CAPACITY.  Limits: H % 256 == 0; 1 <= E <= 8192.
 * ep_cast_transpose_t_bytes (host only, 0 for invalid arguments) gives the
 * size of out_t; a convention of this library, the pages define no such call.
 */
EP_API size_t ep_cast_transpose_t_bytes(int64_t capacity_rows, int E, int H);
EP_API int ep_cast_transpose_experts(const void* y, const int32_t* expert_offset, int E, int H,
                                     const float* scale, int64_t capacity_rows, void* out_c,
                                     void* out_t, float* amax, int32_t* status, ep_stream_t stream);

/*
 * Self-test of the bounded waits (diagnostic, not part of the data path).
 * Launches one kernel that waits, with the helper every kernel of the library
 * uses for its on-chip waits, on a barrier that nothing completes.  After
 * about one second the wait gives up: the kernel ORs EP_STATUS_TIMEOUT into
 * *status (device int32, required) and returns, and the context stays usable.
 * Returns EP_OK once the kernel is enqueued; the caller synchronises and reads
 * *status.  A diagnostic of this library; the pages define no such call (their
 * waits on peer memory are unbounded).
 */
EP_API int ep_selftest_wait_timeout(int32_t* status, ep_stream_t stream);

/* Human-readable name of an EP_* return code (static string, never NULL;
 * "unknown ep status code" for other values).  Host only.  A convention of
 * this library; the pages define no such call. */
EP_API const char* ep_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* EP_GB300_H */
