// Routing layout: per-expert and per-rank counts, a stable exclusive scan over
// the per-rank counts, and the receive slot of every (token, rank) pair.
//
// Two kernels, both over chunks of kLT tokens (one token per thread):
//   count: decode each token's expert ids into its destination-rank bit set
//          (deduplication by construction), tally the chunk's per-rank and
//          per-expert counts into the workspace;
//   scan:  every CTA reduces the per-chunk rank counts (all chunks, and those
//          before its own), derives rank_offset and its chunk's base row per
//          rank, then numbers its tokens in ascending order with warp ballots.
// Integer counts only, no atomics whose order could leak into a result: the
// layout is a pure function of topk_idx.
#include <cuda.h>

#include <mutex>

#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kLTShift = 7;
constexpr int kLT = 1 << kLTShift;  // tokens per CTA, one per thread
constexpr int kLWarps = kLT / 32;

inline size_t a256(size_t b) { return (b + 255) & ~size_t(255); }

struct LayoutWs {
  uint32_t* mask;       // [T]     bit r set iff r in D(t)
  int32_t* chunk_rank;  // [C][W]  tokens of chunk c with r in D(t)
  int32_t* chunk_exp;   // [C][E]  (t, j) entries of chunk c with expert e
  unsigned long long* claim;  // token counter of the dispatch that finishes the layout
};

inline int64_t num_chunks(int64_t T) { return T <= 0 ? 1 : (T + kLT - 1) / kLT; }

LayoutWs carve(void* ws, int64_t T, int W, int E) {
  char* p = static_cast<char*>(ws);
  const int64_t C = num_chunks(T);
  LayoutWs w;
  w.mask = reinterpret_cast<uint32_t*>(p);
  p += a256(sizeof(uint32_t) * (size_t)T);
  w.chunk_rank = reinterpret_cast<int32_t*>(p);
  p += a256(sizeof(int32_t) * (size_t)(C * W));
  w.chunk_exp = reinterpret_cast<int32_t*>(p);
  p += a256(sizeof(int32_t) * (size_t)(C * (size_t)E));
  w.claim = reinterpret_cast<unsigned long long*>(p);
  return w;
}

// The k expert ids of a token row, loaded into registers before any is used:
// VEC reads the row as int4 (k == KV, KV % 4 == 0, 16-byte aligned rows),
// otherwise KV guarded scalar loads (k <= KV; missing entries read as -1).
template <int KV, bool VEC>
__device__ __forceinline__ void load_row(const int32_t* __restrict__ row, int k, bool live,
                                         int (&e)[KV]) {
  if constexpr (VEC) {
#pragma unroll
    for (int v = 0; v < KV / 4; ++v) {
      const int4 q = live ? __ldg(reinterpret_cast<const int4*>(row) + v) : make_int4(-1, -1, -1, -1);
      e[4 * v + 0] = q.x;
      e[4 * v + 1] = q.y;
      e[4 * v + 2] = q.z;
      e[4 * v + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < KV; ++j) e[j] = (live && j < k) ? __ldg(row + j) : -1;
  }
}

// Destination ranks of a token: rank = expert / experts-per-rank, one entry per
// distinct rank ("perf(ep): optimize IntraNode dispatch kernel for MI350X",
// Technical Details 1).  The bit set is the cached routing of that section: it
// is computed here once and consumed by the scan.  All k ids of a token are
// loaded before any is used, so the chunk costs one memory round trip.
template <int KV, bool VEC>
__global__ void __launch_bounds__(kLT)
    layout_count_kernel(const int32_t* __restrict__ topk_idx, int64_t T, int k, int E, int W,
                        int Er, LayoutWs ws, int32_t* __restrict__ status,
                        int32_t* __restrict__ local_slot) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int32_t s_hist[];  // [E]
  __shared__ int32_t s_warp_rank[kLWarps][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t t = (int64_t)blockIdx.x * kLT + tid;
  const bool live = t < T;
  const int32_t* row = topk_idx + (live ? t * k : 0);
  uint32_t m = 0;
  bool bad = false;
  int ids[KV > 0 ? KV : 1];
  if constexpr (KV > 0) load_row<KV, VEC>(row, k, live, ids);
  for (int e = tid; e < E; e += kLT) s_hist[e] = 0;
  __syncthreads();

  const int kk = KV > 0 ? KV : k;
#pragma unroll
  for (int j = 0; j < kk; ++j) {
    int e;
    if constexpr (KV > 0)
      e = ids[j];
    else
      e = live ? __ldg(row + j) : -1;
    const bool in_row = KV == 0 || VEC || j < k;
    const bool ok = in_row && (unsigned)e < (unsigned)E;
    bad |= live && in_row && !ok;
    if (ok) {
      m |= 1u << (e / Er);
      atomicAdd(&s_hist[e], 1);
    }
  }
  if (live) ws.mask[t] = m;
  // the dispatch that finishes this layout claims tokens from this counter
  // (it reads it only after this kernel has completed)
  if (blockIdx.x == 0 && tid == 0) *ws.claim = 0ull;

  int cnt = 0;
  for (int r = 0; r < W; ++r) {
    const unsigned b = __ballot_sync(kFull, (m >> r) & 1u);
    if (lane == r) cnt = __popc(b);
  }
  if (lane < W) s_warp_rank[warp][lane] = cnt;
  if (__any_sync(kFull, bad) && lane == 0 && status != nullptr) atomicOr(status, EP_STATUS_BAD_EXPERT);
  __syncthreads();

  if (tid < W) {
    int s = 0;
#pragma unroll
    for (int w = 0; w < kLWarps; ++w) s += s_warp_rank[w][tid];
    ws.chunk_rank[(int64_t)blockIdx.x * W + tid] = s;
  }
  for (int e = tid; e < E; e += kLT) ws.chunk_exp[(int64_t)blockIdx.x * E + e] = s_hist[e];

  // Optionally the position p of (t, r) inside the chunk (rows of r in earlier
  // warps of the chunk plus rows of r in earlier lanes of this warp), stored
  // as -2 - p so that it can never be mistaken for a receive row (>= 0) or for
  // "not a destination" (-1).  A later kernel adds the chunk's base row.
  if (local_slot != nullptr) {
    const unsigned lt = lanemask_lt();
    int32_t* srow = local_slot + (live ? t * W : 0);
    for (int r = 0; r < W; ++r) {
      const unsigned in_r = (m >> r) & 1u;
      const unsigned b = __ballot_sync(kFull, in_r);
      int before = 0;
      for (int w = 0; w < warp; ++w) before += s_warp_rank[w][r];
      if (live) srow[r] = in_r ? -2 - (before + __popc(b & lt)) : -1;
    }
  }
}

// Stable exclusive scan and slots.  The receive rows of rank r are
// [rank_offset[r], rank_offset[r+1]) in ascending token order; the slot of
// (t, r) is rank_offset[r] + (rows of r in earlier chunks) + (rows of r in
// earlier warps of this chunk) + (rows of r in earlier lanes of this warp).
// Per-expert totals are spread over the grid: CTA c sums experts c, c+C, ...
// with one warp per expert and the chunks spread over the lanes.
__global__ void __launch_bounds__(kLT)
    layout_scan_kernel(int64_t T, int E, int W, int64_t C, LayoutWs ws,
                       int32_t* __restrict__ num_tokens_per_expert,
                       int32_t* __restrict__ num_tokens_per_rank, int32_t* __restrict__ rank_offset,
                       int32_t* __restrict__ slot) {
  pdl_wait();
  pdl_launch_dependents();  // the next kernel may become resident (its own wait still holds)
  __shared__ int32_t s_total[32], s_before[32];
  __shared__ int32_t s_warp_cnt[kLWarps][32];
  __shared__ int32_t s_base[kLWarps][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t c = blockIdx.x;
  const int64_t t = c * kLT + tid;
  const bool live = t < T;
  const uint32_t m = live ? ws.mask[t] : 0u;

  for (int r = warp; r < W; r += kLWarps) {
    int tot = 0, bef = 0;
    for (int64_t q = lane; q < C; q += 32) {
      const int v = ws.chunk_rank[q * W + r];
      tot += v;
      if (q < c) bef += v;
    }
    tot = warp_sum(tot);
    bef = warp_sum(bef);
    if (lane == 0) {
      s_total[r] = tot;
      s_before[r] = bef;
    }
  }
  int cnt = 0;
  for (int r = 0; r < W; ++r) {
    const unsigned b = __ballot_sync(kFull, (m >> r) & 1u);
    if (lane == r) cnt = __popc(b);
  }
  if (lane < W) s_warp_cnt[warp][lane] = cnt;
  __syncthreads();
  if (tid < W) {
    int off = 0;
    for (int r = 0; r < tid; ++r) off += s_total[r];
    if (c == 0) {
      rank_offset[tid] = off;
      num_tokens_per_rank[tid] = s_total[tid];
      if (tid == W - 1) rank_offset[W] = off + s_total[tid];
    }
    int acc = off + s_before[tid];
#pragma unroll
    for (int w = 0; w < kLWarps; ++w) {
      s_base[w][tid] = acc;
      acc += s_warp_cnt[w][tid];
    }
  }
  __syncthreads();

  const unsigned lt = lanemask_lt();
  int32_t* srow = slot + (live ? t * W : 0);
  if ((W & 3) == 0 && (reinterpret_cast<uintptr_t>(slot) & 15) == 0) {
    for (int r0 = 0; r0 < W; r0 += 4) {
      int v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const unsigned in_r = (m >> (r0 + i)) & 1u;
        const unsigned b = __ballot_sync(kFull, in_r);
        v[i] = in_r ? s_base[warp][r0 + i] + __popc(b & lt) : -1;
      }
      if (live) reinterpret_cast<int4*>(srow)[r0 >> 2] = make_int4(v[0], v[1], v[2], v[3]);
    }
  } else {
    for (int r = 0; r < W; ++r) {
      const unsigned in_r = (m >> r) & 1u;
      const unsigned b = __ballot_sync(kFull, in_r);
      if (live) srow[r] = in_r ? s_base[warp][r] + __popc(b & lt) : -1;
    }
  }

  // per-expert totals over the chunks: with many chunks a warp per expert
  // (chunks over the lanes), with few a thread per expert
  if (C >= 16) {
    for (int64_t e = c + (int64_t)warp * gridDim.x; e < E; e += (int64_t)kLWarps * gridDim.x) {
      int s = 0;
      for (int64_t q = lane; q < C; q += 32) s += ws.chunk_exp[q * E + e];
      s = warp_sum(s);
      if (lane == 0) num_tokens_per_expert[e] = s;
    }
  } else {
    for (int64_t e = c * kLT + tid; e < E; e += (int64_t)gridDim.x * kLT) {
      int s = 0;
#pragma unroll 16
      for (int64_t q = 0; q < C; ++q) s += ws.chunk_exp[q * E + e];
      num_tokens_per_expert[e] = s;
    }
  }
}

// Whole layout in one CTA, for T <= kSingleMaxT: no workspace traffic and one
// launch instead of two dependent ones.  Measured on GB300 it saves about half
// a microsecond at T <= 1024 (one batch per thread) but doubles the time at
// T = 4096, where one SM works through the batches alone: larger batches take
// the two-kernel path below.
// Thread i takes tokens i, i + 1024, ...; per token: the k ids (one vector
// load per 4 ids, all issued before use), the rank bit set (kept in shared
// memory) and the per-expert histogram (shared atomics).  Per batch of 1024
// tokens each warp counts its 32 tokens per rank with ballots; one warp per
// rank then scans those counts in token order (batch, warp), which gives every
// (batch, warp, rank) its first receive row; a token's slot adds the rows of
// the earlier lanes of its warp (ballot + popc).
constexpr int kSingleThreads = 1024;
constexpr int kSingleWarps = kSingleThreads / 32;
constexpr int kSingleMaxT = (int)kLayoutSingleMaxT;
constexpr int kSingleMaxBatches = kSingleMaxT / kSingleThreads;

template <int KV, bool VEC>
__global__ void __launch_bounds__(kSingleThreads, 1)
    layout_single_kernel(const int32_t* __restrict__ topk_idx, int T, int k, int E, int W, int Er,
                         int32_t* __restrict__ num_tokens_per_expert,
                         int32_t* __restrict__ num_tokens_per_rank,
                         int32_t* __restrict__ rank_offset, int32_t* __restrict__ slot,
                         int32_t* __restrict__ status) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int32_t s_dyn[];
  int32_t* s_hist = s_dyn;                                   // [E]
  uint32_t* s_mask = reinterpret_cast<uint32_t*>(s_dyn + E);  // [T]
  __shared__ int32_t s_cnt[kSingleMaxBatches][kSingleWarps][32];  // rows per (batch, warp, rank)
  __shared__ int32_t s_off[33];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nbatch = (T + kSingleThreads - 1) / kSingleThreads;
  for (int e = tid; e < E; e += kSingleThreads) s_hist[e] = 0;
  __syncthreads();

  bool bad = false;
  for (int i = 0; i < nbatch; ++i) {
    const int t = i * kSingleThreads + tid;
    const bool live = t < T;
    int ids[KV > 0 ? KV : 1];
    if constexpr (KV > 0) load_row<KV, VEC>(topk_idx + (live ? (int64_t)t * k : 0), k, live, ids);
    uint32_t m = 0;
    const int kk = KV > 0 ? KV : k;
#pragma unroll
    for (int j = 0; j < kk; ++j) {
      int e;
      if constexpr (KV > 0)
        e = ids[j];
      else
        e = live ? __ldg(topk_idx + (int64_t)t * k + j) : -1;
      const bool in_row = KV == 0 || VEC || j < k;
      const bool ok = in_row && (unsigned)e < (unsigned)E;
      bad |= live && in_row && !ok;
      if (ok) {
        m |= 1u << (e / Er);
        atomicAdd(&s_hist[e], 1);
      }
    }
    if (live) s_mask[t] = m;
    int cnt = 0;
    for (int r = 0; r < W; ++r) {
      const unsigned b = __ballot_sync(kFull, (m >> r) & 1u);
      if (lane == r) cnt = __popc(b);
    }
    if (lane < W) s_cnt[i][warp][lane] = cnt;
  }
  if (__any_sync(kFull, bad) && lane == 0 && status != nullptr) atomicOr(status, EP_STATUS_BAD_EXPERT);
  __syncthreads();

  // warp r: exclusive scan of rank r's counts over (batch, warp) in token order
  for (int r = warp; r < W; r += kSingleWarps) {
    int carry = 0;
    for (int i = 0; i < nbatch; ++i) {
      const int v = s_cnt[i][lane][r];
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      s_cnt[i][lane][r] = carry + incl - v;
      carry += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) s_off[r] = carry;  // total of rank r, for now
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int r = 0; r < W; ++r) {
      const int tot = s_off[r];
      num_tokens_per_rank[r] = tot;
      rank_offset[r] = acc;
      s_off[r] = acc;
      acc += tot;
    }
    rank_offset[W] = acc;
  }
  __syncthreads();

  const unsigned lt = lanemask_lt();
  const bool vec_slot = (W & 3) == 0 && (reinterpret_cast<uintptr_t>(slot) & 15) == 0;
  for (int i = 0; i < nbatch; ++i) {
    const int t = i * kSingleThreads + tid;
    const bool live = t < T;
    const uint32_t m = live ? s_mask[t] : 0u;
    int32_t* srow = slot + (live ? (int64_t)t * W : 0);
    if (vec_slot) {
      for (int r0 = 0; r0 < W; r0 += 4) {
        int v[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = r0 + q;
          const unsigned in_r = (m >> r) & 1u;
          const unsigned b = __ballot_sync(kFull, in_r);
          v[q] = in_r ? s_off[r] + s_cnt[i][warp][r] + __popc(b & lt) : -1;
        }
        if (live) reinterpret_cast<int4*>(srow)[r0 >> 2] = make_int4(v[0], v[1], v[2], v[3]);
      }
    } else {
      for (int r = 0; r < W; ++r) {
        const unsigned in_r = (m >> r) & 1u;
        const unsigned b = __ballot_sync(kFull, in_r);
        if (live) srow[r] = in_r ? s_off[r] + s_cnt[i][warp][r] + __popc(b & lt) : -1;
      }
    }
  }
  for (int e = tid; e < E; e += kSingleThreads) num_tokens_per_expert[e] = s_hist[e];
}

}  // namespace

int64_t layout_num_chunks(int64_t T) { return num_chunks(T); }

size_t layout_workspace_bytes(int64_t T, int W, int E) {
  const int64_t C = num_chunks(T);
  return a256(sizeof(uint32_t) * (size_t)T) + a256(sizeof(int32_t) * (size_t)(C * W)) +
         a256(sizeof(int32_t) * (size_t)(C * E)) + a256(sizeof(unsigned long long));
}

cudaError_t launch_layout_count(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                                void* workspace, int32_t* local_slot, int32_t* status,
                                cudaStream_t stream, LayoutChunks* chunks) {
  const bool vec = (reinterpret_cast<uintptr_t>(topk_idx) & 15) == 0;
  const int64_t C = num_chunks(T);
  const LayoutWs ws = carve(workspace, T, W, E);
  chunks->chunk_rank = ws.chunk_rank;
  chunks->chunk_exp = ws.chunk_exp;
  chunks->C = C;
  chunks->shift = kLTShift;
  chunks->claim = ws.claim;
  const size_t smem = sizeof(int32_t) * (size_t)E;
  if (k == 8 && vec)
    return launch_pdl(layout_count_kernel<8, true>, dim3((unsigned)C), dim3(kLT), smem, stream,
                      topk_idx, T, k, E, W, E / W, ws, status, local_slot);
  if (k == 4 && vec)
    return launch_pdl(layout_count_kernel<4, true>, dim3((unsigned)C), dim3(kLT), smem, stream,
                      topk_idx, T, k, E, W, E / W, ws, status, local_slot);
  if (k <= 16)
    return launch_pdl(layout_count_kernel<16, false>, dim3((unsigned)C), dim3(kLT), smem, stream,
                      topk_idx, T, k, E, W, E / W, ws, status, local_slot);
  return launch_pdl(layout_count_kernel<0, false>, dim3((unsigned)C), dim3(kLT), smem, stream,
                    topk_idx, T, k, E, W, E / W, ws, status, local_slot);
}

cudaError_t launch_layout(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                          int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                          int32_t* rank_offset, int32_t* slot, void* workspace, int32_t* status,
                          cudaStream_t stream) {
  const bool vec = (reinterpret_cast<uintptr_t>(topk_idx) & 15) == 0;
  if (T <= kSingleMaxT) {
    const size_t smem1 = sizeof(int32_t) * ((size_t)E + (size_t)T);
    static bool attr_set[128];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 128 && !attr_set[dev]) {
      const int most = (int)(sizeof(int32_t) * (8192 + kSingleMaxT));  // E <= 8192
      cudaError_t e;
      if ((e = cudaFuncSetAttribute(layout_single_kernel<8, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, most)) != cudaSuccess ||
          (e = cudaFuncSetAttribute(layout_single_kernel<4, true>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, most)) != cudaSuccess ||
          (e = cudaFuncSetAttribute(layout_single_kernel<16, false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, most)) != cudaSuccess ||
          (e = cudaFuncSetAttribute(layout_single_kernel<0, false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, most)) != cudaSuccess)
        return e;
      attr_set[dev] = true;
    }
    const int Ti = (int)T;
    if (k == 8 && vec)
      return launch_pdl(layout_single_kernel<8, true>, dim3(1), dim3(kSingleThreads), smem1, stream,
                        topk_idx, Ti, k, E, W, E / W, num_tokens_per_expert, num_tokens_per_rank,
                        rank_offset, slot, status);
    if (k == 4 && vec)
      return launch_pdl(layout_single_kernel<4, true>, dim3(1), dim3(kSingleThreads), smem1, stream,
                        topk_idx, Ti, k, E, W, E / W, num_tokens_per_expert, num_tokens_per_rank,
                        rank_offset, slot, status);
    if (k <= 16)
      return launch_pdl(layout_single_kernel<16, false>, dim3(1), dim3(kSingleThreads), smem1,
                        stream, topk_idx, Ti, k, E, W, E / W, num_tokens_per_expert,
                        num_tokens_per_rank, rank_offset, slot, status);
    return launch_pdl(layout_single_kernel<0, false>, dim3(1), dim3(kSingleThreads), smem1, stream,
                      topk_idx, Ti, k, E, W, E / W, num_tokens_per_expert, num_tokens_per_rank,
                      rank_offset, slot, status);
  }
  const int64_t C = num_chunks(T);
  const LayoutWs ws = carve(workspace, T, W, E);
  const size_t smem = sizeof(int32_t) * (size_t)E;
  cudaError_t err;
  if (k == 8 && vec)
    err = launch_pdl(layout_count_kernel<8, true>, dim3((unsigned)C), dim3(kLT), smem, stream,
                     topk_idx, T, k, E, W, E / W, ws, status, nullptr);
  else if (k == 4 && vec)
    err = launch_pdl(layout_count_kernel<4, true>, dim3((unsigned)C), dim3(kLT), smem, stream,
                     topk_idx, T, k, E, W, E / W, ws, status, nullptr);
  else if (k <= 16)
    err = launch_pdl(layout_count_kernel<16, false>, dim3((unsigned)C), dim3(kLT), smem, stream,
                     topk_idx, T, k, E, W, E / W, ws, status, nullptr);
  else
    err = launch_pdl(layout_count_kernel<0, false>, dim3((unsigned)C), dim3(kLT), smem, stream,
                     topk_idx, T, k, E, W, E / W, ws, status, nullptr);
  if (err != cudaSuccess) return err;
  return launch_pdl(layout_scan_kernel, dim3((unsigned)C), dim3(kLT), 0, stream, T, E, W, C, ws,
                    num_tokens_per_expert, num_tokens_per_rank, rank_offset, slot);
}

}  // namespace ep

// ---------------------------------------------------------------------------
// Layout without a caller-provided workspace.
//
// Some callers cannot allocate device memory where they need the layout: C or
// embedded hosts with no device allocator of their own, and latency-critical
// paths where cudaMalloc is off limits because it blocks the host and
// synchronises the device.  For them the library keeps the layout workspace in
// a fixed device array of EP_LAYOUT_NOALLOC_SCRATCH_BYTES, reserved on every
// GPU that loads the library until the process exits.
//
// Host code cannot use the array's name as a device address (on the host it
// names a stand-in), so the runtime is asked for the address with
// cudaGetSymbolAddress, with the caller's device current.  The address belongs
// to a CUDA context, not to a device number: the lookup is cached per device
// together with the unique id of the context that was current (cuCtxGetId), and
// repeated whenever that id changes (the primary context re-created after
// cudaDeviceReset, or another context made current on the device).  Every call
// uses the same array: calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on it.  Nothing in it needs
// clearing between calls: each call writes every word it reads before reading
// it.
static __device__ __align__(256) unsigned char
    g_layout_noalloc_scratch[EP_LAYOUT_NOALLOC_SCRATCH_BYTES];

namespace ep {
namespace {

constexpr int kMaxDevices = 128;

// The driver's cuCtxGetCurrent and cuCtxGetId, resolved at run time through
// the runtime (the library does not link the driver library itself).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static const DriverFns fns = [] {
    DriverFns f;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
    return f;
  }();
  return fns;
}

// Unique id of the current context; false when it cannot be had (no context
// current yet, or an old driver).
bool current_context_id(unsigned long long* id) {
  const DriverFns& f = driver_fns();
  if (f.get_current == nullptr || f.get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return f.get_id(ctx, id) == CUDA_SUCCESS;
}

struct ScratchEntry {
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
ScratchEntry g_noalloc_cache[kMaxDevices];
std::mutex g_noalloc_mutex;

cudaError_t noalloc_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  ScratchEntry& c = g_noalloc_cache[dev];
  if (have_id && c.addr != nullptr && c.ctx_id == id) {
    *out = c.addr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_layout_noalloc_scratch);  // makes a context current if none was
  if (e != cudaSuccess) return e;
  unsigned long long id_now = 0;
  if (current_context_id(&id_now)) {
    c.ctx_id = id_now;
    c.addr = p;
  } else {
    c.addr = nullptr;  // no id to key on: look the address up on every call
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace
}  // namespace ep

extern "C" EP_API int ep_dispatch_layout_noalloc(const int32_t* topk_idx, int64_t T, int k, int E,
                                                 int W, int32_t* num_tokens_per_expert,
                                                 int32_t* num_tokens_per_rank, int32_t* rank_offset,
                                                 int32_t* slot, int32_t* status, ep_stream_t stream) {
  if (T < 0 || k < 1 || W < 1 || W > 32 || E < 1 || E > 8192 || E % W != 0)
    return EP_ERR_INVALID_ARG;
  if (T * (k < W ? k : W) > 0x7fffffffLL || T > 0x7fffffffLL / W) return EP_ERR_UNSUPPORTED;
  if (ep::layout_workspace_bytes(T, W, E) > (size_t)EP_LAYOUT_NOALLOC_SCRATCH_BYTES)
    return EP_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (ep::noalloc_scratch_address(&scratch) != cudaSuccess) return EP_ERR_CUDA;
  return ep_dispatch_layout(topk_idx, T, k, E, W, num_tokens_per_expert, num_tokens_per_rank,
                            rank_offset, slot, scratch, (size_t)EP_LAYOUT_NOALLOC_SCRATCH_BYTES,
                            status, stream);
}


// ---------------------------------------------------------------------------
// Local expert ids of the receive rows, in place.  Row s belongs to rank r
// with rank_offset[r] <= s < rank_offset[r+1]; each of its k ids e becomes
// e - r * (E / W) when e is a valid expert hosted by rank r, and -1 otherwise,
// so that rank r's expert side reads directly which of its experts a row needs.
namespace ep {
namespace {

__global__ void __launch_bounds__(256)
    localize_ids_kernel(int32_t* __restrict__ recv_topk_idx, const int32_t* __restrict__ rank_offset,
                        int64_t cap, int k, int E, int W) {
  pdl_wait();
  __shared__ int32_t s_off[33];
  if (threadIdx.x <= (unsigned)W) s_off[threadIdx.x] = rank_offset[threadIdx.x];
  __syncthreads();
  const int64_t rows = (int64_t)s_off[W] < cap ? (int64_t)s_off[W] : cap;
  const int Er = E / W;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < rows * k;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t s = i / k;
    int lo = 0, hi = W - 1;  // the rank whose region holds row s
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)s_off[mid] <= s) lo = mid; else hi = mid - 1;
    }
    const int32_t e = recv_topk_idx[i];
    recv_topk_idx[i] = (e >= 0 && e < E && e / Er == lo) ? e - lo * Er : -1;
  }
  pdl_launch_dependents();
}

}  // namespace

cudaError_t launch_localize_ids(int32_t* recv_topk_idx, const int32_t* rank_offset, int64_t cap,
                                int k, int E, int W, cudaStream_t stream) {
  const int64_t sms = device_sm_count();
  const int grid = (int)(sms > 0 ? sms * 4 : 1);
  return launch_pdl(localize_ids_kernel, dim3(grid), dim3(256), 0, stream, recv_topk_idx,
                    rank_offset, cap, k, E, W);
}

}  // namespace ep
