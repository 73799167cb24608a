// Routing layout and bf16 dispatch in one launch, for small batches.
//
// A decode-sized batch moves little data, so two dependent launches (layout,
// then dispatch) and the slot round trip between them are most of its cost.
// Here every CTA recomputes the whole layout from the token ids (at most
// kFusedMaxT tokens: a few tens of KB, read from L2 by all but the first CTA),
// writes the slots of the tokens it owns (token t belongs to CTA t mod G; CTA
// 0 also writes the counts and offsets) and then sends those tokens at once.
// This is the single-pass routing of the low-latency kernel discussed on
// "perf(ep): optimize IntraNode dispatch kernel for MI350X" (the IntraNodeLL
// comparison: one routing pass, no separate count/reserve/copy phases), made
// deterministic by the same stable numbering as ep_dispatch_layout.
#include "dispatch_common.cuh"

namespace ep {
namespace {

constexpr int kFThreads = 256;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFusedMaxT = 1024;
constexpr int kFBatches = kFusedMaxT / kFThreads;  // token batches of one per thread
constexpr int kFMaxLocal = 32;                     // tokens owned by one CTA at most
constexpr uint32_t kFMaxTmaRow = 16384;            // larger rows: register copies

// The k expert ids of a token row, loaded before use (int4 when the row is
// 16-byte aligned and k is a multiple of 4, else guarded scalar loads).
template <int KV, bool VEC>
__device__ __forceinline__ void fused_load_row(const int32_t* __restrict__ row, int k, bool live,
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

template <int KV, bool VEC, class RT>
__global__ void __launch_bounds__(kFThreads, 1)
    dispatch_fused_kernel(const uint8_t* __restrict__ x, const int32_t* __restrict__ topk_idx,
                          const float* __restrict__ topk_w, int T, int H, int k, int E, int W,
                          int Er, int32_t* __restrict__ num_tokens_per_expert,
                          int32_t* __restrict__ num_tokens_per_rank,
                          int32_t* __restrict__ rank_offset, int32_t* __restrict__ slot,
                          int64_t cap, uint8_t* __restrict__ recv_x,
                          int32_t* __restrict__ recv_topk_idx, float* __restrict__ recv_topk_w,
                          int32_t* __restrict__ recv_src, int32_t* __restrict__ status, RT rt) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ typename RT::View s_rv;  // per-rank regions: the table
  __shared__ uint64_t s_bar[kFWarps];
  __shared__ int32_t s_cnt[kFBatches][kFWarps][32];  // rows per (batch, warp, rank)
  __shared__ int32_t s_off[33];
  __shared__ int32_t s_lslot[kFMaxLocal][32];        // slots of the tokens this CTA owns
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t row_bytes = (uint32_t)H * 2u;
  const bool tma = row_bytes >= 1024 && row_bytes <= kFMaxTmaRow;
  const uint32_t row_pad = (row_bytes + 127u) & ~127u;
  int32_t* s_hist = reinterpret_cast<int32_t*>(smem + (tma ? (size_t)kFWarps * row_pad : 0));
  const bool first = blockIdx.x == 0;
  if (lane == 0) mbar_init(&s_bar[warp], 1);
  fence_barrier_init();
  if (first)
    for (int e = tid; e < E; e += kFThreads) s_hist[e] = 0;
  __syncthreads();
  load_region_view(rt, W, s_rv);
  pdl_wait();

  // ---------------- layout of the whole batch (every CTA)
  const int G = gridDim.x, c = blockIdx.x;
  const int nb = (T + kFThreads - 1) / kFThreads;
  uint32_t masks[kFBatches];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kFBatches; ++i) {
    masks[i] = 0;
    if (i >= nb) continue;
    const int t = i * kFThreads + tid;
    const bool live = t < T;
    int ids[KV];
    fused_load_row<KV, VEC>(topk_idx + (live ? (int64_t)t * k : 0), k, live, ids);
    uint32_t m = 0;
#pragma unroll
    for (int j = 0; j < KV; ++j) {
      const bool in_row = VEC || j < k;
      const bool ok = in_row && (unsigned)ids[j] < (unsigned)E;
      bad |= live && in_row && !ok;
      if (ok) {
        m |= 1u << (ids[j] / Er);
        if (first) atomicAdd(&s_hist[ids[j]], 1);
      }
    }
    masks[i] = m;
    int cnt = 0;
    for (int r = 0; r < W; ++r) {
      const unsigned b = __ballot_sync(kFull, (m >> r) & 1u);
      if (lane == r) cnt = __popc(b);
    }
    if (lane < W) s_cnt[i][warp][lane] = cnt;
  }
  if (first && __any_sync(kFull, bad) && lane == 0 && status != nullptr)
    atomicOr(status, EP_STATUS_BAD_EXPERT);
  __syncthreads();
  // warp r: exclusive scan of rank r's counts over (batch, warp) in token order
  for (int r = warp; r < W; r += kFWarps) {
    int carry = 0;
    for (int i = 0; i < nb; ++i) {
      const int v = lane < kFWarps ? s_cnt[i][lane][r] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane < kFWarps) s_cnt[i][lane][r] = carry + incl - v;
      carry += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) s_off[r] = carry;  // total of rank r, for now
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int r = 0; r < W; ++r) {
      const int tot = s_off[r];
      if (first) {
        num_tokens_per_rank[r] = tot;
        rank_offset[r] = acc;
      }
      s_off[r] = acc;
      acc += tot;
    }
    if (first) rank_offset[W] = acc;
  }
  __syncthreads();
  // slots: every token's are known here; write those of the tokens this CTA owns
  const unsigned lt = lanemask_lt();
#pragma unroll
  for (int i = 0; i < kFBatches; ++i) {
    if (i >= nb) continue;
    const int t = i * kFThreads + tid;
    const bool mine = t < T && t % G == c;
    for (int r = 0; r < W; ++r) {
      const unsigned in_r = (masks[i] >> r) & 1u;
      const unsigned b = __ballot_sync(kFull, in_r);
      const int v = in_r ? s_off[r] + s_cnt[i][warp][r] + __popc(b & lt) : -1;
      if (mine) {
        slot[(int64_t)t * W + r] = v;
        s_lslot[t / G][r] = v;
      }
    }
  }
  if (first)
    for (int e = tid; e < E; e += kFThreads) num_tokens_per_expert[e] = s_hist[e];
  __syncthreads();

  // ---------------- dispatch of the tokens this CTA owns (warp per token)
  const int n_local = c < T ? (T - 1 - c) / G + 1 : 0;
  uint8_t* buf = smem + (size_t)warp * row_pad;
  bool cap_err = false, timed_out = false;
  uint32_t uses = 0;  // phases of this warp's barrier used so far
  for (int l = warp; l < n_local; l += kFWarps) {
    const int64_t t = c + (int64_t)l * G;
    const int s = lane < W ? s_lslot[l][lane] : -1;
    // the row in its storage and that storage's capacity (per-rank regions:
    // the row inside rank lane's region, from this kernel's own offsets)
    int64_t srow = s, lim = cap;
    if (RT::kRegions && s >= 0) {
      srow = storage_row<RT>(s, s_off[lane]);
      lim = storage_rows<RT>(lane, cap, s_rv);
    }
    const bool keep = s >= 0 && srow < lim;
    cap_err |= __any_sync(kFull, s >= 0 && srow >= lim);
    const unsigned dmask = __ballot_sync(kFull, keep);
    Dests d;
    d.nd = __popc(dmask);
    const int r = nth_set_bit_of_lane(dmask, lane);
    const int row = __shfl_sync(kFull, (int)srow, r & 31);
    d.my_row = r >= 0 ? row : -1;
    d.my_rank = r;
    d.cap_err = false;
    if (tma) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&s_bar[warp], row_bytes);
        bulk_load(buf, x + t * row_bytes, row_bytes, &s_bar[warp]);
      }
      carry_metadata<RT>(topk_idx, topk_w, t, k, d, recv_topk_idx, recv_topk_w, recv_src, lane,
                         &s_rv);
      const bool ok = mbar_wait_bounded(&s_bar[warp], uses & 1u);
      ++uses;
      if (!__all_sync(kFull, ok)) {
        timed_out = true;
        break;
      }
      if (lane < d.nd)
        bulk_store(rows_base<RT>(s_rv, r & 31, recv_x) + (int64_t)d.my_row * row_bytes, buf,
                   row_bytes);
      bulk_commit();
      bulk_wait_read<0>();  // the buffer is reused for the warp's next token
      __syncwarp();
    } else {
      carry_metadata<RT>(topk_idx, topk_w, t, k, d, recv_topk_idx, recv_topk_w, recv_src, lane,
                         &s_rv);
      const uint4* src = reinterpret_cast<const uint4*>(x + t * row_bytes);
      const int n16 = (int)(row_bytes / 16);
      for (int q = 0; q < d.nd; ++q) {
        const int64_t dst_row = __shfl_sync(kFull, d.my_row, q);
        const int dst_rank = __shfl_sync(kFull, r, q);
        uint4* dst = reinterpret_cast<uint4*>(rows_base<RT>(s_rv, dst_rank & 31, recv_x) +
                                              dst_row * row_bytes);
        for (int cidx = lane; cidx < n16; cidx += 32) st_v4(dst + cidx, ld_stream_v4(src + cidx));
      }
    }
  }
  if (tma) {
    // a load still landing in shared memory must finish before the CTA exits
    if (timed_out && lane == 0) (void)mbar_wait_bounded(&s_bar[warp], (uses - 1u) & 1u);
    bulk_wait_all();
  }
  __syncthreads();  // the CTA releases the dependent launch when all its warps are done
  pdl_launch_dependents();
  if (lane == 0 && status != nullptr) {
    if (cap_err) atomicOr(status, EP_STATUS_CAPACITY);
    if (timed_out) atomicOr(status, EP_STATUS_TIMEOUT);
  }
}

template <int KV, bool VEC, class RT>
cudaError_t launch_fused(const void* x, const int32_t* topk_idx, const float* topk_w, int T,
                         int H, int k, int E, int W, int32_t* ne, int32_t* nr, int32_t* off,
                         int32_t* slot, int64_t cap, void* recv_x, int32_t* ridx, float* rw,
                         int32_t* rsrc, int32_t* status, cudaStream_t stream, const RT& rt) {
  const uint32_t row_bytes = (uint32_t)H * 2u;
  const bool tma = row_bytes >= 1024 && row_bytes <= kFMaxTmaRow;
  const uint32_t row_pad = (row_bytes + 127u) & ~127u;
  const size_t smem = (tma ? (size_t)kFWarps * row_pad : 0) + sizeof(int32_t) * (size_t)E;
  static bool attr_set[128];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 128 && !attr_set[dev]) {
    const int most = (int)((size_t)kFWarps * kFMaxTmaRow + sizeof(int32_t) * 8192);
    cudaError_t e = cudaFuncSetAttribute(dispatch_fused_kernel<KV, VEC, RT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int grid = device_sm_count();
  if (grid > T) grid = T;
  const int at_least = (T + kFMaxLocal - 1) / kFMaxLocal;  // a CTA owns at most kFMaxLocal tokens
  if (grid < at_least) grid = at_least;
  if (grid < 1) grid = 1;
  return launch_pdl(dispatch_fused_kernel<KV, VEC, RT>, dim3(grid), dim3(kFThreads), smem, stream,
                    static_cast<const uint8_t*>(x), topk_idx, topk_w, T, H, k, E, W, E / W, ne, nr,
                    off, slot, cap, static_cast<uint8_t*>(recv_x), ridx, rw, rsrc, status, rt);
}

}  // namespace

int64_t fused_max_tokens() { return kFusedMaxT; }

namespace {
template <class RT>
cudaError_t launch_fused_rt(const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T,
                            int H, int k, int E, int W, int32_t* ne, int32_t* nr, int32_t* off,
                            int32_t* slot, int64_t cap, void* recv_x, int32_t* ridx, float* rw,
                            int32_t* rsrc, int32_t* status, cudaStream_t stream, const RT& rt) {
  const int Ti = (int)T;
  const bool vec = (reinterpret_cast<uintptr_t>(topk_idx) & 15) == 0;
  if (k == 8 && vec)
    return launch_fused<8, true>(x, topk_idx, topk_w, Ti, H, k, E, W, ne, nr, off, slot, cap,
                                 recv_x, ridx, rw, rsrc, status, stream, rt);
  if (k == 4 && vec)
    return launch_fused<4, true>(x, topk_idx, topk_w, Ti, H, k, E, W, ne, nr, off, slot, cap,
                                 recv_x, ridx, rw, rsrc, status, stream, rt);
  return launch_fused<16, false>(x, topk_idx, topk_w, Ti, H, k, E, W, ne, nr, off, slot, cap,
                                 recv_x, ridx, rw, rsrc, status, stream, rt);
}
}  // namespace

cudaError_t launch_dispatch_fused(const void* x, const int32_t* topk_idx, const float* topk_w,
                                  int64_t T, int H, int k, int E, int W, int32_t* ne, int32_t* nr,
                                  int32_t* off, int32_t* slot, int64_t cap, void* recv_x,
                                  int32_t* ridx, float* rw, int32_t* rsrc, int32_t* status,
                                  cudaStream_t stream) {
  return launch_fused_rt(x, topk_idx, topk_w, T, H, k, E, W, ne, nr, off, slot, cap, recv_x, ridx,
                         rw, rsrc, status, stream, OneBuffer{});
}

cudaError_t launch_dispatch_fused_regions(const void* x, const int32_t* topk_idx,
                                          const float* topk_w, int64_t T, int H, int k, int E,
                                          int W, int32_t* ne, int32_t* nr, int32_t* off,
                                          int32_t* slot, const RankRegions& regions,
                                          int32_t* status, cudaStream_t stream) {
  return launch_fused_rt(x, topk_idx, topk_w, T, H, k, E, W, ne, nr, off, slot, /*cap=*/0,
                         nullptr, nullptr, nullptr, nullptr, status, stream, regions);
}

}  // namespace ep
