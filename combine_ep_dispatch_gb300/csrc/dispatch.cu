// Dispatch of bf16 rows: one warp per token reads the token's row once and
// writes it to the receive row of every destination rank, and carries the
// top-k ids, weights and the source index along.  Rows of 1 KB and more go
// through the bulk-copy (TMA) engine, smaller ones through 16-byte loads and
// stores.  (FP8 rows: dispatch_fp8.cu.)
#include "dispatch_common.cuh"

namespace ep {
namespace {

constexpr int kDThreads = 256;

// bf16 payload: lane l moves 16-byte chunks l, l+32, ... of the row; U chunks
// are loaded before the stores of a round so that each lane keeps U loads in
// flight.  The row is read once whatever the number of destinations.
template <int U, class RT>
__global__ void __launch_bounds__(kDThreads)
    dispatch_bf16_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ topk_idx,
                         const float* __restrict__ topk_w, int64_t T, int n16, int k, int W,
                         const int32_t* __restrict__ slot, int64_t cap, uint4* __restrict__ recv_x,
                         int32_t* __restrict__ recv_topk_idx, float* __restrict__ recv_topk_w,
                         int32_t* __restrict__ recv_src, int32_t* __restrict__ status, RT rt) {
  __shared__ typename RT::View s_rv;
  load_region_view(rt, W, s_rv);
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int32_t first_row = region_first_row(rt, W, lane);
  const int64_t gwarp = ((int64_t)blockIdx.x * kDThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDThreads) >> 5;
  bool cap_err = false;
  for (int64_t t = gwarp; t < T; t += nwarps) {
    const Dests d = token_dests<RT>(slot, t, W, cap, lane, &s_rv, first_row);
    cap_err |= d.cap_err;
    carry_metadata<RT>(topk_idx, topk_w, t, k, d, recv_topk_idx, recv_topk_w, recv_src, lane,
                       &s_rv);
    const uint4* src = x + t * n16;
    for (int c0 = 0; c0 < n16; c0 += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < n16) v[u] = ld_stream_v4(src + c);
      }
      for (int dg = 0; dg < d.nd; dg += 8) {
        int rows[8], ranks[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          rows[q] = __shfl_sync(kFull, d.my_row, (dg + q) & 31);
          ranks[q] = RT::kRegions ? __shfl_sync(kFull, d.my_rank, (dg + q) & 31) : 0;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (dg + q < d.nd) {
            uint4* const base = reinterpret_cast<uint4*>(
                rows_base<RT>(s_rv, ranks[q] & 31, reinterpret_cast<uint8_t*>(recv_x)));
            uint4* dst = base + (int64_t)rows[q] * n16;
#pragma unroll
            for (int u = 0; u < U; ++u) {
              const int c = c0 + u * 32 + lane;
              if (c < n16) st_v4(dst + c, v[u]);
            }
          }
        }
      }
    }
  }
  __syncthreads();  // the CTA releases the dependent launch when all its warps are done
  pdl_launch_dependents();
  if (cap_err && lane == 0 && status != nullptr) atomicOr(status, EP_STATUS_CAPACITY);
}

// bf16 payload through the bulk-copy (TMA) engine.  Each warp runs its own
// pipeline over its tokens with kTmaStages private row buffers in shared
// memory: lane 0 brings the token's row in with one bulk copy (global ->
// shared) and, once it has landed, sends it out with one bulk copy (shared ->
// global) per destination row; a buffer is refilled with a later token once
// the copies out of it have finished reading it.  A row copy is then one
// instruction instead of H/256 warp-wide 16-byte stores, which keeps the
// load/store pipe free; the other lanes fetch the next token's slots early and
// carry the metadata.
constexpr int kTmaStages = 3;            // row buffers per warp
// The token loop reads the next token's stage before it refills the previous
// one: three stages at least, so that the two are different.
static_assert(kTmaStages >= 3, "the bulk-copy dispatch needs three row buffers per warp");
constexpr int kTmaBarBytes = 1024;       // barrier area ahead of the row buffers
constexpr int kTmaSmemBudget = 100000;   // row buffers per CTA
constexpr int kTmaMaxWarps = 8;
// The received rows are stored with an L2 evict_last policy: it keeps the
// rows just written in L2 for their consumer (the expert GEMM reads them next)
// and moves part of their write-back out of this kernel.  Measured on GB300 it
// shortens the layout + dispatch + combine step by 1.3 to 2.5 us at T=4096
// (H=7168) and T=8192 (H=4096); evict_first changed nothing.
constexpr int kL2EvictLast = 2;
constexpr int kTmaCtasPerSm = 2;
constexpr uint32_t kTmaMinRowBytes = 1024;  // smaller rows: 16-byte stores from registers

// A plain load: with a Finalize the kernel also writes the slot table (each
// entry by the warp that read it, after reading it).
__device__ __forceinline__ int load_slot(const int32_t* slot, int64_t t, int W, int lane,
                                         int64_t T) {
  return (t < T && lane < W) ? slot[t * W + lane] : -1;
}

template <class RT>
__global__ void __launch_bounds__(kTmaMaxWarps * 32, kTmaCtasPerSm)
    dispatch_bf16_tma_kernel(const uint8_t* __restrict__ x, const int32_t* __restrict__ topk_idx,
                             const float* __restrict__ topk_w, int64_t T, uint32_t row_bytes,
                             uint32_t stage_bytes, int k, int W, int32_t* slot,
                             int64_t cap, uint8_t* __restrict__ recv_x,
                             int32_t* __restrict__ recv_topk_idx, float* __restrict__ recv_topk_w,
                             int32_t* __restrict__ recv_src, int32_t* __restrict__ status,
                             int x_early, Finalize fin, RT rt) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta_warps = blockDim.x >> 5;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem) + warp * kTmaStages;
  uint8_t* buf = smem + kTmaBarBytes + (size_t)warp * kTmaStages * stage_bytes;
  if (lane == 0) {
    for (int s = 0; s < kTmaStages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncwarp();

  const int64_t gw = (int64_t)blockIdx.x * cta_warps + warp;
  const int64_t NW = (int64_t)gridDim.x * cta_warps;
  const int64_t n = gw < T ? (T - 1 - gw) / NW + 1 : 0;  // tokens gw, gw+NW, ...
  int64_t issued = 0;                                      // tokens whose row load was issued
  // The first rows depend on x only.  With x_early (set only when this launch
  // directly follows the layout kernels, whose own wait already covered x's
  // producer) they are loaded while the layout still runs; otherwise after
  // the wait, like every other access.
  auto first_loads = [&](int64_t upto) {
    if (lane == 0) {
      for (; issued < n && issued < upto; ++issued) {
        mbar_arrive_expect_tx(&full[issued], row_bytes);
        bulk_load(buf + issued * stage_bytes, x + (gw + issued * NW) * row_bytes, row_bytes,
                  &full[issued]);
      }
    }
  };
  __shared__ typename RT::View s_rv;  // per-rank regions: the table
  load_region_view(rt, W, s_rv);
  if (x_early) first_loads(kTmaStages);
  pdl_wait();
  first_loads(kTmaStages);

  const bool fin_mode = fin.chunk_rank != nullptr;  // uniform over the grid
  __shared__ int32_t s_tot[32], s_off[33];
  int32_t* const s_base =
      reinterpret_cast<int32_t*>(smem + kTmaBarBytes + (size_t)cta_warps * kTmaStages * stage_bytes);
  if (fin_mode) build_chunk_base(fin, W, s_base, s_tot, s_off);
  // each region's first global row: rank_offset, or (finishing the layout,
  // which writes rank_offset during this kernel) the CTA's own scan of it
  const int32_t first_row = fin_mode ? (RT::kRegions && lane < W ? s_off[lane] : 0)
                                     : region_first_row(rt, W, lane);
  // the receive row of (tt, lane), written back to the slot table (the warp
  // owns token tt's entries)
  auto finalize = [&](int s_loc, int64_t tt) -> int {
    if (!fin_mode || lane >= W || tt >= T) return s_loc;
    const int s_fin = final_slot(s_loc, tt, lane, W, fin.shift, s_base, s_off);
    slot[tt * W + lane] = s_fin;
    return s_fin;
  };

  const bool meta_lanes = 2 * k + 1 <= 32;
  bool cap_err = false, timed_out = false;
  // Token order.  Stage q % kTmaStages holds the warp's q-th token, s_ring
  // records which (-1: none).  The first kTmaStages tokens of warp gw are gw,
  // gw + NW, gw + 2 NW (loaded early).  After that, with a claim counter (the
  // dispatch that finishes the layout: the count kernel zeroed it) a warp
  // takes the next unclaimed token of [kTmaStages NW, T) whenever it refills a
  // stage, so warps that drew tokens with few destinations take more of them
  // and all finish together; without one it keeps the fixed stride.
  __shared__ int64_t s_ring[kTmaMaxWarps][kTmaStages];
  unsigned long long* const claim = fin.claim;
  if (lane == 0)
    for (int q = 0; q < kTmaStages; ++q) s_ring[warp][q] = q < n ? gw + q * NW : -1;
  __syncwarp();
  bool more = true;  // later tokens may still exist
  int64_t t = s_ring[warp][0];
  int s_cur = t >= 0 ? finalize(load_slot(slot, t, W, lane, T), t) : -1;
  int64_t j = 0;
  for (; t >= 0; ++j) {
    const int st = (int)(j % kTmaStages);
    const uint32_t parity = (uint32_t)((j / kTmaStages) & 1);
    // one metadata word per lane: k ids, k weights, the source index
    int32_t mv = 0;
    if (meta_lanes && lane <= 2 * k) {
      if (lane < k)
        mv = __ldg(topk_idx + t * k + lane);
      else if (lane < 2 * k)
        mv = __float_as_int(__ldg(topk_w + t * k + (lane - k)));
      else
        mv = (int32_t)t;
    }
    const int64_t t_next = s_ring[warp][(j + 1) % kTmaStages];
    const int s_next = t_next >= 0 ? load_slot(slot, t_next, W, lane, T) : -1;
    int64_t srow = s_cur, lim = cap;  // the row in its storage and that storage's capacity
    if (RT::kRegions && s_cur >= 0) {
      srow = storage_row<RT>(s_cur, first_row);
      lim = storage_rows<RT>(lane, cap, s_rv);
    }
    const bool keep = s_cur >= 0 && srow < lim;
    cap_err |= __any_sync(kFull, s_cur >= 0 && srow >= lim);
    const unsigned dmask = __ballot_sync(kFull, keep);
    const int nd = __popc(dmask);
    const int r = nth_set_bit_of_lane(dmask, lane);
    const int my_row = __shfl_sync(kFull, (int)srow, r & 31);

    // every lane observes the row's arrival, lane q sends it to destination q
    const bool ok = mbar_wait_bounded(&full[st], parity);
    if (!__all_sync(kFull, ok)) {
      timed_out = true;
      break;
    }
    if (lane < nd) {
      uint8_t* const base = rows_base<RT>(s_rv, r, recv_x);
      bulk_store_hint(base + (int64_t)my_row * row_bytes, buf + st * stage_bytes, row_bytes,
                      make_l2_policy<kL2EvictLast>());
    }
    bulk_commit();
    if (meta_lanes) {
      for (int q = 0; q < nd; ++q) {
        const int64_t row = __shfl_sync(kFull, my_row, q);
        int32_t* ridx = recv_topk_idx;
        float* rw = recv_topk_w;
        int32_t* rsrc = recv_src;
        if constexpr (RT::kRegions) {
          const int rq = __shfl_sync(kFull, r, q);
          ridx = s_rv.topk_idx[rq];
          rw = s_rv.topk_w[rq];
          rsrc = s_rv.src[rq];
        }
        if (lane < k) {
          if (ridx) ridx[row * k + lane] = mv;
        } else if (lane < 2 * k) {
          if (rw) rw[row * k + (lane - k)] = __int_as_float(mv);
        } else if (lane == 2 * k) {
          if (rsrc) rsrc[row] = mv;
        }
      }
    } else {
      Dests d;
      d.nd = nd;
      d.my_row = r >= 0 ? my_row : -1;
      d.my_rank = r;
      d.cap_err = false;
      carry_metadata<RT>(topk_idx, topk_w, t, k, d, recv_topk_idx, recv_topk_w, recv_src, lane,
                         &s_rv);
    }
    // refill the previous token's stage with the warp's (j + kTmaStages - 1)-th
    // token, once the copies out of it (issued by several lanes) have read it
    if (j >= 1) {
      const int sp = (int)((j - 1) % kTmaStages);
      int64_t tn = -1;
      if (more) {
        if (claim != nullptr) {
          unsigned long long c = 0;
          if (lane == 0) c = atomicAdd(claim, 1ull);
          tn = (int64_t)kTmaStages * NW + (int64_t)__shfl_sync(kFull, c, 0);
        } else {
          tn = gw + (j + kTmaStages - 1) * NW;
        }
        if (tn >= T) {
          tn = -1;
          more = false;
        }
      }
      if (tn >= 0) {
        bulk_wait_read<1>();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[sp], row_bytes);
          bulk_load(buf + sp * stage_bytes, x + tn * row_bytes, row_bytes, &full[sp]);
          ++issued;
        }
      }
      if (lane == 0) s_ring[warp][sp] = tn;
      __syncwarp();
    }
    issued = __shfl_sync(kFull, issued, 0);
    t = t_next;
    s_cur = t_next >= 0 ? finalize(s_next, t_next) : -1;
  }
  if (fin_mode) finish_expert_totals(fin);
  if (lane == 0) {
    // never leave with a bulk copy still using this CTA's shared memory
    for (int64_t q = j; q < issued; ++q)
      (void)mbar_wait_bounded(&full[q % kTmaStages], (uint32_t)((q / kTmaStages) & 1));
  }
  bulk_wait_all();
  // The dependent launch is released once every warp of the CTA is done.
  // Released by each warp as it finished, it let the next grid launch while
  // other warps still sent rows: measured on GB300, layout + dispatch +
  // combine at T=8192, H=4096 (top-8 of 128 experts, 8 ranks) took 157 us
  // instead of 140 us (at H=7168 no change).
  __syncthreads();
  pdl_launch_dependents();
  if (lane == 0 && status != nullptr) {
    if (cap_err) atomicOr(status, EP_STATUS_CAPACITY);
    if (timed_out) atomicOr(status, EP_STATUS_TIMEOUT);
  }
}

}  // namespace

template <class RT>
cudaError_t launch_dispatch_fp8(const void* x, const int32_t* topk_idx, const float* topk_w,
                                int64_t T, int H, int k, int W, const int32_t* slot,
                                int64_t capacity_rows, void* recv_x, float* recv_scale,
                                int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                                int32_t* status, cudaStream_t stream, int x_early,
                                const Finalize& fin, const RT& rt);
extern template cudaError_t launch_dispatch_fp8<OneBuffer>(
    const void*, const int32_t*, const float*, int64_t, int, int, int, const int32_t*, int64_t,
    void*, float*, int32_t*, float*, int32_t*, int32_t*, cudaStream_t, int, const Finalize&,
    const OneBuffer&);
extern template cudaError_t launch_dispatch_fp8<RankRegions>(
    const void*, const int32_t*, const float*, int64_t, int, int, int, const int32_t*, int64_t,
    void*, float*, int32_t*, float*, int32_t*, int32_t*, cudaStream_t, int, const Finalize&,
    const RankRegions&);

namespace {

// Launch shape of the bulk-copy kernel for rows of H bf16 values; false when
// the register kernel serves this row size.
struct TmaShape {
  uint32_t row_bytes, stage_bytes;
  int cta_warps;
};
bool tma_shape(int H, TmaShape* sh) {
  sh->row_bytes = (uint32_t)H * 2u;
  sh->stage_bytes = (sh->row_bytes + 127u) & ~127u;
  const int fit = (int)(kTmaSmemBudget / ((size_t)kTmaStages * sh->stage_bytes));
  sh->cta_warps = fit < kTmaMaxWarps ? fit : kTmaMaxWarps;
  return sh->row_bytes >= kTmaMinRowBytes && fit >= 1;
}

template <class RT>
cudaError_t launch_tma(const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T,
                       int k, int W, int32_t* slot, int64_t capacity_rows, void* recv_x,
                       int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                       int32_t* status, cudaStream_t stream, int x_early, const TmaShape& sh,
                       const Finalize& fin, const RT& rt) {
  size_t smem = kTmaBarBytes + (size_t)sh.cta_warps * kTmaStages * sh.stage_bytes;
  if (fin.chunk_rank != nullptr) smem += ((size_t)(fin.C * W) * sizeof(int32_t) + 15) & ~size_t(15);
  static bool attr_set[128];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 128 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(dispatch_bf16_tma_kernel<RT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTmaBarBytes + kTmaSmemBudget + kFinMaxBytes);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t want = (T + sh.cta_warps - 1) / sh.cta_warps;
  const int64_t sms = (int64_t)device_sm_count() * kTmaCtasPerSm;
  const int grid = (int)(want < sms ? want : sms);
  return launch_pdl(dispatch_bf16_tma_kernel<RT>, dim3(grid < 1 ? 1 : grid),
                    dim3(sh.cta_warps * 32), smem, stream, static_cast<const uint8_t*>(x), topk_idx,
                    topk_w, T, sh.row_bytes, sh.stage_bytes, k, W, slot, capacity_rows,
                    static_cast<uint8_t*>(recv_x), recv_topk_idx, recv_topk_w, recv_src, status,
                    x_early, fin, rt);
}

// The dispatch of a final slot table into receive storage RT (one buffer, or
// per-rank regions).
template <class RT>
cudaError_t launch_dispatch_rt(const void* x, const int32_t* topk_idx, const float* topk_w,
                               int64_t T, int H, int k, int W, const int32_t* slot,
                               int64_t capacity_rows, int quant, void* recv_x, float* recv_scale,
                               int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                               int32_t* status, cudaStream_t stream, int x_early, const RT& rt,
                               unsigned long long* claim = nullptr) {
  if (T == 0) return cudaSuccess;
  const uint4* x4 = static_cast<const uint4*>(x);
  Finalize none{};
  if (quant == EP_QUANT_BF16) {
    TmaShape sh;
    if (tma_shape(H, &sh)) {
      // the kernel writes the slot table only with a Finalize; it takes tokens
      // from `claim` (zeroed by the layout kernel before it) when given one
      Finalize claims{};
      claims.claim = claim;
      return launch_tma(x, topk_idx, topk_w, T, k, W, const_cast<int32_t*>(slot), capacity_rows,
                        recv_x, recv_topk_idx, recv_topk_w, recv_src, status, stream, x_early,
                        sh, claims, rt);
    }
    const int n16 = H / 8;
    if (n16 % (32 * 7) == 0) {
      auto kern = dispatch_bf16_kernel<7, RT>;
      return launch_pdl(kern, dim3(grid_for(kern, T, kDThreads)), dim3(kDThreads), 0, stream, x4,
                        topk_idx, topk_w, T, n16, k, W, slot, capacity_rows,
                        static_cast<uint4*>(recv_x), recv_topk_idx, recv_topk_w, recv_src, status,
                        rt);
    }
    auto kern = dispatch_bf16_kernel<8, RT>;
    return launch_pdl(kern, dim3(grid_for(kern, T, kDThreads)), dim3(kDThreads), 0, stream, x4,
                      topk_idx, topk_w, T, n16, k, W, slot, capacity_rows,
                      static_cast<uint4*>(recv_x), recv_topk_idx, recv_topk_w, recv_src, status, rt);
  }
  return launch_dispatch_fp8<RT>(x, topk_idx, topk_w, T, H, k, W, slot, capacity_rows, recv_x,
                                 recv_scale, recv_topk_idx, recv_topk_w, recv_src, status, stream,
                                 x_early, none, rt);
}

}  // namespace

cudaError_t launch_dispatch(const void* x, const int32_t* topk_idx, const float* topk_w,
                            int64_t T, int H, int k, int W, const int32_t* slot,
                            int64_t capacity_rows, int quant, void* recv_x, float* recv_scale,
                            int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                            int32_t* status, cudaStream_t stream, int x_early,
                            unsigned long long* claim) {
  return launch_dispatch_rt(x, topk_idx, topk_w, T, H, k, W, slot, capacity_rows, quant, recv_x,
                            recv_scale, recv_topk_idx, recv_topk_w, recv_src, status, stream,
                            x_early, OneBuffer{}, claim);
}

cudaError_t launch_dispatch_regions(const void* x, const int32_t* topk_idx, const float* topk_w,
                                    int64_t T, int H, int k, int W, const int32_t* slot,
                                    int quant, const RankRegions& regions, int32_t* status,
                                    cudaStream_t stream) {
  return launch_dispatch_rt(x, topk_idx, topk_w, T, H, k, W, slot, /*capacity_rows=*/0, quant,
                            nullptr, nullptr, nullptr, nullptr, nullptr, status, stream,
                            /*x_early=*/0, regions);
}

namespace {
// The dispatch finishes the layout (count kernel + dispatch, no scan kernel):
// FP8 rows, or bf16 rows that take the bulk-copy kernel, beyond the one-CTA
// layout's batches, with a chunk table that fits kFinMaxBytes.
bool finalize_applies(int64_t T, int H, int W, int quant, TmaShape* sh) {
  if (T <= kLayoutSingleMaxT || layout_num_chunks(T) * W * (int64_t)sizeof(int32_t) > kFinMaxBytes)
    return false;
  if (quant == EP_QUANT_FP8_E4M3_B128) return true;
  return quant == EP_QUANT_BF16 && tma_shape(H, sh);
}
}  // namespace

// Small bf16 batches: the one-launch dispatch (every CTA recomputes the
// layout) is the fastest step up to this many tokens (GB300, decode shapes).
constexpr int64_t kPreferFusedMaxT = 512;
bool prefer_fused(int64_t T, int H, int k, int quant) {
  return quant == EP_QUANT_BF16 && T > 0 && T <= kPreferFusedMaxT && T <= fused_max_tokens() &&
         k <= 16 && H % 8 == 0;
}

int dispatch_with_layout_launches(int64_t T, int H, int k, int W, int quant) {
  TmaShape sh;
  if (prefer_fused(T, H, k, quant)) return 1;               // layout + dispatch in one kernel
  if (finalize_applies(T, H, W, quant, &sh)) return 2;      // count, dispatch
  const int layout = T <= kLayoutSingleMaxT ? 1 : 2;       // one CTA, or count + scan
  return layout + (T > 0 ? 1 : 0);
}

cudaError_t launch_dispatch_with_layout(const void* x, const int32_t* topk_idx, const float* topk_w,
                                        int64_t T, int H, int k, int E, int W,
                                        int32_t* num_tokens_per_expert,
                                        int32_t* num_tokens_per_rank, int32_t* rank_offset,
                                        int32_t* slot, void* workspace, int64_t capacity_rows,
                                        int quant, void* recv_x, float* recv_scale,
                                        int32_t* recv_topk_idx, float* recv_topk_w,
                                        int32_t* recv_src, int32_t* status, cudaStream_t stream) {
  if (prefer_fused(T, H, k, quant))
    return launch_dispatch_fused(x, topk_idx, topk_w, T, H, k, E, W, num_tokens_per_expert,
                                 num_tokens_per_rank, rank_offset, slot, capacity_rows, recv_x,
                                 recv_topk_idx, recv_topk_w, recv_src, status, stream);
  TmaShape sh;
  if (finalize_applies(T, H, W, quant, &sh)) {
    // count kernel (positions inside chunks) -> dispatch that finishes the layout
    LayoutChunks ch;
    cudaError_t e = launch_layout_count(topk_idx, T, k, E, W, workspace, slot, status, stream, &ch);
    if (e != cudaSuccess) return e;
    Finalize fin{ch.chunk_rank, ch.chunk_exp, ch.C, ch.shift, E, num_tokens_per_expert,
                 num_tokens_per_rank, rank_offset, ch.claim};
    if (quant == EP_QUANT_FP8_E4M3_B128)
      return launch_dispatch_fp8(x, topk_idx, topk_w, T, H, k, W, slot, capacity_rows, recv_x,
                                 recv_scale, recv_topk_idx, recv_topk_w, recv_src, status, stream,
                                 /*x_early=*/1, fin, OneBuffer{});
    return launch_tma(x, topk_idx, topk_w, T, k, W, slot, capacity_rows, recv_x, recv_topk_idx,
                      recv_topk_w, recv_src, status, stream, /*x_early=*/1, sh, fin, OneBuffer{});
  }
  // the whole layout, then the dispatch, which loads its first rows of x while
  // the layout kernels run
  cudaError_t e = launch_layout(topk_idx, T, k, E, W, num_tokens_per_expert, num_tokens_per_rank,
                                rank_offset, slot, workspace, status, stream);
  if (e != cudaSuccess) return e;
  return launch_dispatch(x, topk_idx, topk_w, T, H, k, W, slot, capacity_rows, quant, recv_x,
                         recv_scale, recv_topk_idx, recv_topk_w, recv_src, status, stream,
                         /*x_early=*/1);
}

// The same into per-rank regions, by the same paths: the one-launch kernel
// for small bf16 batches, count kernel + a dispatch that finishes the layout
// where that applies, else the whole layout and then the dispatch.
cudaError_t launch_dispatch_regions_with_layout(
    const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T, int H, int k, int E,
    int W, int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank, int32_t* rank_offset,
    int32_t* slot, void* workspace, int quant, const RankRegions& regions, int32_t* status,
    cudaStream_t stream) {
  if (prefer_fused(T, H, k, quant))
    return launch_dispatch_fused_regions(x, topk_idx, topk_w, T, H, k, E, W, num_tokens_per_expert,
                                         num_tokens_per_rank, rank_offset, slot, regions, status,
                                         stream);
  TmaShape sh;
  if (finalize_applies(T, H, W, quant, &sh)) {
    LayoutChunks ch;
    cudaError_t e = launch_layout_count(topk_idx, T, k, E, W, workspace, slot, status, stream, &ch);
    if (e != cudaSuccess) return e;
    Finalize fin{ch.chunk_rank, ch.chunk_exp, ch.C, ch.shift, E, num_tokens_per_expert,
                 num_tokens_per_rank, rank_offset, ch.claim};
    if (quant == EP_QUANT_FP8_E4M3_B128)
      return launch_dispatch_fp8(x, topk_idx, topk_w, T, H, k, W, slot, /*capacity_rows=*/0,
                                 nullptr, nullptr, nullptr, nullptr, nullptr, status, stream,
                                 /*x_early=*/1, fin, regions);
    return launch_tma(x, topk_idx, topk_w, T, k, W, slot, /*capacity_rows=*/0, nullptr, nullptr,
                      nullptr, nullptr, status, stream, /*x_early=*/1, sh, fin, regions);
  }
  cudaError_t e = launch_layout(topk_idx, T, k, E, W, num_tokens_per_expert, num_tokens_per_rank,
                                rank_offset, slot, workspace, status, stream);
  if (e != cudaSuccess) return e;
  return launch_dispatch_rt(x, topk_idx, topk_w, T, H, k, W, slot, /*capacity_rows=*/0, quant,
                            nullptr, nullptr, nullptr, nullptr, nullptr, status, stream,
                            /*x_early=*/1, regions);
}

}  // namespace ep
