// Device helpers shared by the dispatch kernels (bf16 and FP8 payloads).
#pragma once

#include "ep_device.cuh"

namespace ep {

// Where the receive rows live.  OneBuffer: one allocation for all ranks, rank
// r's rows are the global rows [rank_offset[r], rank_offset[r+1]) of it (the
// layout's slot is the row).  RankRegions: one allocation per rank
// (ep_dispatch_regions, ep_combine_regions), passed as a table of base
// pointers: the row of (t, r) is slot[t][r] - rank_offset[r] of rank r's
// region, and each region has its own capacity.  Kernels copy the table into
// shared memory before their dependency wait (it comes with the launch), and
// lane r of every warp loads rank_offset[r], the first global row of rank r's
// region, after it (rank_offset comes from the layout): the lanes of a warp
// stand for the ranks whenever a slot row is read.
struct OneBuffer {
  static constexpr bool kRegions = false;
  struct View {
    int32_t unused;
  };
};

struct RankRegions {
  static constexpr bool kRegions = true;
  uint8_t* x[kMaxRanks];          // rank r's receive rows (bf16 rows or e4m3 codes)
  float* scale[kMaxRanks];        // FP8 block scales of those rows, or null
  int32_t* topk_idx[kMaxRanks];   // metadata of those rows, each may be null
  float* topk_w[kMaxRanks];
  int32_t* src[kMaxRanks];
  int64_t rows[kMaxRanks];        // capacity of each region
  const int32_t* rank_offset;     // [W + 1] from the layout (device memory)
  struct View {
    uint8_t* x[kMaxRanks];
    float* scale[kMaxRanks];
    int32_t* topk_idx[kMaxRanks];
    float* topk_w[kMaxRanks];
    int32_t* src[kMaxRanks];
    int64_t rows[kMaxRanks];
  };
};

// Fills the shared view of a region table (the pointers and capacities that
// come with the launch); every thread of the CTA calls it, before the
// kernel's dependency wait.
template <class RT>
__device__ __forceinline__ void load_region_view(const RT& rt, int W, typename RT::View& v) {
  if constexpr (RT::kRegions) {
    for (int r = threadIdx.x; r < W; r += blockDim.x) {
      v.x[r] = rt.x[r];
      v.scale[r] = rt.scale[r];
      v.topk_idx[r] = rt.topk_idx[r];
      v.topk_w[r] = rt.topk_w[r];
      v.src[r] = rt.src[r];
      v.rows[r] = rt.rows[r];
    }
    __syncthreads();
  }
}

// First global row of rank `lane`'s region (per-rank regions, lane < W); read
// after the dependency wait.  0 otherwise.
template <class RT>
__device__ __forceinline__ int32_t region_first_row(const RT& rt, int W, int lane) {
  if constexpr (RT::kRegions)
    return lane < W ? rt.rank_offset[lane] : 0;
  else
    return 0;
}

// Row of the slot entry s (>= 0) of rank r inside r's storage (first_row: the
// region's first global row, region_first_row of lane r), and that storage's
// capacity: the global row and `cap` for one buffer, the row inside the region
// and the region's capacity for per-rank regions.
template <class RT>
__device__ __forceinline__ int64_t storage_row(int s, int32_t first_row) {
  if constexpr (RT::kRegions)
    return (int64_t)s - first_row;
  else
    return s;
}
template <class RT>
__device__ __forceinline__ int64_t storage_rows(int r, int64_t cap, const typename RT::View& v) {
  if constexpr (RT::kRegions)
    return v.rows[r];
  else
    return cap;
}

// Base of rank r's receive rows: the one buffer, or rank r's region.
template <class RT>
__device__ __forceinline__ uint8_t* rows_base(const typename RT::View& v, int r, uint8_t* one) {
  if constexpr (RT::kRegions)
    return v.x[r];
  else
    return one;
}

// Destinations of token t in ascending rank order: lane i < nd holds the i-th
// destination's row (in its storage, see storage_row) and rank.  Rows at or
// beyond their storage's capacity are dropped and reported.  (The cached
// (token, rank) -> row map of "perf(ep): optimize IntraNode dispatch kernel
// for MI350X", Technical Details 1, is `slot`.)
struct Dests {
  int nd;
  int my_row;
  int my_rank;
  bool cap_err;
};

template <class RT = OneBuffer>
__device__ __forceinline__ Dests token_dests(const int32_t* __restrict__ slot, int64_t t, int W,
                                             int64_t cap, int lane,
                                             const typename RT::View* v = nullptr,
                                             int32_t first_row = 0) {
  int s = -1;
  if (lane < W) s = __ldg(slot + t * W + lane);
  int64_t row = s, lim = cap;
  if constexpr (RT::kRegions) {
    if (s >= 0) {
      row = storage_row<RT>(s, first_row);
      lim = storage_rows<RT>(lane, cap, *v);
    }
  }
  const bool keep = s >= 0 && row < lim;
  const bool over = s >= 0 && row >= lim;
  const unsigned dmask = __ballot_sync(kFull, keep);
  const int r = nth_set_bit_of_lane(dmask, lane);
  const int rr = __shfl_sync(kFull, (int)row, r & 31);
  Dests d;
  d.nd = __popc(dmask);
  d.my_row = r >= 0 ? rr : -1;
  d.my_rank = r;
  d.cap_err = __any_sync(kFull, over);
  return d;
}

// One 32-bit word, whatever its type.
__device__ __forceinline__ void st_b32(void* p, uint32_t v) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Metadata of one token for all its destinations: per destination row, k ids,
// k weights and the source index (2k+1 words), written by the whole warp at
// once ("perf(ep): optimize IntraNode dispatch kernel for MI350X", Technical
// Details 4).  Lane j takes word j of the token (id j, weight j - k, or the
// source index at j = 2k), reads it once, and stores it to every destination
// row with one multiply-add for the address: no division, no per-destination
// reloads.  With per-rank regions the destination's rank picks the array.
template <class RT = OneBuffer>
__device__ __forceinline__ void carry_metadata(const int32_t* __restrict__ topk_idx,
                                               const float* __restrict__ topk_w, int64_t t, int k,
                                               const Dests& d, int32_t* __restrict__ recv_topk_idx,
                                               float* __restrict__ recv_topk_w,
                                               int32_t* __restrict__ recv_src, int lane,
                                               const typename RT::View* v = nullptr) {
  const int per = 2 * k + 1;
  for (int w0 = 0; w0 < per; w0 += 32) {
    const int j = w0 + lane;
    int kind = -1;  // 0: id, 1: weight, 2: source index
    uint32_t* col = nullptr;  // the word's address in receive row 0
    uint32_t stride = 1, val = 0;
    if (j < k) {
      kind = 0;
      stride = (uint32_t)k;
      val = (uint32_t)__ldg(topk_idx + t * k + j);
      if (recv_topk_idx != nullptr) col = reinterpret_cast<uint32_t*>(recv_topk_idx) + j;
    } else if (j < 2 * k) {
      kind = 1;
      stride = (uint32_t)k;
      val = __float_as_uint(__ldg(topk_w + t * k + (j - k)));
      if (recv_topk_w != nullptr) col = reinterpret_cast<uint32_t*>(recv_topk_w) + (j - k);
    } else if (j == 2 * k) {
      kind = 2;
      val = (uint32_t)t;
      if (recv_src != nullptr) col = reinterpret_cast<uint32_t*>(recv_src);
    }
    for (int qq = 0; qq < d.nd; ++qq) {
      const uint32_t row = (uint32_t)__shfl_sync(kFull, d.my_row, qq);
      if constexpr (RT::kRegions) {
        const int r = __shfl_sync(kFull, d.my_rank, qq);
        uint32_t* base = nullptr;
        if (kind == 0 && v->topk_idx[r] != nullptr)
          base = reinterpret_cast<uint32_t*>(v->topk_idx[r]) + j;
        else if (kind == 1 && v->topk_w[r] != nullptr)
          base = reinterpret_cast<uint32_t*>(v->topk_w[r]) + (j - k);
        else if (kind == 2 && v->src[r] != nullptr)
          base = reinterpret_cast<uint32_t*>(v->src[r]);
        if (base != nullptr) st_b32(base + (uint64_t)row * stride, val);
      } else {
        if (col != nullptr) st_b32(col + (uint64_t)row * stride, val);
      }
    }
  }
}

// Finishing the layout inside a dispatch kernel (ep_dispatch_with_layout):
// the slot table holds, for each kept (t, r), its position p inside its chunk
// of 2^shift tokens encoded as -2 - p, and chunk_rank the chunks' per-rank
// counts.  Every CTA scans the counts per rank over the chunks in shared
// memory (build_chunk_base); a token's receive row on rank r is then
// rank_offset[r] + rows of r in earlier chunks + p (final_slot).  Values >= -1
// are final already, so a reader may meet either form.  chunk_rank ==
// nullptr: the slot table is final (ordinary dispatch).
struct Finalize {
  const int32_t* chunk_rank;  // [C][W]
  const int32_t* chunk_exp;   // [C][E]
  int64_t C;
  int shift;
  int E;
  int32_t* num_tokens_per_expert;
  int32_t* num_tokens_per_rank;
  int32_t* rank_offset;
  unsigned long long* claim;  // zero at the dispatch's start (the count kernel zeroes it), or null
};
constexpr int kFinMaxBytes = 16384;  // shared memory for the chunk table (C * W ints)

// s_base[c * W + r] = rows of r in chunks before c; s_tot[r] = rows of r;
// s_off[r] = rank_offset[r] (s_off[W] = R).  CTA 0 writes the per-rank totals
// and offsets.  Every thread of the CTA must call it.
__device__ __forceinline__ void build_chunk_base(const Finalize& fin, int W, int32_t* s_base,
                                                 int32_t* s_tot, int32_t* s_off) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int64_t n_ent = fin.C * W;
  for (int64_t i = threadIdx.x; i < n_ent; i += blockDim.x) s_base[i] = fin.chunk_rank[i];
  __syncthreads();
  for (int r = warp; r < W; r += nwarps) {  // exclusive scan of rank r over the chunks
    int carry = 0;
    for (int64_t c0 = 0; c0 < fin.C; c0 += 32) {
      const int64_t c = c0 + lane;
      const int v = c < fin.C ? s_base[c * W + r] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += u;
      }
      if (c < fin.C) s_base[c * W + r] = carry + incl - v;
      carry += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) s_tot[r] = carry;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0;
    for (int r = 0; r < W; ++r) {
      s_off[r] = off;
      off += s_tot[r];
    }
    s_off[W] = off;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i <= W; i += blockDim.x) {
      fin.rank_offset[i] = s_off[i];
      if (i < W) fin.num_tokens_per_rank[i] = s_tot[i];
    }
  }
}

// The receive row of (t, r) from an entry of the slot table.
__device__ __forceinline__ int final_slot(int v, int64_t t, int r, int W, int shift,
                                          const int32_t* s_base, const int32_t* s_off) {
  return v <= -2 ? s_off[r] + s_base[(t >> shift) * W + r] + (-2 - v) : v;
}

// Per-expert totals over the chunks: a warp per expert, the chunks over its
// lanes, the experts spread over the grid's warps.
__device__ __forceinline__ void finish_expert_totals(const Finalize& fin) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int64_t e = blockIdx.x + (int64_t)warp * gridDim.x; e < fin.E;
       e += (int64_t)nwarps * gridDim.x) {
    int sum = 0;
    for (int64_t c = lane; c < fin.C; c += 32) sum += fin.chunk_exp[c * fin.E + e];
    sum = warp_sum(sum);
    if (lane == 0) fin.num_tokens_per_expert[e] = sum;
  }
}

// ep_dispatch_regions / ep_combine_regions: the dispatch of a final slot
// table into per-rank regions, and the combine that reads them.
cudaError_t launch_dispatch_regions(const void* x, const int32_t* topk_idx, const float* topk_w,
                                    int64_t T, int H, int k, int W, const int32_t* slot,
                                    int quant, const RankRegions& regions, int32_t* status,
                                    cudaStream_t stream);
cudaError_t launch_combine_regions(const RankRegions& y_regions, const int32_t* slot, int64_t T,
                                   int H, int W, void* out, int32_t* status, cudaStream_t stream);
// The one-launch layout + dispatch into per-rank regions (small batches).
cudaError_t launch_dispatch_fused_regions(const void* x, const int32_t* topk_idx,
                                          const float* topk_w, int64_t T, int H, int k, int E,
                                          int W, int32_t* ne, int32_t* nr, int32_t* off,
                                          int32_t* slot, const RankRegions& regions,
                                          int32_t* status, cudaStream_t stream);
// ep_dispatch_regions_with_layout: the layout, then (or finished by) the
// dispatch into per-rank regions, in one call.
cudaError_t launch_dispatch_regions_with_layout(
    const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T, int H, int k, int E,
    int W, int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank, int32_t* rank_offset,
    int32_t* slot, void* workspace, int quant, const RankRegions& regions, int32_t* status,
    cudaStream_t stream);

template <typename K>
inline int grid_for(K kernel, int64_t T, int threads) {
  static int cache[128];
  const int per_sm = occupancy_cached(kernel, threads, cache);
  const int64_t want = (T * 32 + threads - 1) / threads;  // one warp per token
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  int64_t g = want < cap ? want : cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace ep
