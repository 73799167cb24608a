// Device helpers shared by the dispatch kernels (bf16 and FP8 payloads).
#pragma once

#include "ep_device.cuh"

namespace ep {

// Destinations of token t in ascending rank order: lane i < nd holds the i-th
// destination's receive row.  Rows at or beyond the capacity are dropped and
// reported.  (The cached (token, rank) -> row map of "perf(ep): optimize
// IntraNode dispatch kernel for MI350X", Technical Details 1, is `slot`.)
struct Dests {
  int nd;
  int my_row;
  bool cap_err;
};

__device__ __forceinline__ Dests token_dests(const int32_t* __restrict__ slot, int64_t t, int W,
                                             int64_t cap, int lane) {
  int s = -1;
  if (lane < W) s = __ldg(slot + t * W + lane);
  const bool keep = s >= 0 && (int64_t)s < cap;
  const bool over = s >= 0 && (int64_t)s >= cap;
  const unsigned dmask = __ballot_sync(kFull, keep);
  const int r = nth_set_bit_of_lane(dmask, lane);
  const int row = __shfl_sync(kFull, s, r & 31);
  Dests d;
  d.nd = __popc(dmask);
  d.my_row = r >= 0 ? row : -1;
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
// reloads.
__device__ __forceinline__ void carry_metadata(const int32_t* __restrict__ topk_idx,
                                               const float* __restrict__ topk_w, int64_t t, int k,
                                               const Dests& d, int32_t* __restrict__ recv_topk_idx,
                                               float* __restrict__ recv_topk_w,
                                               int32_t* __restrict__ recv_src, int lane) {
  const int per = 2 * k + 1;
  for (int w0 = 0; w0 < per; w0 += 32) {
    const int j = w0 + lane;
    uint32_t* col = nullptr;  // the word's address in receive row 0
    uint32_t stride = 1, val = 0;
    if (j < k) {
      if (recv_topk_idx != nullptr) {
        col = reinterpret_cast<uint32_t*>(recv_topk_idx) + j;
        stride = (uint32_t)k;
        val = (uint32_t)__ldg(topk_idx + t * k + j);
      }
    } else if (j < 2 * k) {
      if (recv_topk_w != nullptr) {
        col = reinterpret_cast<uint32_t*>(recv_topk_w) + (j - k);
        stride = (uint32_t)k;
        val = __float_as_uint(__ldg(topk_w + t * k + (j - k)));
      }
    } else if (j == 2 * k && recv_src != nullptr) {
      col = reinterpret_cast<uint32_t*>(recv_src);
      val = (uint32_t)t;
    }
    for (int qq = 0; qq < d.nd; ++qq) {
      const uint32_t row = (uint32_t)__shfl_sync(kFull, d.my_row, qq);
      if (col != nullptr) st_b32(col + (uint64_t)row * stride, val);
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
