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

// Metadata of one token for all its destinations: per destination row, k ids,
// k weights and the source index (2k+1 words), written by the whole warp at
// once ("perf(ep): optimize IntraNode dispatch kernel for MI350X", Technical
// Details 4).
__device__ __forceinline__ void carry_metadata(const int32_t* __restrict__ topk_idx,
                                               const float* __restrict__ topk_w, int64_t t, int k,
                                               const Dests& d, int32_t* __restrict__ recv_topk_idx,
                                               float* __restrict__ recv_topk_w,
                                               int32_t* __restrict__ recv_src, int lane) {
  const int per = 2 * k + 1;
  const int total = d.nd * per;
  for (int base = 0; base < total; base += 32) {
    const int i = base + lane;
    const int dd = i / per;
    const int j = i - dd * per;
    const int row = __shfl_sync(kFull, d.my_row, dd & 31);
    if (i < total) {
      if (j < k) {
        if (recv_topk_idx) recv_topk_idx[(int64_t)row * k + j] = __ldg(topk_idx + t * k + j);
      } else if (j < 2 * k) {
        if (recv_topk_w) recv_topk_w[(int64_t)row * k + (j - k)] = __ldg(topk_w + t * k + (j - k));
      } else if (recv_src) {
        recv_src[row] = (int32_t)t;
      }
    }
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
