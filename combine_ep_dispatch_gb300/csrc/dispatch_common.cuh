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
