// Dispatch: one warp per token reads the token's row once and writes it to the
// receive row of every destination rank (bf16 bit copy, or FP8 e4m3 with one
// fp32 scale per 1x128 block), and carries the top-k ids, weights and the
// source index along.
#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kDThreads = 256;

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

// bf16 payload: lane l moves 16-byte chunks l, l+32, ... of the row; U chunks
// are loaded before the stores of a round so that each lane keeps U loads in
// flight.  The row is read once whatever the number of destinations.
template <int U>
__global__ void __launch_bounds__(kDThreads)
    dispatch_bf16_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ topk_idx,
                         const float* __restrict__ topk_w, int64_t T, int n16, int k, int W,
                         const int32_t* __restrict__ slot, int64_t cap, uint4* __restrict__ recv_x,
                         int32_t* __restrict__ recv_topk_idx, float* __restrict__ recv_topk_w,
                         int32_t* __restrict__ recv_src, int32_t* __restrict__ status) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * kDThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDThreads) >> 5;
  bool cap_err = false;
  for (int64_t t = gwarp; t < T; t += nwarps) {
    const Dests d = token_dests(slot, t, W, cap, lane);
    cap_err |= d.cap_err;
    carry_metadata(topk_idx, topk_w, t, k, d, recv_topk_idx, recv_topk_w, recv_src, lane);
    const uint4* src = x + t * n16;
    for (int c0 = 0; c0 < n16; c0 += 32 * U) {
      uint4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < n16) v[u] = ld_stream_v4(src + c);
      }
      for (int dg = 0; dg < d.nd; dg += 8) {
        int rows[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) rows[q] = __shfl_sync(kFull, d.my_row, (dg + q) & 31);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (dg + q < d.nd) {
            uint4* dst = recv_x + (int64_t)rows[q] * n16;
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
  pdl_launch_dependents();
  if (cap_err && lane == 0 && status != nullptr) atomicOr(status, EP_STATUS_CAPACITY);
}

// Two fp32 values to two e4m3 codes, round to nearest even, saturating to
// +-448: `lo` goes to the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One e4m3 code per value, of v / s with s > 0, exactly as if v / s were first
// rounded to fp32 by IEEE division and that quotient then rounded to e4m3
// (nearest, ties to even, saturating to +-448).  The e4m3 code is a
// monotonic function of the quotient, so it is decided by a cheap quotient
// q = v * (1/s) whenever the fp32 values 16 bit patterns below and above q
// (in magnitude) map to the same code: |q - fl(v/s)| is only a few ulps
// (rcp.approx has at most 1 ulp error, the product adds half an ulp), so the
// correctly rounded quotient lies between them.  Otherwise (q near a rounding
// boundary of e4m3, which happens for a few values in 10^5) the code comes from
// the IEEE division itself.  `r` is 1/s from rcp.approx; r_ok is false when s
// is subnormal or 1/s not finite, in which case every value takes the division.
__device__ __forceinline__ uint32_t e4m3_of_quotient(float v, float s, float r, bool r_ok) {
  if (r_ok) {
    const float q = v * r;
    const uint32_t m = __float_as_uint(q) & 0x7fffffffu;
    const float lo = __uint_as_float(m > 16u ? m - 16u : 0u);
    const float hi = __uint_as_float(m + 16u);
    const uint32_t both = e4m3x2(lo, hi);
    if ((both & 0xffu) == (both >> 8)) return (e4m3x2(q, 0.0f) & 0xffu);
  }
  return e4m3x2(__fdiv_rn(v, s), 0.0f) & 0xffu;
}

__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// FP8 payload.  A 128-column block is 256 bytes of bf16 = 8 lanes x 32 bytes,
// so a warp covers four blocks per round (lanes 8b..8b+7 for block b).  Per
// block: amax over the block (an 8-lane max reduction), scale = amax / 448
// (IEEE division), codes of x / scale (e4m3_of_quotient).  A token row is
// split into `nseg` segments of block quadruples, one warp per (token,
// segment), so that small batches still fill the GPU; each segment is
// quantised once and its codes and scales are stored to every destination.
template <int U>
__global__ void __launch_bounds__(kDThreads)
    dispatch_fp8_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ topk_idx,
                        const float* __restrict__ topk_w, int64_t T, int H, int k, int W,
                        const int32_t* __restrict__ slot, int64_t cap, uint8_t* __restrict__ recv_x,
                        float* __restrict__ recv_scale, int32_t* __restrict__ recv_topk_idx,
                        float* __restrict__ recv_topk_w, int32_t* __restrict__ recv_src,
                        int nseg, int32_t* __restrict__ status) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int qb = lane >> 3, hl = lane & 7;  // block within the quad, lane within the block
  const int nb = H >> 7;
  const int n16 = H >> 3;
  const int nquad = (nb + 3) >> 2;
  const int per_seg = (nquad + nseg - 1) / nseg;
  const int64_t gwarp = ((int64_t)blockIdx.x * kDThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDThreads) >> 5;
  bool cap_err = false;
  for (int64_t u = gwarp; u < T * nseg; u += nwarps) {
    const int64_t t = u / nseg;
    const int seg = (int)(u - t * nseg);
    const Dests d = token_dests(slot, t, W, cap, lane);
    if (seg == 0) {
      cap_err |= d.cap_err;
      carry_metadata(topk_idx, topk_w, t, k, d, recv_topk_idx, recv_topk_w, recv_src, lane);
    }
    const uint4* src = x + t * n16;
    const int q_end = (seg + 1) * per_seg < nquad ? (seg + 1) * per_seg : nquad;
    for (int q0 = seg * per_seg; q0 < q_end; q0 += U) {
      uint4 codes[U];
      float sc[U];
#pragma unroll
      for (int v = 0; v < U; ++v) {
        const int b = (q0 + v) * 4 + qb;
        uint4 a = make_uint4(0u, 0u, 0u, 0u), c = make_uint4(0u, 0u, 0u, 0u);
        if (q0 + v < q_end && b < nb) {
          a = ld_stream_v4(src + b * 16 + hl * 2);
          c = ld_stream_v4(src + b * 16 + hl * 2 + 1);
        }
        const float f[16] = {bf16_lo(a.x), bf16_hi(a.x), bf16_lo(a.y), bf16_hi(a.y),
                             bf16_lo(a.z), bf16_hi(a.z), bf16_lo(a.w), bf16_hi(a.w),
                             bf16_lo(c.x), bf16_hi(c.x), bf16_lo(c.y), bf16_hi(c.y),
                             bf16_lo(c.z), bf16_hi(c.z), bf16_lo(c.w), bf16_hi(c.w)};
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(f[i]));
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        const float s = __fdiv_rn(m, 448.0f);
        sc[v] = s;
        uint32_t w4[4] = {0u, 0u, 0u, 0u};
        if (s != 0.0f) {
          const float r = rcp_approx(s);
          const bool r_ok = s >= 1.17549435e-38f && r < 3.0e38f;  // normal s, finite 1/s
#pragma unroll
          for (int i = 0; i < 16; ++i) w4[i >> 2] |= e4m3_of_quotient(f[i], s, r, r_ok) << (8 * (i & 3));
        }
        codes[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      for (int dg = 0; dg < d.nd; dg += 8) {
        int rows[8];
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) rows[qq] = __shfl_sync(kFull, d.my_row, (dg + qq) & 31);
#pragma unroll
        for (int qq = 0; qq < 8; ++qq) {
          if (dg + qq < d.nd) {
            uint8_t* dst = recv_x + (int64_t)rows[qq] * H;
            float* dsc = recv_scale + (int64_t)rows[qq] * nb;
#pragma unroll
            for (int v = 0; v < U; ++v) {
              const int b = (q0 + v) * 4 + qb;
              if (q0 + v < q_end && b < nb) {
                st_v4(reinterpret_cast<uint4*>(dst + b * 128 + hl * 16), codes[v]);
                if (hl == 0) dsc[b] = sc[v];
              }
            }
          }
        }
      }
    }
  }
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
#ifndef EP_TMA_STAGES
#define EP_TMA_STAGES 3
#endif
#ifndef EP_TMA_SMEM_BUDGET
#define EP_TMA_SMEM_BUDGET (200 * 1024)
#endif
#ifndef EP_TMA_MAX_WARPS
#define EP_TMA_MAX_WARPS 8
#endif
#ifndef EP_TMA_CTAS_PER_SM
#define EP_TMA_CTAS_PER_SM 1
#endif
constexpr int kTmaStages = EP_TMA_STAGES;            // row buffers per warp
constexpr int kTmaBarBytes = 1024;                   // barrier area ahead of the row buffers
constexpr int kTmaSmemBudget = EP_TMA_SMEM_BUDGET;   // row buffers per CTA
constexpr int kTmaMaxWarps = EP_TMA_MAX_WARPS;
constexpr int kTmaCtasPerSm = EP_TMA_CTAS_PER_SM;
constexpr uint32_t kTmaMinRowBytes = 1024;  // smaller rows: 16-byte stores from registers

__device__ __forceinline__ int load_slot(const int32_t* __restrict__ slot, int64_t t, int W,
                                         int lane, int64_t T) {
  return (t < T && lane < W) ? __ldg(slot + t * W + lane) : -1;
}

__global__ void __launch_bounds__(kTmaMaxWarps * 32, 1)
    dispatch_bf16_tma_kernel(const uint8_t* __restrict__ x, const int32_t* __restrict__ topk_idx,
                             const float* __restrict__ topk_w, int64_t T, uint32_t row_bytes,
                             uint32_t stage_bytes, int k, int W, const int32_t* __restrict__ slot,
                             int64_t cap, uint8_t* __restrict__ recv_x,
                             int32_t* __restrict__ recv_topk_idx, float* __restrict__ recv_topk_w,
                             int32_t* __restrict__ recv_src, int32_t* __restrict__ status) {
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
  pdl_wait();

  const int64_t gw = (int64_t)blockIdx.x * cta_warps + warp;
  const int64_t NW = (int64_t)gridDim.x * cta_warps;
  const int64_t n = gw < T ? (T - 1 - gw) / NW + 1 : 0;  // tokens gw, gw+NW, ...
  int64_t issued = 0;                                      // tokens whose row load was issued
  if (lane == 0) {
    for (; issued < n && issued < kTmaStages; ++issued) {
      mbar_arrive_expect_tx(&full[issued], row_bytes);
      bulk_load(buf + issued * stage_bytes, x + (gw + issued * NW) * row_bytes, row_bytes,
                &full[issued]);
    }
  }
  const bool meta_lanes = 2 * k + 1 <= 32;
  bool cap_err = false, timed_out = false;
  int s_cur = load_slot(slot, gw, W, lane, T);
  int64_t j = 0;
  for (; j < n; ++j) {
    const int64_t t = gw + j * NW;
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
    const int s_next = load_slot(slot, t + NW, W, lane, T);
    const bool keep = s_cur >= 0 && (int64_t)s_cur < cap;
    cap_err |= __any_sync(kFull, s_cur >= 0 && (int64_t)s_cur >= cap);
    const unsigned dmask = __ballot_sync(kFull, keep);
    const int nd = __popc(dmask);
    const int r = nth_set_bit_of_lane(dmask, lane);
    const int my_row = __shfl_sync(kFull, s_cur, r & 31);

    bool ok = true;
    if (lane == 0) ok = mbar_wait_bounded(&full[st], parity);
    if (!__shfl_sync(kFull, ok, 0)) {
      timed_out = true;
      break;
    }
    for (int q = 0; q < nd; ++q) {
      const int row = __shfl_sync(kFull, my_row, q);
      if (lane == 0) bulk_store(recv_x + (int64_t)row * row_bytes, buf + st * stage_bytes, row_bytes);
    }
    if (lane == 0) bulk_commit();
    if (meta_lanes) {
      for (int q = 0; q < nd; ++q) {
        const int64_t row = __shfl_sync(kFull, my_row, q);
        if (lane < k) {
          if (recv_topk_idx) recv_topk_idx[row * k + lane] = mv;
        } else if (lane < 2 * k) {
          if (recv_topk_w) recv_topk_w[row * k + (lane - k)] = __int_as_float(mv);
        } else if (lane == 2 * k) {
          if (recv_src) recv_src[row] = mv;
        }
      }
    } else {
      Dests d;
      d.nd = nd;
      d.my_row = r >= 0 ? my_row : -1;
      d.cap_err = false;
      carry_metadata(topk_idx, topk_w, t, k, d, recv_topk_idx, recv_topk_w, recv_src, lane);
    }
    // refill the previous token's buffer once the copies out of it have read it
    if (lane == 0 && j >= 1 && issued < n) {
      bulk_wait_read<1>();
      const int sp = (int)((j - 1) % kTmaStages);
      mbar_arrive_expect_tx(&full[sp], row_bytes);
      bulk_load(buf + sp * stage_bytes, x + (gw + issued * NW) * row_bytes, row_bytes, &full[sp]);
      ++issued;
    }
    issued = __shfl_sync(kFull, issued, 0);
    s_cur = s_next;
  }
  if (lane == 0) {
    // never leave with a bulk copy still using this CTA's shared memory
    for (int64_t q = j; q < issued; ++q)
      (void)mbar_wait_bounded(&full[q % kTmaStages], (uint32_t)((q / kTmaStages) & 1));
    bulk_wait_all();
  }
  __syncwarp();
  pdl_launch_dependents();
  if (lane == 0 && status != nullptr) {
    if (cap_err) atomicOr(status, EP_STATUS_CAPACITY);
    if (timed_out) atomicOr(status, EP_STATUS_TIMEOUT);
  }
}

template <typename K>
int grid_for(K kernel, int64_t T, int threads) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (T * 32 + threads - 1) / threads;  // one warp per token
  const int64_t cap = (int64_t)device_sm_count() * per_sm;
  int64_t g = want < cap ? want : cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_dispatch(const void* x, const int32_t* topk_idx, const float* topk_w,
                            int64_t T, int H, int k, int W, const int32_t* slot,
                            int64_t capacity_rows, int quant, void* recv_x, float* recv_scale,
                            int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                            int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const uint4* x4 = static_cast<const uint4*>(x);
  if (quant == EP_QUANT_BF16) {
    const uint32_t row_bytes = (uint32_t)H * 2u;
    const uint32_t stage_bytes = (row_bytes + 127u) & ~127u;
    const int cta_warps_fit = (int)(kTmaSmemBudget / ((size_t)kTmaStages * stage_bytes));
    if (!EP_FORCE_LSU && row_bytes >= kTmaMinRowBytes && cta_warps_fit >= 1) {
      const int cta_warps = cta_warps_fit < kTmaMaxWarps ? cta_warps_fit : kTmaMaxWarps;
      const size_t smem = kTmaBarBytes + (size_t)cta_warps * kTmaStages * stage_bytes;
      static bool attr_set[128];
      int dev = 0;
      cudaGetDevice(&dev);
      if (dev >= 0 && dev < 128 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(dispatch_bf16_tma_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kTmaBarBytes + kTmaSmemBudget);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
      }
      const int64_t want = (T + cta_warps - 1) / cta_warps;
      const int64_t sms = (int64_t)device_sm_count() * kTmaCtasPerSm;
      const int grid = (int)(want < sms ? want : sms);
      return launch_pdl(dispatch_bf16_tma_kernel, dim3(grid < 1 ? 1 : grid), dim3(cta_warps * 32),
                        smem, stream, static_cast<const uint8_t*>(x), topk_idx, topk_w, T,
                        row_bytes, stage_bytes, k, W, slot, capacity_rows,
                        static_cast<uint8_t*>(recv_x), recv_topk_idx, recv_topk_w, recv_src,
                        status);
    }
    const int n16 = H / 8;
    if (n16 % (32 * 7) == 0) {
      auto kern = dispatch_bf16_kernel<7>;
      return launch_pdl(kern, dim3(grid_for(kern, T, kDThreads)), dim3(kDThreads), 0, stream, x4,
                        topk_idx, topk_w, T, n16, k, W, slot, capacity_rows,
                        static_cast<uint4*>(recv_x), recv_topk_idx, recv_topk_w, recv_src, status);
    }
    auto kern = dispatch_bf16_kernel<8>;
    return launch_pdl(kern, dim3(grid_for(kern, T, kDThreads)), dim3(kDThreads), 0, stream, x4,
                      topk_idx, topk_w, T, n16, k, W, slot, capacity_rows,
                      static_cast<uint4*>(recv_x), recv_topk_idx, recv_topk_w, recv_src, status);
  }
  // segments per token: enough (token, segment) units to give every resident warp
  // a few, but no more segments than block quadruples
  auto kern = dispatch_fp8_kernel<2>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kDThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t warps = (int64_t)device_sm_count() * per_sm * (kDThreads / 32);
  const int nquad = (H / 128 + 3) / 4;
  int nseg = (int)((2 * warps + T - 1) / T);
  nseg = nseg < 1 ? 1 : (nseg > nquad ? nquad : nseg);
  const int64_t units = T * nseg;
  const int64_t grid = (units * 32 + kDThreads - 1) / kDThreads < device_sm_count() * per_sm
                           ? (units * 32 + kDThreads - 1) / kDThreads
                           : (int64_t)device_sm_count() * per_sm;
  return launch_pdl(kern, dim3((unsigned)(grid < 1 ? 1 : grid)), dim3(kDThreads), 0, stream, x4,
                    topk_idx, topk_w, T, H, k, W, slot, capacity_rows,
                    static_cast<uint8_t*>(recv_x), recv_scale, recv_topk_idx, recv_topk_w, recv_src,
                    nseg, status);
}

}  // namespace ep
