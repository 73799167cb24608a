// Combine: one warp per token gathers the token's receive rows and sums them in
// fp32 in ascending rank order from +0, then rounds once to bf16.
#include "dispatch_common.cuh"

namespace ep {
namespace {

constexpr int kCThreads = 256;
constexpr int kCU = 2;             // 16-byte chunks per lane and row in one round
constexpr double kCSegUnits = 4.0;  // (token, segment) units per warp slot for small batches

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
  acc[0] = acc[0] + __uint_as_float(v.x << 16);
  acc[1] = acc[1] + __uint_as_float(v.x & 0xffff0000u);
  acc[2] = acc[2] + __uint_as_float(v.y << 16);
  acc[3] = acc[3] + __uint_as_float(v.y & 0xffff0000u);
  acc[4] = acc[4] + __uint_as_float(v.z << 16);
  acc[5] = acc[5] + __uint_as_float(v.z & 0xffff0000u);
  acc[6] = acc[6] + __uint_as_float(v.w << 16);
  acc[7] = acc[7] + __uint_as_float(v.w & 0xffff0000u);
}

// acc[i] = fma(wt, y[i], acc[i]): one rounding per step.
__device__ __forceinline__ void fma_bf16x8(float (&acc)[8], float wt, const uint4& v) {
  acc[0] = __fmaf_rn(wt, __uint_as_float(v.x << 16), acc[0]);
  acc[1] = __fmaf_rn(wt, __uint_as_float(v.x & 0xffff0000u), acc[1]);
  acc[2] = __fmaf_rn(wt, __uint_as_float(v.y << 16), acc[2]);
  acc[3] = __fmaf_rn(wt, __uint_as_float(v.y & 0xffff0000u), acc[3]);
  acc[4] = __fmaf_rn(wt, __uint_as_float(v.z << 16), acc[4]);
  acc[5] = __fmaf_rn(wt, __uint_as_float(v.z & 0xffff0000u), acc[5]);
  acc[6] = __fmaf_rn(wt, __uint_as_float(v.w << 16), acc[6]);
  acc[7] = __fmaf_rn(wt, __uint_as_float(v.w & 0xffff0000u), acc[7]);
}

// A warp takes one (token, segment) unit at a time: segment s of a token is
// the 16-byte chunks [s * seg16, (s + 1) * seg16) of its hidden dimension, so
// that small batches still give every SM enough warps (S segments per token).
// Lane l handles chunks l, l+32, ... of the segment.  For a round of U chunks
// the loads of up to 8 destination rows are all issued before the first
// addition (8*U loads in flight per lane); the additions then run in
// ascending column order, which fixes the rounding of the sum.  WEIGHTED:
// each row enters as a fused multiply-add with the weight of its column,
// w[t][c] ("perf(ep): optimize IntraNode dispatch kernel for MI350X",
// Remaining gap: combine accumulates the rows with FMA).
template <int U, bool WEIGHTED, bool SEG, class RT>
__global__ void __launch_bounds__(kCThreads)
    combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ slot,
                   const float* __restrict__ w, int64_t T, int n16, int S, int seg16, int W,
                   int64_t cap, uint4* __restrict__ out, int32_t* __restrict__ status, RT rt) {
  __shared__ typename RT::View s_rv;  // per-rank regions of y: the table
  load_region_view(rt, W, s_rv);
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int32_t first_row = region_first_row(rt, W, lane);
  const int64_t gwarp = ((int64_t)blockIdx.x * kCThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kCThreads) >> 5;
  if constexpr (!SEG) S = 1;  // whole rows: the unit is the token
  const int64_t units = T * S;
  bool cap_err = false;
  int s_next = (gwarp < units && lane < W) ? __ldg(slot + (SEG ? gwarp / S : gwarp) * W + lane) : -1;
  for (int64_t un = gwarp; un < units; un += nwarps) {
    const int64_t t = SEG ? un / S : un;
    const int c_lo = SEG ? (int)(un - t * S) * seg16 : 0;
    const int c_hi = SEG ? min(c_lo + seg16, n16) : n16;
    int s = s_next;
    const int64_t un2 = un + nwarps;
    s_next = (un2 < units && lane < W) ? __ldg(slot + (SEG ? un2 / S : un2) * W + lane) : -1;

    int64_t srow = s, lim = cap;  // the row in its storage and that storage's capacity
    if (RT::kRegions && s >= 0) {
      srow = storage_row<RT>(s, first_row);
      lim = storage_rows<RT>(lane, cap, s_rv);
    }
    const bool keep = s >= 0 && srow < lim;
    cap_err |= __any_sync(kFull, s >= 0 && srow >= lim);
    const unsigned dmask = __ballot_sync(kFull, keep);
    const int nd = __popc(dmask);
    const int r = nth_set_bit_of_lane(dmask, lane);
    const int my_row = __shfl_sync(kFull, (int)srow, r & 31);  // lane i: row of i-th destination
    float my_w = 0.0f;
    if constexpr (WEIGHTED) {
      const float wl = lane < W ? __ldg(w + t * W + lane) : 0.0f;
      my_w = __shfl_sync(kFull, wl, r & 31);               // and its weight
    }
    // lane i's destination row as an address, formed once per unit (for
    // per-rank regions: its region's base plus the row inside it)
    const uint4* my_src = y;
    if (r >= 0)
      my_src = reinterpret_cast<const uint4*>(rows_base<RT>(
                   s_rv, r, reinterpret_cast<uint8_t*>(const_cast<uint4*>(y)))) +
               (int64_t)my_row * n16;
    uint4* dst = out + t * n16;
    for (int c0 = c_lo; c0 < c_hi; c0 += 32 * U) {
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
      for (int dg = 0; dg < nd; dg += 8) {
        float wts[8];
        const uint4* ybase[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          wts[q] = WEIGHTED ? __shfl_sync(kFull, my_w, (dg + q) & 31) : 1.0f;
          ybase[q] = reinterpret_cast<const uint4*>(__shfl_sync(
              kFull, reinterpret_cast<unsigned long long>(my_src), (dg + q) & 31));
        }
        uint4 v[8][U];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int c = c0 + u * 32 + lane;
            v[q][u] = make_uint4(0u, 0u, 0u, 0u);
            if (dg + q < nd && c < c_hi)
              v[q][u] = ld_stream_v4(ybase[q] + c);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (dg + q < nd) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
              if constexpr (WEIGHTED)
                fma_bf16x8(acc[u], wts[q], v[q][u]);
              else
                add_bf16x8(acc[u], v[q][u]);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < c_hi) {
          const uint4 o = make_uint4(bf16x2_rn(acc[u][0], acc[u][1]), bf16x2_rn(acc[u][2], acc[u][3]),
                                     bf16x2_rn(acc[u][4], acc[u][5]), bf16x2_rn(acc[u][6], acc[u][7]));
          st_v4(dst + c, o);
        }
      }
    }
  }
  pdl_launch_dependents();
  if (cap_err && lane == 0 && status != nullptr) atomicOr(status, EP_STATUS_CAPACITY);
}

// Combine through the bulk-copy (TMA) engine.  A ring of kCStages stages in
// shared memory holds one row chunk each (a whole row for H <= 8192).  Warp 0
// produces: for each of the CTA's tokens and each chunk, lane q loads the
// chunk of the token's q-th destination row (ascending rank) into the next
// stage with one bulk copy, once that stage is free, and writes the stage's
// descriptor (token, chunk, last-row flag).  Warps 1..kCWarps consume the
// stages strictly in ring order: each thread adds its 16-byte pieces of the
// stage to fp32 running sums in registers and, at the token's last row,
// rounds them to bf16 and stores them.  So the sum runs in ascending rank
// order, a stage is handed back as soon as it has been added, and no token has
// to sit in shared memory whole: the ring only holds bytes in flight.
// Whole-row copies and several issuing lanes keep the copy engine streaming.
// Used for kCTmaMinT <= T <= kCTmaMaxT: measured on
// GB300 (H=7168, top-8, W=8) it beats the register kernel at T=1024 (26 us
// against 27-28 us) and loses at T=4096 (71 us against 66 us); below T=768 the
// register kernel with row segments keeps more loads in flight (T=256: 12 us
// against 14.8 us).
constexpr int64_t kCTmaMaxT = 1024;
constexpr int64_t kCTmaMinT = 768;
constexpr int kCWarps = 8;                                       // consumer warps
constexpr uint32_t kCStage = 16384;                              // bytes per stage
constexpr int kCStages = (208 * 1024) / kCStage;                 // ring length
constexpr int kCPieces = kCStage / (16 * 32 * kCWarps);          // pieces per thread per stage
constexpr int kCHead = 1024;                                     // barriers + descriptors
constexpr uint32_t kDescLast = 1u, kDescNone = 2u, kDescDone = 4u;
static_assert(kCStage % (16 * 32 * kCWarps) == 0, "stage must split evenly over consumers");
static_assert(kCStages * (16 + 16) <= kCHead, "header too small");
static_assert(kCStages <= 32, "one producer lane per stage of a token at most");

__global__ void __launch_bounds__((kCWarps + 1) * 32, 1)
    combine_tma_kernel(const uint8_t* __restrict__ y, const int32_t* __restrict__ slot, int64_t T,
                       uint32_t row_bytes, uint32_t chunk_bytes, int W, int64_t cap,
                       uint8_t* __restrict__ out, int32_t* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kCStages;
  int64_t* desc_tok = reinterpret_cast<int64_t*>(empty + kCStages);
  uint32_t* desc_info = reinterpret_cast<uint32_t*>(desc_tok + kCStages);  // chunk << 8 | flags
  uint8_t* ring = smem + kCHead;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kCStages) {
    mbar_init(&full[threadIdx.x], 1);
    mbar_init(&empty[threadIdx.x], kCWarps);
  }
  fence_barrier_init();
  __syncthreads();
  pdl_wait();

  const int64_t G = gridDim.x;
  const int64_t n_tok = (int64_t)blockIdx.x < T ? (T - 1 - blockIdx.x) / G + 1 : 0;
  const int nch = (int)((row_bytes + chunk_bytes - 1) / chunk_bytes);
  bool timed_out = false;

  if (warp == 0) {
    // ---------------- producer
    bool cap_err = false;
    int64_t g = 0;  // stages issued
    int s_next = (n_tok > 0 && lane < W) ? __ldg(slot + (int64_t)blockIdx.x * W + lane) : -1;
    for (int64_t i = 0; i < n_tok && !timed_out; ++i) {
      const int64_t t = blockIdx.x + i * G;
      const int s_cur = s_next;
      s_next = (i + 1 < n_tok && lane < W) ? __ldg(slot + (t + G) * W + lane) : -1;
      const bool keep = s_cur >= 0 && (int64_t)s_cur < cap;
      cap_err |= __any_sync(kFull, s_cur >= 0 && (int64_t)s_cur >= cap);
      const unsigned dmask = __ballot_sync(kFull, keep);
      const int nd = __popc(dmask);
      const int r = nth_set_bit_of_lane(dmask, lane);
      const int my_row = __shfl_sync(kFull, s_cur, r & 31);  // lane q: row of the q-th destination
      const int need = nd > 0 ? nd : 1;
      for (int c = 0; c < nch && !timed_out; ++c) {
        const uint32_t off = (uint32_t)c * chunk_bytes;
        const uint32_t bytes = row_bytes - off < chunk_bytes ? row_bytes - off : chunk_bytes;
        bool ok = true;
        if (lane < need) {
          const int64_t gq = g + lane;
          const int st = (int)(gq % kCStages);
          if (gq >= kCStages)
            ok = mbar_wait_bounded(&empty[st], (uint32_t)(((gq / kCStages) - 1) & 1));
          if (ok) {
            desc_tok[st] = t;
            desc_info[st] = ((uint32_t)c << 8) | (lane == need - 1 ? kDescLast : 0u) |
                            (nd == 0 ? kDescNone : 0u);
            if (nd > 0) {
              mbar_arrive_expect_tx(&full[st], bytes);
              bulk_load(ring + (size_t)st * kCStage, y + (int64_t)my_row * row_bytes + off, bytes,
                        &full[st]);
            } else {
              mbar_arrive_expect_tx(&full[st], 0);
            }
          }
        }
        timed_out = !__all_sync(kFull, ok);
        g += need;
      }
    }
    if (!timed_out && lane == 0) {  // end marker
      const int st = (int)(g % kCStages);
      if (g < kCStages || mbar_wait_bounded(&empty[st], (uint32_t)(((g / kCStages) - 1) & 1))) {
        desc_info[st] = kDescDone;
        mbar_arrive_expect_tx(&full[st], 0);
      } else {
        timed_out = true;
      }
      ++g;
    }
    // copies still landing in shared memory must finish before the CTA exits
    for (int64_t q = (g > kCStages ? g - kCStages : 0) + lane; q < g; q += 32)
      (void)mbar_wait_bounded(&full[q % kCStages], (uint32_t)((q / kCStages) & 1));
    if (lane == 0 && status != nullptr) {
      if (cap_err) atomicOr(status, EP_STATUS_CAPACITY);
      if (timed_out) atomicOr(status, EP_STATUS_TIMEOUT);
    }
  } else if (n_tok > 0) {
    // ---------------- consumers
    const int ct = threadIdx.x - 32;
    float acc[kCPieces][8];
#pragma unroll
    for (int pc = 0; pc < kCPieces; ++pc)
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[pc][e] = 0.0f;
    for (int64_t g = 0;; ++g) {
      const int st = (int)(g % kCStages);
      if (!mbar_wait_bounded(&full[st], (uint32_t)((g / kCStages) & 1))) {
        timed_out = true;
        break;
      }
      const uint32_t info = desc_info[st];
      if (info & kDescDone) break;
      const int64_t t = desc_tok[st];
      const uint32_t off = (info >> 8) * chunk_bytes;
      const uint32_t bytes = row_bytes - off < chunk_bytes ? row_bytes - off : chunk_bytes;
      const uint8_t* sb = ring + (size_t)st * kCStage;
      if (!(info & kDescNone)) {
#pragma unroll
        for (int pc = 0; pc < kCPieces; ++pc) {
          const uint32_t p = (uint32_t)(pc * 32 * kCWarps + ct);
          if (p * 16 < bytes) add_bf16x8(acc[pc], *reinterpret_cast<const uint4*>(sb + p * 16));
        }
      }
      if (info & kDescLast) {
        uint4* dst = reinterpret_cast<uint4*>(out + t * row_bytes + off);
#pragma unroll
        for (int pc = 0; pc < kCPieces; ++pc) {
          const uint32_t p = (uint32_t)(pc * 32 * kCWarps + ct);
          if (p * 16 < bytes)
            st_v4(dst + p, make_uint4(bf16x2_rn(acc[pc][0], acc[pc][1]),
                                      bf16x2_rn(acc[pc][2], acc[pc][3]),
                                      bf16x2_rn(acc[pc][4], acc[pc][5]),
                                      bf16x2_rn(acc[pc][6], acc[pc][7])));
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[pc][e] = 0.0f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (timed_out && lane == 0 && status != nullptr) atomicOr(status, EP_STATUS_TIMEOUT);
  }
  __syncthreads();
  pdl_launch_dependents();
}

}  // namespace

// One warp per token, as many CTAs as fit on the device at once (grid-stride
// over the tokens beyond that).
template <typename K1, typename KS, class RT>
cudaError_t launch_combine_regs(K1 kern_rows, KS kern_seg, const void* y, const int32_t* slot,
                                const float* w, int64_t T, int H, int W, int64_t capacity_rows,
                                void* out, int32_t* status, cudaStream_t stream, const RT& rt) {
  static int cache[128];
  const int per_sm = occupancy_cached(kern_seg, kCThreads, cache);
  const int64_t most = (int64_t)device_sm_count() * per_sm;
  // Segments, when the batch has fewer tokens than the device has warp slots:
  // enough (token, segment) units for kCSegUnits units per slot, each
  // segment at least one full round (32 * U chunks).  Measured on GB300 with
  // H = 7168, top-8: T = 256 runs in 12 us instead of 17 us, T = 512 in 16 us
  // instead of 22 us; from T = 4096 on whole rows are best.
  const int n16 = H / 8;
  const int64_t resident = most * (kCThreads / 32);
  const int64_t target = (int64_t)(kCSegUnits * (double)resident);
  int64_t S = (T > 0 && T < resident) ? (target + T - 1) / T : 1;
  const int64_t max_s = n16 / (32 * kCU);
  if (S > max_s) S = max_s;
  if (S < 1) S = 1;
  int seg16 = (int)((n16 + S - 1) / S);
  seg16 = (seg16 + 31) & ~31;
  S = (n16 + seg16 - 1) / seg16;
  const int64_t want = (T * S * 32 + kCThreads - 1) / kCThreads;
  const int grid = (int)(want < most ? want : most);
  return launch_pdl(S > 1 ? kern_seg : kern_rows, dim3(grid < 1 ? 1 : grid), dim3(kCThreads), 0,
                    stream, static_cast<const uint4*>(y), slot, w, T, n16, (int)S, seg16, W,
                    capacity_rows, static_cast<uint4*>(out), status, rt);
}

cudaError_t launch_combine(const void* y, const int32_t* slot, int64_t T, int H, int W,
                           int64_t capacity_rows, void* out, int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const uint32_t row_bytes = (uint32_t)H * 2u;
  // (a token's rows must fit the ring at once: W <= kCStages)
  if (row_bytes >= 1024 && W <= kCStages && T <= kCTmaMaxT && T >= kCTmaMinT) {
    // chunks of at most one stage, equal up to 16 bytes
    const uint32_t nch = (row_bytes + kCStage - 1) / kCStage;
    const uint32_t chunk = ((row_bytes / nch + 15u) & ~15u);
    const size_t smem = kCHead + (size_t)kCStages * kCStage;
    static bool attr_set[128];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 128 && !attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(combine_tma_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
    const int64_t sms = device_sm_count();
    const int grid = (int)(T < sms ? T : sms);
    return launch_pdl(combine_tma_kernel, dim3(grid < 1 ? 1 : grid), dim3((kCWarps + 1) * 32),
                      smem, stream, static_cast<const uint8_t*>(y), slot, T, row_bytes, chunk, W,
                      capacity_rows, static_cast<uint8_t*>(out), status);
  }
  return launch_combine_regs(combine_kernel<kCU, false, false, OneBuffer>,
                             combine_kernel<kCU, false, true, OneBuffer>, y, slot, nullptr, T, H, W,
                             capacity_rows, out, status, stream, OneBuffer{});
}

cudaError_t launch_combine_regions(const RankRegions& y_regions, const int32_t* slot, int64_t T,
                                   int H, int W, void* out, int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_combine_regs(combine_kernel<kCU, false, false, RankRegions>,
                             combine_kernel<kCU, false, true, RankRegions>, nullptr, slot, nullptr,
                             T, H, W, /*capacity_rows=*/0, out, status, stream, y_regions);
}

cudaError_t launch_combine_weighted(const void* y, const int32_t* slot, const float* w, int64_t T,
                                    int H, int C, int64_t capacity_rows, void* out,
                                    int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_combine_regs(combine_kernel<kCU, true, false, OneBuffer>,
                             combine_kernel<kCU, true, true, OneBuffer>, y, slot, w, T, H, C,
                             capacity_rows, out, status, stream, OneBuffer{});
}

}  // namespace ep
