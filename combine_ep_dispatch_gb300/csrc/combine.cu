// Combine: one warp per token gathers the token's receive rows and sums them in
// fp32 in ascending rank order from +0, then rounds once to bf16.
#include "dispatch_common.cuh"

namespace ep {
namespace {

constexpr int kCThreads = 256;
constexpr int kCU = 2;             // 16-byte chunks per lane and row in one round

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

// Work split.  With NW warps in the grid, the first floor(T / NW) * NW tokens
// go out whole, token w + i * NW to warp w; the rounds of the remaining
// tokens (a round being 32 * U 16-byte chunks of a row), in token-major
// order, are cut into one contiguous range per warp, lengths differing by one
// round at most, so that no warp is left idle while others finish the batch.
// A warp thus takes a sequence of pieces (token, rounds [r0, r1)); for each
// it sums the token's rows over the columns of those rounds.  Lane l handles
// chunks l, l+32, ... of a round.  The loads of up to 8 destination rows are
// all issued before the first addition (8*U loads in flight per lane); the
// additions then run in ascending column order, which fixes the rounding of
// the sum.  WEIGHTED: each row enters as a fused multiply-add with the weight
// of its column, w[t][c] ("perf(ep): optimize IntraNode dispatch kernel for
// MI350X", Remaining gap: combine accumulates the rows with FMA).
template <int U, bool WEIGHTED, class RT>
__global__ void __launch_bounds__(kCThreads)
    combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ slot,
                   const float* __restrict__ w, int64_t T, int n16, int rpt, int W,
                   int64_t cap, uint4* __restrict__ out, int32_t* __restrict__ status, RT rt) {
  __shared__ typename RT::View s_rv;  // per-rank regions of y: the table
  load_region_view(rt, W, s_rv);
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int32_t first_row = region_first_row(rt, W, lane);
  const int64_t gwarp = ((int64_t)blockIdx.x * kCThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kCThreads) >> 5;
  const int64_t whole = T / nwarps;                   // whole tokens per warp
  const int64_t tail = (T - whole * nwarps) * rpt;    // rounds of the other tokens
  const int64_t q_end = whole * nwarps * rpt + (gwarp + 1) * tail / nwarps;
  int64_t i = 0, q = whole * nwarps * rpt + gwarp * tail / nwarps;
  // the next piece of this warp: token and rounds [r0, r1); false at the end
  auto next_piece = [&](int64_t& t, int& r0, int& r1) -> bool {
    if (i < whole) {
      t = gwarp + i * nwarps;
      r0 = 0;
      r1 = rpt;
      ++i;
      return true;
    }
    if (q < q_end) {
      t = q / rpt;
      r0 = (int)(q - t * rpt);
      const int64_t e = (t + 1) * rpt < q_end ? (t + 1) * rpt : q_end;
      r1 = (int)(e - t * rpt);
      q = e;
      return true;
    }
    return false;
  };
  bool cap_err = false;
  int64_t t_nx = 0;
  int r0_nx = 0, r1_nx = 0;
  bool has = next_piece(t_nx, r0_nx, r1_nx);
  int s_next = (has && lane < W) ? __ldg(slot + t_nx * W + lane) : -1;
  while (has) {
    const int64_t t = t_nx;
    const int c_lo = r0_nx * 32 * U;
    const int c_hi = min(r1_nx * 32 * U, n16);
    int s = s_next;
    has = next_piece(t_nx, r0_nx, r1_nx);
    s_next = (has && lane < W) ? __ldg(slot + t_nx * W + lane) : -1;

    int64_t srow = s, lim = cap;  // the row in its storage and that storage's capacity
    if (RT::kRegions && s >= 0) {
      srow = storage_row<RT>(s, first_row);
      lim = storage_rows<RT>(lane, cap, s_rv);
    }
    const bool keep = s >= 0 && srow < lim;
    cap_err |= __any_sync(kFull, s >= 0 && srow >= lim);
    const unsigned dmask = __ballot_sync(kFull, keep);
    const int nd = __popc(dmask);
    const int rk = nth_set_bit_of_lane(dmask, lane);
    const int my_row = __shfl_sync(kFull, (int)srow, rk & 31);  // lane i: row of i-th destination
    float my_w = 0.0f;
    if constexpr (WEIGHTED) {
      const float wl = lane < W ? __ldg(w + t * W + lane) : 0.0f;
      my_w = __shfl_sync(kFull, wl, rk & 31);               // and its weight
    }
    // lane i's destination row as an address, formed once per token (for
    // per-rank regions: its region's base plus the row inside it)
    const uint4* my_src = y;
    if (rk >= 0)
      my_src = reinterpret_cast<const uint4*>(rows_base<RT>(
                   s_rv, rk, reinterpret_cast<uint8_t*>(const_cast<uint4*>(y)))) +
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
            if (dg + q < nd && c < c_hi) v[q][u] = ld_stream_v4(ybase[q] + c);
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
  // The dependent launch is released once every warp of the CTA is done (as
  // in the bulk-copy dispatch).  Released by each warp as it finished, the
  // next step's kernels launched while other warps still summed rows: back
  // to back over buffer sets larger than L2 (no flush), layout + dispatch +
  // combine at T=4096, H=7168 took 124.0 us per step instead of 119.6 us.
  __syncthreads();
  pdl_launch_dependents();
  if (cap_err && lane == 0 && status != nullptr) atomicOr(status, EP_STATUS_CAPACITY);
}

}  // namespace

// As many CTAs as fit on the device at once, each warp one range of rounds;
// fewer CTAs when there are fewer rounds than warp slots (one round a warp).
template <typename K, class RT>
cudaError_t launch_combine_regs(K kern, const void* y, const int32_t* slot, const float* w,
                                int64_t T, int H, int W, int64_t capacity_rows, void* out,
                                int32_t* status, cudaStream_t stream, const RT& rt) {
  static int cache[128];
  const int per_sm = occupancy_cached(kern, kCThreads, cache);
  const int64_t most = (int64_t)device_sm_count() * per_sm;
  const int n16 = H / 8;
  const int rpt = (n16 + 32 * kCU - 1) / (32 * kCU);
  const int64_t want = (T * rpt * 32 + kCThreads - 1) / kCThreads;
  const int grid = (int)(want < most ? want : most);
  return launch_pdl(kern, dim3(grid < 1 ? 1 : grid), dim3(kCThreads), 0, stream,
                    static_cast<const uint4*>(y), slot, w, T, n16, rpt, W, capacity_rows,
                    static_cast<uint4*>(out), status, rt);
}

cudaError_t launch_combine(const void* y, const int32_t* slot, int64_t T, int H, int W,
                           int64_t capacity_rows, void* out, int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_combine_regs(combine_kernel<kCU, false, OneBuffer>, y, slot, nullptr, T, H, W,
                             capacity_rows, out, status, stream, OneBuffer{});
}

cudaError_t launch_combine_regions(const RankRegions& y_regions, const int32_t* slot, int64_t T,
                                   int H, int W, void* out, int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_combine_regs(combine_kernel<kCU, false, RankRegions>, nullptr, slot, nullptr, T,
                             H, W, /*capacity_rows=*/0, out, status, stream, y_regions);
}

cudaError_t launch_combine_weighted(const void* y, const int32_t* slot, const float* w, int64_t T,
                                    int H, int C, int64_t capacity_rows, void* out,
                                    int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_combine_regs(combine_kernel<kCU, true, OneBuffer>, y, slot, w, T, H, C,
                             capacity_rows, out, status, stream, OneBuffer{});
}

}  // namespace ep
