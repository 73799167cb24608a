// Combine: one warp per token gathers the token's receive rows and sums them in
// fp32 in ascending rank order from +0, then rounds once to bf16.
#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kCThreads = 256;

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

// Lane l handles 16-byte chunks l, l+32, ... of the hidden dimension.  For a
// round of U chunks the loads of up to 8 destination rows are all issued before
// the first addition (8*U loads in flight per lane); the additions then run in
// ascending rank order, which fixes the rounding of the sum.
template <int U>
__global__ void __launch_bounds__(kCThreads)
    combine_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ slot, int64_t T, int n16,
                   int W, int64_t cap, uint4* __restrict__ out, int32_t* __restrict__ status) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int64_t gwarp = ((int64_t)blockIdx.x * kCThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kCThreads) >> 5;
  bool cap_err = false;
  for (int64_t t = gwarp; t < T; t += nwarps) {
    int s = -1;
    if (lane < W) s = __ldg(slot + t * W + lane);
    const bool keep = s >= 0 && (int64_t)s < cap;
    cap_err |= __any_sync(kFull, s >= 0 && (int64_t)s >= cap);
    const unsigned dmask = __ballot_sync(kFull, keep);
    const int nd = __popc(dmask);
    const int r = nth_set_bit_of_lane(dmask, lane);
    const int my_row = __shfl_sync(kFull, s, r & 31);  // lane i: row of i-th destination
    uint4* dst = out + t * n16;
    for (int c0 = 0; c0 < n16; c0 += 32 * U) {
      float acc[U][8];
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
      for (int dg = 0; dg < nd; dg += 8) {
        int rows[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) rows[q] = __shfl_sync(kFull, my_row, (dg + q) & 31);
        uint4 v[8][U];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const int c = c0 + u * 32 + lane;
            v[q][u] = make_uint4(0u, 0u, 0u, 0u);
            if (dg + q < nd && c < n16) v[q][u] = ld_stream_v4(y + (int64_t)rows[q] * n16 + c);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (dg + q < nd) {
#pragma unroll
            for (int u = 0; u < U; ++u) add_bf16x8(acc[u], v[q][u]);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < n16) {
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

}  // namespace

cudaError_t launch_combine(const void* y, const int32_t* slot, int64_t T, int H, int W,
                           int64_t capacity_rows, void* out, int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  auto kern = combine_kernel<2>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kCThreads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t want = (T * 32 + kCThreads - 1) / kCThreads;
  const int64_t most = (int64_t)device_sm_count() * per_sm;
  const int grid = (int)(want < most ? want : most);
  return launch_pdl(kern, dim3(grid < 1 ? 1 : grid), dim3(kCThreads), 0, stream,
                    static_cast<const uint4*>(y), slot, T, H / 8, W, capacity_rows,
                    static_cast<uint4*>(out), status);
}

}  // namespace ep
