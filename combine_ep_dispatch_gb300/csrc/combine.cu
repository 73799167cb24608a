// Combine: one warp per token gathers the token's receive rows and sums them in
// fp32 in ascending rank order from +0, then rounds once to bf16.
#include "ep_device.cuh"

namespace ep {
namespace {

#ifndef EP_COMBINE_U
#define EP_COMBINE_U 2
#endif
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

// Combine through the bulk-copy (TMA) engine, for W <= 8.  The work unit of a
// warp is (token, column chunk of kCChunk bytes).  Lane 0 loads the chunk of
// each of the token's rows into a private shared-memory stage with one bulk
// copy per row, kCStages units ahead of the one being summed; the warp then
// sums the stage's rows in ascending rank order (each lane 16-byte pieces of
// the chunk) and stores the bf16 result.  Deep look-ahead with few threads
// keeps enough bytes in flight to stream the rows at full bandwidth.
#ifndef EP_COMBINE_STAGES
#define EP_COMBINE_STAGES 3
#endif
#ifndef EP_COMBINE_CHUNK_BYTES
#define EP_COMBINE_CHUNK_BYTES 2048
#endif
#ifndef EP_COMBINE_SMEM_BUDGET
#define EP_COMBINE_SMEM_BUDGET (200 * 1024)
#endif
#ifndef EP_COMBINE_MAX_WARPS
#define EP_COMBINE_MAX_WARPS 8
#endif
constexpr int kCStages = EP_COMBINE_STAGES;
constexpr uint32_t kCChunk = EP_COMBINE_CHUNK_BYTES;
constexpr int kCMaxRows = 8;
constexpr uint32_t kCStageBytes = kCMaxRows * kCChunk;
constexpr int kCBarBytes = 1024;
constexpr int kCSmemBudget = EP_COMBINE_SMEM_BUDGET;
constexpr int kCMaxWarps = EP_COMBINE_MAX_WARPS;

__global__ void __launch_bounds__(kCMaxWarps * 32, 1)
    combine_tma_kernel(const uint8_t* __restrict__ y, const int32_t* __restrict__ slot, int64_t T,
                       uint32_t row_bytes, int W, int64_t cap, uint8_t* __restrict__ out,
                       int32_t* __restrict__ status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta_warps = blockDim.x >> 5;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem) + warp * kCStages;  // < 256 bytes
  int* nd_ring = reinterpret_cast<int*>(smem + 256) + warp * kCStages;    // < 128 bytes
  int* rows = reinterpret_cast<int*>(smem + 512) + warp * kCMaxRows;       // < 256 bytes
  uint8_t* buf = smem + kCBarBytes + (size_t)warp * kCStages * kCStageBytes;
  if (lane == 0) {
    for (int s = 0; s < kCStages; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  pdl_wait();

  const int64_t gw = (int64_t)blockIdx.x * cta_warps + warp;
  const int64_t NW = (int64_t)gridDim.x * cta_warps;
  const int64_t n_tok = gw < T ? (T - 1 - gw) / NW + 1 : 0;
  const int nch = (int)((row_bytes + kCChunk - 1) / kCChunk);
  const int64_t n_units = n_tok * nch;

  // issue side (lane 0 only): the next unit to load and its token's rows
  int64_t issued = 0;
  int nd_issue = 0;
  bool cap_err = false, timed_out = false;
  auto issue_next = [&]() {
    const int64_t jt = issued / nch;
    const int c = (int)(issued - jt * nch);
    if (c == 0) {
      const int64_t t = gw + jt * NW;
      nd_issue = 0;
#pragma unroll
      for (int r = 0; r < kCMaxRows; ++r) {
        const int s = r < W ? __ldg(slot + t * W + r) : -1;
        if (s >= 0 && (int64_t)s < cap) rows[nd_issue++] = s;
        cap_err |= s >= 0 && (int64_t)s >= cap;
      }
    }
    const int st = (int)(issued % kCStages);
    const uint32_t off = (uint32_t)c * kCChunk;
    const uint32_t bytes = row_bytes - off < kCChunk ? row_bytes - off : kCChunk;
    nd_ring[st] = nd_issue;
    mbar_arrive_expect_tx(&full[st], (uint32_t)nd_issue * bytes);
    for (int q = 0; q < nd_issue; ++q)
      bulk_load(buf + st * kCStageBytes + q * kCChunk, y + (int64_t)rows[q] * row_bytes + off,
                bytes, &full[st]);
    ++issued;
  };
  if (lane == 0)
    while (issued < n_units && issued < kCStages) issue_next();

  int64_t u = 0;
  for (; u < n_units; ++u) {
    const int st = (int)(u % kCStages);
    const uint32_t parity = (uint32_t)((u / kCStages) & 1);
    bool ok = true;
    if (lane == 0) ok = mbar_wait_bounded(&full[st], parity);
    if (!__shfl_sync(kFull, ok, 0)) {
      timed_out = true;
      break;
    }
    const int nd = nd_ring[st];
    const int64_t jt = u / nch;
    const int c = (int)(u - jt * nch);
    const int64_t t = gw + jt * NW;
    const uint32_t off = (uint32_t)c * kCChunk;
    const uint32_t bytes = row_bytes - off < kCChunk ? row_bytes - off : kCChunk;
    const uint8_t* sb = buf + st * kCStageBytes;
    uint4* dst = reinterpret_cast<uint4*>(out + t * row_bytes + off);
#pragma unroll 4
    for (uint32_t p = lane; p < bytes / 16; p += 32) {
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
      uint4 v[kCMaxRows];
#pragma unroll
      for (int q = 0; q < kCMaxRows; ++q)
        if (q < nd) v[q] = *reinterpret_cast<const uint4*>(sb + q * kCChunk + p * 16);
#pragma unroll
      for (int q = 0; q < kCMaxRows; ++q)
        if (q < nd) add_bf16x8(acc, v[q]);
      st_v4(dst + p, make_uint4(bf16x2_rn(acc[0], acc[1]), bf16x2_rn(acc[2], acc[3]),
                                bf16x2_rn(acc[4], acc[5]), bf16x2_rn(acc[6], acc[7])));
    }
    __syncwarp();  // every lane has read the stage: it may be refilled
    if (lane == 0 && issued < n_units) issue_next();
  }
  if (lane == 0) {
    // loads still landing in shared memory must finish before the CTA exits
    for (int64_t q = u; q < issued; ++q)
      (void)mbar_wait_bounded(&full[q % kCStages], (uint32_t)((q / kCStages) & 1));
  }
  __syncwarp();
  pdl_launch_dependents();
  if (lane == 0 && status != nullptr) {
    if (cap_err) atomicOr(status, EP_STATUS_CAPACITY);
    if (timed_out) atomicOr(status, EP_STATUS_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_combine(const void* y, const int32_t* slot, int64_t T, int H, int W,
                           int64_t capacity_rows, void* out, int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const uint32_t row_bytes = (uint32_t)H * 2u;
  const int cta_warps_fit = (int)(kCSmemBudget / ((size_t)kCStages * kCStageBytes));
  if (!EP_FORCE_LSU && W <= kCMaxRows && row_bytes >= 1024 && cta_warps_fit >= 1) {
    const int cta_warps = cta_warps_fit < kCMaxWarps ? cta_warps_fit : kCMaxWarps;
    const size_t smem = kCBarBytes + (size_t)cta_warps * kCStages * kCStageBytes;
    static bool attr_set[128];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 128 && !attr_set[dev]) {
      cudaError_t e = cudaFuncSetAttribute(combine_tma_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kCBarBytes + kCSmemBudget);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
    const int64_t want = (T + cta_warps - 1) / cta_warps;
    const int64_t sms = device_sm_count();
    const int grid = (int)(want < sms ? want : sms);
    return launch_pdl(combine_tma_kernel, dim3(grid < 1 ? 1 : grid), dim3(cta_warps * 32), smem,
                      stream, static_cast<const uint8_t*>(y), slot, T, row_bytes, W,
                      capacity_rows, static_cast<uint8_t*>(out), status);
  }
  auto kern = combine_kernel<EP_COMBINE_U>;
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
