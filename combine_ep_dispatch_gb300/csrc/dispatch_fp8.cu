// Dispatch of FP8 rows: each token row is quantised once, per 1x128 column
// block, to e4m3 codes with one fp32 scale, and the codes and scales are
// written to the receive row of every destination rank, with the metadata.
#include "dispatch_common.cuh"

namespace ep {
namespace {

constexpr int kDThreads = 256;

// Two fp32 values to two e4m3 codes, round to nearest even, saturating to
// +-448: `lo` goes to the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// e4m3 codes of v / s (s > 0), exactly as if v / s were first rounded to fp32
// by IEEE division and that quotient then rounded to e4m3 (nearest, ties to
// even, saturating to +-448).
//
// The code is a monotonic function of the fp32 quotient, so a cheap quotient
// q = v * r, r = rcp.approx(s) (at most 1 ulp off, the product adds half an
// ulp: a few ulps from the correctly rounded quotient), gives the same code
// unless a rounding boundary of e4m3 lies within a few ulps of q.  For
// 2^-6 <= |q| (normal e4m3) the boundaries, midpoints between neighbouring
// e4m3 values (1 + (2j+1)/16) * 2^e, are exactly the fp32 values whose low 20
// mantissa bits are 0x80000, so "near a boundary" is a bit test on q with a
// margin of 16 bit patterns each way.  Values with 0 < |q| < 2^-6 (e4m3
// subnormals) and values near a boundary take the IEEE division; that is a
// few values in 10^5 for normally distributed rows.
__device__ __forceinline__ bool e4m3_needs_division(float q) {
  const uint32_t m = __float_as_uint(q) & 0x7fffffffu;
  return (m - 1u) < 0x3c7fffffu || ((m + (16u - 0x80000u)) & 0xfffffu) <= 32u;
}

__device__ __noinline__ uint32_t e4m3_by_division(float v, float s) {
  return e4m3x2(__fdiv_rn(v, s), 0.0f) & 0xffu;
}

__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// Largest |x| of the 16 bf16 values in w[0..7], as fp32 (exact).
__device__ __forceinline__ float bf16x16_absmax(const uint32_t (&w)[8]) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t a = w[i] & 0x7fff7fffu, r;
    asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(m));
    m = r;
  }
  const uint32_t hi = m >> 16, lo = m & 0xffffu;
  return __uint_as_float((hi > lo ? hi : lo) << 16);
}

// Codes of the 16 bf16 values in w[0..7] (element 2i low half of w[i]) divided
// by s > 0, packed little-endian into 16 bytes.
__device__ __forceinline__ uint4 e4m3x16_of_quotients(const uint32_t (&w)[8], float s) {
  const float r = rcp_approx(s);
  const bool fast = s >= 1.17549435e-38f && r < 3.0e38f;  // normal s, finite 1/s
  uint32_t out[4];
  uint32_t slow = fast ? 0u : 0xffffu;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float q0 = __uint_as_float(w[i] << 16) * r;
    const float q1 = __uint_as_float(w[i] & 0xffff0000u) * r;
    const uint32_t c = e4m3x2(q0, q1);
    if (i & 1)
      out[i >> 1] |= c << 16;
    else
      out[i >> 1] = c;
    slow |= (e4m3_needs_division(q0) ? 1u : 0u) << (2 * i);
    slow |= (e4m3_needs_division(q1) ? 1u : 0u) << (2 * i + 1);
  }
  if (slow) {
    for (int e = 0; e < 16; ++e) {
      if (slow & (1u << e)) {
        const uint32_t bits = (e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16);
        const uint32_t code = e4m3_by_division(__uint_as_float(bits), s);
        const int sh = 8 * (e & 3);
        out[e >> 2] = (out[e >> 2] & ~(0xffu << sh)) | (code << sh);
      }
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
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
        if (q0 + v < q_end && b < nb) {  // the lane's 32 contiguous bytes (L1-cached pair)
          a = __ldg(src + b * 16 + hl * 2);
          c = __ldg(src + b * 16 + hl * 2 + 1);
        }
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        float m = bf16x16_absmax(w);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        const float s = __fdiv_rn(m, 448.0f);
        sc[v] = s;
        codes[v] = s != 0.0f ? e4m3x16_of_quotients(w, s) : make_uint4(0u, 0u, 0u, 0u);
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

}  // namespace

cudaError_t launch_dispatch_fp8(const void* x, const int32_t* topk_idx, const float* topk_w,
                                int64_t T, int H, int k, int W, const int32_t* slot,
                                int64_t capacity_rows, void* recv_x, float* recv_scale,
                                int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                                int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const uint4* x4 = static_cast<const uint4*>(x);
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
