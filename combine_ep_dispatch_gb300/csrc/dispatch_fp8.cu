// Dispatch of FP8 rows: each token row is quantised once, per 1x128 column
// block, to e4m3 codes with one fp32 scale, and the codes and scales are
// written to the receive row of every destination rank, with the metadata.
#include "dispatch_common.cuh"

namespace ep {
namespace {

constexpr int kDThreads = 256;
constexpr int kFp8U = 1;     // block quadruples per step
constexpr int kFp8MinB = 4;  // CTAs per SM the register allocation must allow

// Two fp32 values to two e4m3 codes, round to nearest even, saturating to
// +-448: `lo` goes to the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}


// max(|a|, |b|) per bf16 half (the sign bit of each half is the xor of the
// operands' signs and is cleared at the end).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest |x| of the 16 bf16 values in w[0..7], as fp32 (exact): a tree of
// packed |max| operations, then the larger half.
__device__ __forceinline__ float bf16x16_absmax(const uint32_t (&w)[8]) {
  const uint32_t m01 = absmax_bf16x2(w[0], w[1]), m23 = absmax_bf16x2(w[2], w[3]);
  const uint32_t m45 = absmax_bf16x2(w[4], w[5]), m67 = absmax_bf16x2(w[6], w[7]);
  const uint32_t m = absmax_bf16x2(absmax_bf16x2(m01, m23), absmax_bf16x2(m45, m67)) & 0x7fff7fffu;
  const uint32_t hi = m >> 16, lo = m & 0xffffu;
  return __uint_as_float((hi > lo ? hi : lo) << 16);
}

// fl(v / s), the IEEE quotient rounded to nearest even, from y = RN(1/s)
// with fused multiply-adds: q0 = RN(v y), then one correction
// q1 = RN(q0 - (s q0 - v) y) (P. Markstein, IBM J. Res. Dev. 34(1), 1990).
// For arbitrary fp32 operands a second correction is needed; here it is not.
// v is a bf16 value (significand V, at most 8 bits) and s = fl(M/7) * 2^j for
// the 8-bit significand M of the block's amax (block_scale), and every step
// commutes with scaling by a power of two while q0, q1 stay normal: q0 and q1
// are near v / s, and the residual s q0 - v is a multiple of 2^-137 for the
// scales allowed here, so it is exact even when subnormal.  The 255 x 128
// pairs (V, M) are then all the cases there are, and for each of them q1 is
// fl(V / S), checked exhaustively in exact rational arithmetic
// (tests/test_fp8_quotient.py).  q0 alone is wrong for a quarter of them.
// The residual is formed as s q - v and subtracted, which keeps the sign of a
// zero quotient.  Valid for 2^-80 <= s <= 2^100; a quotient below 2^-10, where
// q1 may underflow, has an e4m3 code of zero (with its sign) either way.
__device__ __forceinline__ float quotient_rn(float v, float s, float y) {
  const float q = __fmul_rn(v, y);
  const float r = __fmaf_rn(s, q, -v);
  return __fmaf_rn(-r, y, q);
}

// e4m3 codes of the 16 bf16 values in w[0..7] (element 2i in the low half of
// w[i]) divided by s > 0, packed little-endian into 16 bytes: the code of the
// IEEE-rounded fp32 quotient fl(v/s) rounded to e4m3 (nearest, ties to even,
// saturating to +-448).  y = RN(1/s).  Scales outside [2^-80, 2^100] take the
// IEEE division per value.
__device__ __forceinline__ uint4 e4m3x16_of_quotients(const uint32_t (&w)[8], float s, float y) {
  uint32_t c[8];
  if (s >= 0x1p-80f && s <= 0x1p100f) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float a = __uint_as_float(w[i] << 16), b = __uint_as_float(w[i] & 0xffff0000u);
      c[i] = e4m3x2(quotient_rn(a, s, y), quotient_rn(b, s, y));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      c[i] = e4m3x2(__fdiv_rn(__uint_as_float(w[i] << 16), s),
                    __fdiv_rn(__uint_as_float(w[i] & 0xffff0000u), s));
  }
  return make_uint4(c[0] | (c[1] << 16), c[2] | (c[3] << 16), c[4] | (c[5] << 16),
                    c[6] | (c[7] << 16));
}

// Scale s = fl(m / 448) of a block and y = RN(1/s), the reciprocal the exact
// quotient needs.  m is a bf16 value: m = M * 2^k with an 8-bit significand M,
// so m / 448 = (M / 7) * 2^(k - 6) and, while everything stays normal,
// s = fl(M / 7) * 2^(k - 6) and RN(1/s) = RN(1 / fl(M / 7)) * 2^(6 - k)
// exactly: rounding commutes with scaling by a power of two.  q7[i] = fl(M/7)
// and r7[i] = RN(1/q7[i]) for M = 128 + i are filled once per CTA by the IEEE
// division and reciprocal; blocks whose scale would leave [2^-80, 2^100]
// (biased exponent of m outside [56, 235]), or m = 0, take those operations
// directly.
__device__ __forceinline__ void block_scale(float m, const float* s_q7, const float* s_r7,
                                            float& s, float& y) {
  const uint32_t mb = __float_as_uint(m);
  const uint32_t e8 = mb >> 23;
  if (e8 >= 56u && e8 <= 235u) {
    const int i = (int)((mb >> 16) & 0x7fu);
    s = __fmul_rn(s_q7[i], __uint_as_float((e8 - 13u) << 23));   // * 2^(e8 - 140)
    y = __fmul_rn(s_r7[i], __uint_as_float((267u - e8) << 23));  // * 2^(140 - e8)
  } else {
    s = __fdiv_rn(m, 448.0f);
    y = s != 0.0f ? __frcp_rn(s) : 0.0f;
  }
}

// FP8 payload.  A 128-column block is 256 bytes of bf16 = 8 lanes x 32 bytes,
// so a warp covers four blocks per round (lanes 8b..8b+7 for block b).  Per
// block: amax over the block (an 8-lane max reduction), scale = amax / 448
// (IEEE division), codes of x / scale (e4m3x16_of_quotients).  A token row is
// split into `nseg` segments of block quadruples, one warp per (token,
// segment), so that small batches still fill the GPU; each segment is
// quantised once and its codes and scales are stored to every destination.
template <int U, class RT>
__global__ void __launch_bounds__(kDThreads, kFp8MinB)
    dispatch_fp8_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ topk_idx,
                        const float* __restrict__ topk_w, int64_t T, int H, int k, int W,
                        int32_t* slot, int64_t cap, uint8_t* __restrict__ recv_x,
                        float* __restrict__ recv_scale, int32_t* __restrict__ recv_topk_idx,
                        float* __restrict__ recv_topk_w, int32_t* __restrict__ recv_src,
                        int nseg, int per_seg, int32_t* __restrict__ status, int x_early,
                        Finalize fin, RT rt) {
  __shared__ float s_q7[128], s_r7[128];
  __shared__ int32_t s_dst[kDThreads / 32][32];  // per warp: rows of the unit's destinations
  // per warp: ranks of the unit's destinations (per-rank regions only)
  __shared__ int32_t s_drank[RT::kRegions ? kDThreads / 32 : 1][32];
  __shared__ typename RT::View s_rv;
  if (threadIdx.x < 128) {
    const float q = __fdiv_rn((float)(128 + threadIdx.x), 7.0f);
    s_q7[threadIdx.x] = q;
    s_r7[threadIdx.x] = __frcp_rn(q);
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  int32_t* const my_dst = s_dst[threadIdx.x >> 5];
  int32_t* const my_drank = s_drank[RT::kRegions ? threadIdx.x >> 5 : 0];
  const unsigned below = (1u << lane) - 1u;  // lanes under this one
  const int qb = lane >> 3, hl = lane & 7;  // block within the quad, lane within the block
  const int nb = H >> 7;
  const int n16 = H >> 3;
  const int nquad = (nb + 3) >> 2;
  const int64_t gwarp = ((int64_t)blockIdx.x * kDThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kDThreads) >> 5;
  const bool narrow = T * nseg < 0x7fffffffLL;  // 32-bit unit arithmetic suffices
  const int64_t units = T * nseg;
  bool cap_err = false;
  // The warp walks its steps (unit u, quad round q0) in order and issues the
  // loads of the next step (and, at a unit's last step, the next unit's slot
  // row) before working on the current one, so loads stay in flight while it
  // quantises and stores.
  auto split = [&](int64_t uu, int64_t& tt, int& sg, int& qs, int& qe) {
    tt = narrow ? (int64_t)((uint32_t)uu / (uint32_t)nseg) : uu / nseg;
    sg = (int)(uu - tt * nseg);
    qs = sg * per_seg;
    qe = (sg + 1) * per_seg < nquad ? (sg + 1) * per_seg : nquad;
  };
  auto load_step = [&](int64_t tt, int q, int qe, uint4 (&A)[U], uint4 (&C)[U]) {
    const uint4* src = x + tt * n16;
#pragma unroll
    for (int v = 0; v < U; ++v) {
      const int b = (q + v) * 4 + qb;
      A[v] = make_uint4(0u, 0u, 0u, 0u);
      C[v] = make_uint4(0u, 0u, 0u, 0u);
      if (q + v < qe && b < nb) {  // the lane's 32 contiguous bytes (L1-cached pair)
        A[v] = __ldg(src + b * 16 + hl * 2);
        C[v] = __ldg(src + b * 16 + hl * 2 + 1);
      }
    }
  };
  int64_t u = gwarp, t = 0;
  int seg = 0, q0 = 0, q_end = 0;
  uint4 A[U], C[U];
  int s_raw = -1;  // the current unit's slot entry of this lane
  // the first step's rows depend on x only: with x_early (this launch
  // directly follows the layout kernels, whose wait covered x's producer) they
  // are loaded before the wait
  if (u < units) {
    split(u, t, seg, q0, q_end);
    if (x_early) load_step(t, q0, q_end, A, C);
  }
  load_region_view(rt, W, s_rv);
  pdl_wait();
  // With a Finalize the slot table holds in-chunk positions: every CTA scans
  // the chunk counts first; the warp taking a token's first segment writes
  // its receive rows back (other segments may read either form).
  extern __shared__ int32_t s_base[];  // [C][W] with a Finalize
  __shared__ int32_t s_tot[32], s_off[33];
  const bool fin_mode = fin.chunk_rank != nullptr;  // uniform over the grid
  if (fin_mode) build_chunk_base(fin, W, s_base, s_tot, s_off);
  // each region's first global row: rank_offset, or (finishing the layout,
  // which writes rank_offset during this kernel) the CTA's own scan of it
  const int32_t first_row = fin_mode ? (RT::kRegions && lane < W ? s_off[lane] : 0)
                                     : region_first_row(rt, W, lane);
  // plain loads: with a Finalize the table is also written during the kernel
  auto slot_entry = [&](int64_t tt) { return lane < W ? slot[tt * W + lane] : -1; };
  if (u < units) {
    if (!x_early) load_step(t, q0, q_end, A, C);
    s_raw = slot_entry(t);
  }
  Dests d;
  d.nd = 0;
  d.my_row = -1;
  int sc_row = -1;  // lane (qb, hl): row of destination hl, which receives block qb's scale
  // per-rank regions: lane i's destination row (codes) and lane (qb, hl)'s
  // scale row, as addresses, formed once per unit
  uint8_t* reg_code_row = nullptr;
  float* reg_scale_row = nullptr;
  // Unit by unit; inside a unit, step by step.  Each step issues the loads
  // of the next one (the next unit's first step at a unit's last) before it
  // quantises and stores its own, so loads stay in flight during the
  // compute.  (Nested this way the unit's bookkeeping leaves the per-step
  // path: 13% fewer instructions than one loop over all steps.)
  while (u < units) {
    {  // the unit's destinations and metadata
      if (fin_mode && lane < W) {
        s_raw = final_slot(s_raw, t, lane, W, fin.shift, s_base, s_off);
        if (seg == 0) slot[t * W + lane] = s_raw;
      }
      int64_t srow = s_raw, lim = cap;  // the row in its storage and that storage's capacity
      if (RT::kRegions && s_raw >= 0) {
        srow = storage_row<RT>(s_raw, first_row);
        lim = storage_rows<RT>(lane, cap, s_rv);
      }
      const bool keep = s_raw >= 0 && srow < lim;
      const bool over = s_raw >= 0 && srow >= lim;
      const unsigned dmask = __ballot_sync(kFull, keep);
      // compact the destinations: lane i gets the row of the i-th one
      __syncwarp();  // the previous unit's rows have been read
      if (keep) {
        my_dst[__popc(dmask & below)] = (int)srow;
        if constexpr (RT::kRegions) my_drank[__popc(dmask & below)] = lane;
      }
      __syncwarp();
      d.nd = __popc(dmask);
      d.my_row = lane < d.nd ? my_dst[lane] : -1;
      d.my_rank = RT::kRegions && lane < d.nd ? my_drank[lane] : -1;
      d.cap_err = __any_sync(kFull, over);
      sc_row = hl < d.nd ? my_dst[hl] : -1;
      if constexpr (RT::kRegions) {
        reg_code_row = lane < d.nd ? s_rv.x[my_drank[lane]] + (uint64_t)(uint32_t)my_dst[lane] * (uint32_t)H
                                   : nullptr;
        reg_scale_row = hl < d.nd ? s_rv.scale[my_drank[hl]] + (uint64_t)(uint32_t)sc_row * (uint32_t)nb
                                  : nullptr;
      }
      if (seg == 0) {
        cap_err |= d.cap_err;
        carry_metadata<RT>(topk_idx, topk_w, t, k, d, recv_topk_idx, recv_topk_w, recv_src, lane,
                           &s_rv);
      }
    }
    // the next unit: the fixed stride (claiming units from a counter, as the
    // bf16 kernel claims tokens, measured 3 us slower here: ~12k small units
    // contend on one atomic)
    const int64_t un = u + nwarps;
    int64_t tn = t;
    int segn = 0, qsn = 0, qen = 0, s_rawn = -1;
    const bool has_next = un < units;
    if (has_next) split(un, tn, segn, qsn, qen);
    for (int q = q0; q < q_end; q += U) {
      uint4 A2[U], C2[U];
      if (q + U < q_end) {
        load_step(t, q + U, q_end, A2, C2);
      } else if (has_next) {
        load_step(tn, qsn, qen, A2, C2);
        s_rawn = slot_entry(tn);
      } else {
#pragma unroll
        for (int v = 0; v < U; ++v) A2[v] = C2[v] = make_uint4(0u, 0u, 0u, 0u);
      }
      uint4 codes[U];
      float sc[U];
#pragma unroll
      for (int v = 0; v < U; ++v) {
        const uint32_t w[8] = {A[v].x, A[v].y, A[v].z, A[v].w, C[v].x, C[v].y, C[v].z, C[v].w};
        float m = bf16x16_absmax(w);
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        float sv, yv;
        block_scale(m, s_q7, s_r7, sv, yv);
        sc[v] = sv;
        codes[v] = sv != 0.0f ? e4m3x16_of_quotients(w, sv, yv) : make_uint4(0u, 0u, 0u, 0u);
      }
      // Codes: every destination gets the lane's 16 bytes of each of its
      // blocks.  Scales: lane (qb, hl) writes block qb's scale to destinations
      // hl, hl + 8, ... (one store per step while there are at most 8).
#pragma unroll
      for (int v = 0; v < U; ++v) {
        if (q + v >= q_end) continue;  // warp-uniform
        const int b = (q + v) * 4 + qb;
        const bool has = b < nb;          // the last quadruple may be partial
        if constexpr (RT::kRegions) {
#pragma unroll 1
          for (int qq = 0; qq < d.nd; ++qq) {
            uint8_t* const xr = reinterpret_cast<uint8_t*>(
                __shfl_sync(kFull, reinterpret_cast<unsigned long long>(reg_code_row), qq));
            if (has) st_v4(reinterpret_cast<uint4*>(xr + b * 128 + hl * 16), codes[v]);
          }
          if (has) {
            if (reg_scale_row != nullptr) reg_scale_row[b] = sc[v];
            for (int j = hl + 8; j < d.nd; j += 8)
              s_rv.scale[my_drank[j]][(uint64_t)(uint32_t)my_dst[j] * (uint32_t)nb + b] = sc[v];
          }
        } else {
          uint8_t* const xb = recv_x + b * 128 + hl * 16;
#pragma unroll 1
          for (int qq = 0; qq < d.nd; ++qq) {
            const uint32_t row = (uint32_t)__shfl_sync(kFull, d.my_row, qq);
            if (has) st_v4(reinterpret_cast<uint4*>(xb + (uint64_t)row * (uint32_t)H), codes[v]);
          }
          if (has) {
            if (sc_row >= 0) recv_scale[(uint64_t)(uint32_t)sc_row * (uint32_t)nb + b] = sc[v];
            for (int j = hl + 8; j < d.nd; j += 8)
              recv_scale[(uint64_t)(uint32_t)my_dst[j] * (uint32_t)nb + b] = sc[v];
          }
        }
      }
#pragma unroll
      for (int v = 0; v < U; ++v) {
        A[v] = A2[v];
        C[v] = C2[v];
      }
    }
    u = un;
    t = tn;
    seg = segn;
    q0 = qsn;
    q_end = qen;
    s_raw = s_rawn;
  }
  if (fin_mode) finish_expert_totals(fin);
  __syncthreads();  // the CTA releases the dependent launch when all its warps are done
  pdl_launch_dependents();
  if (cap_err && lane == 0 && status != nullptr) atomicOr(status, EP_STATUS_CAPACITY);
}

}  // namespace

template <class RT>
cudaError_t launch_dispatch_fp8(const void* x, const int32_t* topk_idx, const float* topk_w,
                                int64_t T, int H, int k, int W, const int32_t* slot,
                                int64_t capacity_rows, void* recv_x, float* recv_scale,
                                int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                                int32_t* status, cudaStream_t stream, int x_early,
                                const Finalize& fin, const RT& rt) {
  if (T == 0) return cudaSuccess;
  const uint4* x4 = static_cast<const uint4*>(x);
  // segments per token: enough (token, segment) units to give every resident warp
  // a few, but no more segments than block quadruples
  auto kern = dispatch_fp8_kernel<kFp8U, RT>;
  static int cache[128];
  const int per_sm = occupancy_cached(kern, kDThreads, cache);
  const int64_t warps = (int64_t)device_sm_count() * per_sm * (kDThreads / 32);
  const int nquad = (H / 128 + 3) / 4;
  int nseg = (int)((2 * warps + T - 1) / T);
  nseg = nseg < 1 ? 1 : (nseg > nquad ? nquad : nseg);
  // segments of whole rounds of 2 quads (the kernel's unroll: no half-empty
  // rounds), and no empty segments
  const int per_seg = ((nquad + nseg - 1) / nseg + kFp8U - 1) / kFp8U * kFp8U;
  nseg = (nquad + per_seg - 1) / per_seg;
  const int64_t units = T * nseg;
  const int64_t grid = (units * 32 + kDThreads - 1) / kDThreads < device_sm_count() * per_sm
                           ? (units * 32 + kDThreads - 1) / kDThreads
                           : (int64_t)device_sm_count() * per_sm;
  const size_t smem =
      fin.chunk_rank != nullptr ? ((size_t)(fin.C * W) * sizeof(int32_t) + 15) & ~size_t(15) : 0;
  // the kernel writes the slot table only with a Finalize
  return launch_pdl(kern, dim3((unsigned)(grid < 1 ? 1 : grid)), dim3(kDThreads), smem, stream, x4,
                    topk_idx, topk_w, T, H, k, W, const_cast<int32_t*>(slot), capacity_rows,
                    static_cast<uint8_t*>(recv_x), recv_scale, recv_topk_idx, recv_topk_w, recv_src,
                    nseg, per_seg, status, x_early, fin, rt);
}

template cudaError_t launch_dispatch_fp8<OneBuffer>(
    const void*, const int32_t*, const float*, int64_t, int, int, int, const int32_t*, int64_t,
    void*, float*, int32_t*, float*, int32_t*, int32_t*, cudaStream_t, int, const Finalize&,
    const OneBuffer&);
template cudaError_t launch_dispatch_fp8<RankRegions>(
    const void*, const int32_t*, const float*, int64_t, int, int, int, const int32_t*, int64_t,
    void*, float*, int32_t*, float*, int32_t*, int32_t*, cudaStream_t, int, const Finalize&,
    const RankRegions&);

}  // namespace ep
