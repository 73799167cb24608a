// FP8 cast and transposed cast of the expert-major rows, with the amax fused:
// the expert GEMMs take the rows of expert e (rows off[e] .. off[e+1]-1 of the
// receive buffer) as FP8, row-major for the forward product and transposed
// for the weight gradient.  ("Optimized rocm specific multicast transpose
// kernel", ROCm/TransformerEngine pull 586: both casts of every expert's
// tensor in one launch, amax fused into the same pass, pad-16 rows.)
//
// One launch, grid-stride over tiles of 64 rows x 256 columns that never
// straddle two experts.  Tile order: the tiles of expert 0, then of expert 1,
// ... (ceil(n_e / 64) row tiles x H / 256 column tiles each); inside an
// expert column tile by column tile, its row tiles in order, so that the CTAs
// running at the same time fill whole stretches of the same transposed rows
// (measured: Zipf dsv3 186.7 -> 177.9 us, qwen 192.1 -> 184.5 us, dsv3 166.1
// -> 164.6 us against row tile by row tile); a CTA finds its expert by binary
// search over the tile prefix sums, which every CTA computes once in shared
// memory.
// Per tile:
//   1. each thread loads 8 vectors of 8 bf16 (a warp reads one 512-byte row
//      segment per vector), forms the fp32 products x * s_e, packs their e4m3
//      codes (cvt.rn.satfinite.e4m3x2.f32), stores them to the row-major
//      output (8 bytes per vector) and into a (swizzled) shared tile, and keeps
//      the largest |x|;
//   2. after a barrier, each thread takes 16 rows x 4 columns of the code
//      tile (16 four-byte reads), transposes the 4x4 byte blocks with byte
//      permutes, and stores 4 rows of the transposed output, 16 bytes each;
//   3. the tile's amax (warp and CTA max) goes to amax[e] with an atomic max
//      on the float's bit pattern (valid for values >= 0).
// Two shared code tiles are used in turn, so one barrier per tile (between
// the cast and the transposed cast) suffices: the next tile's cast writes the
// other code tile while slower warps still read this one, and the barrier
// after that cast orders it before the tile after next overwrites this one
// (measured: dsv3 164.7 -> 163.4 us, qwen 185.0 -> 183.7 us, Zipf dsv3
// 176.5 -> 174.8 us against a barrier after each transposed cast).
#include "ep_device.cuh"

namespace ep {
namespace {

constexpr int kCtRows = 64;
constexpr int kCtCols = 256;
constexpr int kCtThreads = 256;
// Shared code tile, [64 rows][256 code bytes].  Phase 2 reads 4-byte words of
// 16 rows at a time with the four row groups (rows 16 apart) in one warp; with
// plain rows those four would hit one bank.  So row r keeps its 4-byte word g
// at g ^ ((r >> 4) << 3): each row group's words move by a different multiple
// of 8 banks, and a phase-2 read touches 32 distinct banks.  (Phase 1 writes
// 8-byte pairs of words; the XOR leaves bits 0-2, so a pair stays aligned.)
// (With rows padded to 264 bytes instead, phase 2 ran 4-way bank conflicts;
// the swizzle took dsv3 from 170.4 to 163.8 us.)
constexpr int kCtStride = kCtCols;  // row stride (bytes)
__device__ __forceinline__ int ct_word(int r, int g) { return g ^ ((r >> 4) << 3); }

__device__ __forceinline__ uint32_t e4m3x2_ct(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Exclusive prefix sums of per-expert quantities over E experts (block-wide):
// s_rt[e] = sum of ceil(n / 64), s_tb[e] = sum of n rounded up to 16.
__device__ void expert_prefixes(const int32_t* __restrict__ off, int E, int32_t* s_rt,
                                int32_t* s_tb, int32_t* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int per = (E + nthreads - 1) / nthreads;
  const int lo = tid * per, hi = min(lo + per, E);
  int a = 0, b = 0;
  for (int e = lo; e < hi; ++e) {
    const int n = max(off[e + 1] - off[e], 0);
    a += (n + kCtRows - 1) / kCtRows;
    b += (n + 15) & ~15;
  }
  int ia = a, ib = b;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ya = __shfl_up_sync(kFull, ia, o), yb = __shfl_up_sync(kFull, ib, o);
    if (lane >= o) {
      ia += ya;
      ib += yb;
    }
  }
  if (lane == 31) {
    s_warp[warp] = ia;
    s_warp[32 + warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    const int va = lane < nwarps ? s_warp[lane] : 0, vb = lane < nwarps ? s_warp[32 + lane] : 0;
    int wa = va, wb = vb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ya = __shfl_up_sync(kFull, wa, o), yb = __shfl_up_sync(kFull, wb, o);
      if (lane >= o) {
        wa += ya;
        wb += yb;
      }
    }
    s_warp[lane] = wa - va;
    s_warp[32 + lane] = wb - vb;
  }
  __syncthreads();
  int ra = s_warp[warp] + ia - a, rb = s_warp[32 + warp] + ib - b;
  for (int e = lo; e < hi; ++e) {
    const int n = max(off[e + 1] - off[e], 0);
    s_rt[e] = ra;
    s_tb[e] = rb;
    ra += (n + kCtRows - 1) / kCtRows;
    rb += (n + 15) & ~15;
  }
  if (hi == E && lo < E) {
    s_rt[E] = ra;
    s_tb[E] = rb;
  }
  if (E == 0 && tid == 0) s_rt[0] = s_tb[0] = 0;
  __syncthreads();
}

// Transposes a 4x4 byte block: in[r] holds row r (byte c = column c); out[c]
// holds column c (byte r = row r).
__device__ __forceinline__ void transpose4x4(const uint32_t (&in)[4], uint32_t (&out)[4]) {
  const uint32_t t0 = __byte_perm(in[0], in[1], 0x5140);  // r0c0 r1c0 r0c1 r1c1
  const uint32_t t1 = __byte_perm(in[0], in[1], 0x7362);  // r0c2 r1c2 r0c3 r1c3
  const uint32_t t2 = __byte_perm(in[2], in[3], 0x5140);
  const uint32_t t3 = __byte_perm(in[2], in[3], 0x7362);
  out[0] = __byte_perm(t0, t2, 0x5410);  // r0c0 r1c0 r2c0 r3c0
  out[1] = __byte_perm(t0, t2, 0x7632);
  out[2] = __byte_perm(t1, t3, 0x5410);
  out[3] = __byte_perm(t1, t3, 0x7632);
}

__global__ void __launch_bounds__(kCtThreads)
    cast_transpose_kernel(const uint4* __restrict__ y, const int32_t* __restrict__ off, int E,
                          int H, const float* __restrict__ scale, int64_t cap,
                          uint8_t* __restrict__ out_c, uint8_t* __restrict__ out_t,
                          float* __restrict__ amax, int32_t* __restrict__ status) {
  extern __shared__ __align__(16) uint8_t smem[];
  // two code tiles used in turn: the transposed cast of one tile and the cast
  // of the next need no barrier between them
  int32_t* s_rt = reinterpret_cast<int32_t*>(smem + 2 * kCtRows * kCtStride);  // [E + 1]
  int32_t* s_tb = s_rt + (E + 1);                                          // [E + 1]
  __shared__ int32_t s_warp[64];
  __shared__ float s_max[2][kCtThreads / 32];
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  expert_prefixes(off, E, s_rt, s_tb, s_warp);
  const int ct_n = H / kCtCols;
  const int64_t tiles = (int64_t)s_rt[E] * ct_n;
  const int n16 = H >> 3;

  int buf = 0;
  for (int64_t tau = blockIdx.x; tau < tiles; tau += gridDim.x) {
    uint8_t* const tile = smem + buf * (kCtRows * kCtStride);
    // the expert e whose tiles [s_rt[e] * ct_n, s_rt[e + 1] * ct_n) hold tau;
    // inside an expert the row tiles of one column tile come first, so the
    // CTAs working at once write whole stretches of the same transposed rows
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)s_rt[mid] * ct_n <= tau) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int64_t i_loc = tau - (int64_t)s_rt[e] * ct_n;
    const int rte = s_rt[e + 1] - s_rt[e];  // row tiles of expert e (>= 1 here)
    const int ct = (int)(i_loc / rte), rt = s_rt[e] + (int)(i_loc % rte);
    const int64_t r0 = off[e];
    if (r0 < 0 || (int64_t)off[e + 1] > cap) {  // rows outside the buffer: not read, not written
      if (tid == 0 && status != nullptr) atomicOr(status, EP_STATUS_CAPACITY);
      continue;
    }
    const int n = off[e + 1] - off[e];
    const int i0 = (rt - s_rt[e]) * kCtRows;
    const int nrows = min(kCtRows, n - i0);
    const int h0 = ct * kCtCols;
    const float s = scale[e];

    // 1. cast: 64 rows x 32 vectors of 8 columns, 8 vectors per thread, all
    //    loaded before the first is used
    float m = 0.0f;
    uint4 wv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int r = (tid + j * kCtThreads) >> 5, cv = tid & 31;
      wv[j] = r < nrows ? ld_stream_v4(y + (r0 + i0 + r) * n16 + (h0 >> 3) + cv)
                        : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int v = tid + j * kCtThreads;
      const int r = v >> 5, cv = v & 31;
      uint2 codes = make_uint2(0u, 0u);
      if (r < nrows) {
        const uint4 w = wv[j];
        const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
        uint32_t c[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a = __uint_as_float(wd[q] << 16), b = __uint_as_float(wd[q] & 0xffff0000u);
          m = fmaxf(m, fmaxf(fabsf(a), fabsf(b)));
          c[q] = e4m3x2_ct(__fmul_rn(a, s), __fmul_rn(b, s));
        }
        codes = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
        *reinterpret_cast<uint2*>(out_c + (r0 + i0 + r) * H + h0 + cv * 8) = codes;
      }
      // rows past the expert's end stay 0: they are the transposed padding
      *reinterpret_cast<uint2*>(tile + r * kCtStride + ct_word(r, 2 * cv) * 4) = codes;
    }
    // amax of the tile
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if (lane == 0) s_max[buf][warp] = m;
    __syncthreads();
    if (tid == 0) {
      float mm = 0.0f;
#pragma unroll
      for (int w = 0; w < kCtThreads / 32; ++w) mm = fmaxf(mm, s_max[buf][w]);
      atomicMax(reinterpret_cast<int*>(amax + e), __float_as_int(mm));
    }

    // 2. transposed cast: thread (column group cg, row group rg) -> 16 rows x 4 columns
    const int cg = tid >> 2, rg = tid & 3;
    const int ld = (n + 15) & ~15;
    const int ib = i0 + rg * 16;  // first transposed byte of this thread in each row
    if (ib < ld) {
      uint32_t col[4][4];  // col[c][k]: rows 4k .. 4k+3 of column c
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t in[4], out[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          in[q] = *reinterpret_cast<const uint32_t*>(tile + (rg * 16 + 4 * k + q) * kCtStride +
                                                     ct_word(rg * 16 + 4 * k + q, cg) * 4);
        transpose4x4(in, out);
#pragma unroll
        for (int c = 0; c < 4; ++c) col[c][k] = out[c];
      }
      uint8_t* tb = out_t + (int64_t)H * s_tb[e];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int h = h0 + cg * 4 + c;
        st_v4(reinterpret_cast<uint4*>(tb + (int64_t)h * ld + ib),
              make_uint4(col[c][0], col[c][1], col[c][2], col[c][3]));
      }
    }
    buf ^= 1;  // the next tile's cast writes the other code tile
  }
  pdl_launch_dependents();
}

}  // namespace

size_t cast_transpose_t_bytes(int64_t R, int E, int H) {
  return (size_t)H * (size_t)(R + 15 * (int64_t)E);
}

cudaError_t launch_cast_transpose(const void* y, const int32_t* expert_offset, int E, int H,
                                  const float* scale, int64_t capacity_rows, uint8_t* out_c,
                                  uint8_t* out_t, float* amax, int32_t* status,
                                  cudaStream_t stream) {
  const size_t smem = 2 * (size_t)kCtRows * kCtStride + 2 * sizeof(int32_t) * ((size_t)E + 1);
  static bool attr_set[128];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 128) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(cast_transpose_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(2 * (size_t)kCtRows * kCtStride + 2 * sizeof(int32_t) * (8192 + 1)));
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, cast_transpose_kernel, kCtThreads,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int grid = device_sm_count() * per_sm;
  return launch_pdl(cast_transpose_kernel, dim3(grid < 1 ? 1 : grid), dim3(kCtThreads), smem,
                    stream, static_cast<const uint4*>(y), expert_offset, E, H, scale,
                    capacity_rows, out_c, out_t, amax, status);
}

}  // namespace ep
