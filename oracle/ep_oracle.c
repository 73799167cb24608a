/*
 * CPU oracle for MoE expert-parallel dispatch / combine.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * statement of what the dispatch/combine path computes.  It is used by the
 * tests, by the package's smoke check and by the benchmark's CPU baseline, and
 * by nothing else: the product path never calls it.  It shares no code, header,
 * table or helper with the CUDA library.
 *
 * Sources (page title, section):
 *  [mori]  "perf(ep): optimize IntraNode dispatch kernel for MI350X"
 *          (ROCm/mori pull 586): Technical Details §1 "Cached routing" --
 *          destination PE of an expert = expert / experts-per-rank, one copy per
 *          (token, destination PE) after per-PE deduplication; §4 "Vectorized
 *          metadata copies" -- the k weights and k indices of a token travel with
 *          its row; "Remaining gap" -- combine receives pre-routed rows and
 *          accumulates them per token.
 *  [yotta] "Optimizing Distributed Inference Kernels for AMD DEVELOPER
 *          CHALLENGE 2025: All-to-All, GEMM-ReduceScatter, and AllGather-GEMM",
 *          §3.1 -- dispatch sends each token's row to every rank that hosts one
 *          of its experts, combine brings the rows back and reduces them.
 *  [te]    "Optimized rocm specific multicast transpose kernel" (ROCm/
 *          TransformerEngine pull 586): the FP8 cast and transposed cast of
 *          every expert's tensor in one launch, with the amax fused.
 *  Readings where the pages leave a step open (fixed by the problem statement
 *  of this library, not by the pages):
 *   - receive rows of rank r form one contiguous region starting at the
 *     exclusive prefix sum of the per-rank row counts; inside a region rows are
 *     in ascending source-token order;
 *   - combine is the unweighted sum of the token's rows, taken in ascending
 *     rank order, in fp32 starting from +0, rounded once to bf16 (RNE);
 *   - FP8: per row and per 128-column block, scale = amax / 448 (fp32 IEEE
 *     division), code = e4m3 round-to-nearest-even with saturation of
 *     (x / scale) (fp32 IEEE division); scale == 0 gives all-zero codes;
 *   - expert ids outside [0, E) are ignored and flag EP_REF_STATUS_BAD_EXPERT;
 *     receive rows at or beyond the capacity are not written and flag
 *     EP_REF_STATUS_CAPACITY.
 *
 * Floating point: compiled with -ffp-contract=off and without fast-math, so
 * every + and / below is one IEEE binary32 operation in round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define EP_REF_STATUS_BAD_EXPERT 1
#define EP_REF_STATUS_CAPACITY 2

#define EP_REF_QUANT_BF16 0
#define EP_REF_QUANT_FP8 1

/* ------------------------------------------------------------------ numbers */

/* bf16 -> fp32: the bf16 bits are the top half of the fp32 bits. */
float ep_ref_f32_from_bf16(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* fp32 -> bf16, round to nearest, ties to even, on the bit pattern: add half an
 * ulp of the kept part (minus one when the kept part is even) and truncate.
 * NaN keeps its sign and becomes a quiet NaN. */
uint16_t ep_ref_bf16_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7fffu + keep_lsb;
  return (uint16_t)(u >> 16);
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities, NaN = S.1111.111, largest finite 448 = 1.75 * 2^8, smallest
 * normal 2^-6, subnormals k * 2^-9 for k = 1..7. */
float ep_ref_f32_from_e4m3(uint8_t c) {
  int s = c >> 7, e = (c >> 3) & 0xf, m = c & 7;
  float v;
  if (e == 0xf && m == 7) return s ? -NAN : NAN;
  if (e == 0)
    v = ldexpf((float)m, -9);
  else
    v = ldexpf((float)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* fp32 -> e4m3, round to nearest, ties to even, saturating at +-448 (the
 * "satfinite" rule: anything whose magnitude is 448 or more maps to 448).
 * Subnormal range (|v| < 2^-6): the code is |v| / 2^-9 rounded to an integer.
 * Normal range: |v| = m * 2^(e-3) with m in [8, 16); m rounded to an integer
 * gives the 3 mantissa bits (m = 16 carries into the exponent).
 * Both roundings use nearbyintf in the default round-to-nearest-even mode, and
 * both scalings by powers of two are exact. */
uint8_t ep_ref_e4m3_from_f32(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  float a = fabsf(v);
  if (isnan(v)) return (uint8_t)(sign | 0x7f);
  if (a >= 448.0f) return (uint8_t)(sign | 0x7e);
  if (a < 0.015625f) { /* 2^-6 */
    int q = (int)nearbyintf(ldexpf(a, 9));
    return (uint8_t)(sign | q); /* q = 8 is the smallest normal, code 0x08 */
  }
  int e;
  (void)frexpf(a, &e);        /* a = f * 2^e, f in [0.5, 1) */
  e -= 1;                     /* a = g * 2^e, g in [1, 2) */
  int m = (int)nearbyintf(ldexpf(a, 3 - e)); /* in [8, 16] */
  if (m == 16) {
    m = 8;
    e += 1;
  }
  int code = ((e + 7) << 3) | (m - 8);
  if (code > 0x7e) code = 0x7e;
  return (uint8_t)(sign | code);
}

void ep_ref_bf16_from_f32_array(const float* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ep_ref_bf16_from_f32(in[i]);
}

void ep_ref_e4m3_from_f32_array(const float* in, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ep_ref_e4m3_from_f32(in[i]);
}

/* ------------------------------------------------------------------- layout */

/* Routing layout.
 *  counts per expert: number of (t, j) with topk_idx[t][j] == e (before
 *    deduplication);
 *  D(t): the set of ranks r = e / (E / W) over the token's valid expert ids;
 *  counts per rank: number of tokens t with r in D(t) (after deduplication);
 *  rank_offset[0..W]: exclusive prefix sum of the per-rank counts
 *    (rank_offset[W] = R, the total number of receive rows);
 *  slot[t][r]: for r in D(t), rank_offset[r] + #{t' < t : r in D(t')};
 *    otherwise -1.
 * Returns 0, or -1 on invalid arguments. */
int ep_ref_layout(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                  int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                  int32_t* rank_offset, int32_t* slot, int32_t* status) {
  if (T < 0 || k < 1 || E < 1 || W < 1 || W > 32 || E % W != 0) return -1;
  int Er = E / W;
  int32_t st = 0;
  for (int e = 0; e < E; ++e) num_tokens_per_expert[e] = 0;
  for (int r = 0; r < W; ++r) num_tokens_per_rank[r] = 0;

  /* per token: the set D(t) as a flag per rank, and the counts */
  for (int64_t t = 0; t < T; ++t) {
    int in_d[32];
    for (int r = 0; r < W; ++r) in_d[r] = 0;
    for (int j = 0; j < k; ++j) {
      int32_t e = topk_idx[t * k + j];
      if (e < 0 || e >= E) {
        st |= EP_REF_STATUS_BAD_EXPERT;
        continue;
      }
      num_tokens_per_expert[e] += 1;
      in_d[e / Er] = 1;
    }
    for (int r = 0; r < W; ++r) {
      slot[t * W + r] = in_d[r] ? 0 : -1; /* mark membership; filled below */
      if (in_d[r]) num_tokens_per_rank[r] += 1;
    }
  }

  rank_offset[0] = 0;
  for (int r = 0; r < W; ++r) rank_offset[r + 1] = rank_offset[r] + num_tokens_per_rank[r];

  /* per rank: walk tokens in ascending order and hand out consecutive rows */
  for (int r = 0; r < W; ++r) {
    int32_t next = rank_offset[r];
    for (int64_t t = 0; t < T; ++t) {
      if (slot[t * W + r] >= 0) slot[t * W + r] = next++;
    }
  }
  if (status) *status |= st;
  return 0;
}

/* ----------------------------------------------------------------- dispatch */

/* Dispatch: for every token t and every rank r in D(t) (slot[t][r] >= 0), in
 * ascending r, the receive row s = slot[t][r] gets
 *   bf16:  recv_x[s][:] = x[t][:]  (bit copy)
 *   fp8:   per 128-column block b: amax = max |x[t][128b + i]|,
 *          scale = amax / 448, recv_scale[s][b] = scale,
 *          recv_x[s][128b + i] = e4m3(x[t][128b + i] / scale)  (0 if scale == 0)
 *   recv_topk_idx[s][:] = topk_idx[t][:], recv_topk_w[s][:] = topk_w[t][:],
 *   recv_src[s] = t.
 * Rows s >= cap are skipped and flag EP_REF_STATUS_CAPACITY. */
int ep_ref_dispatch(const uint16_t* x, const int32_t* topk_idx, const float* topk_w, int64_t T,
                    int H, int k, int W, const int32_t* slot, int64_t cap, int quant,
                    void* recv_x, float* recv_scale, int32_t* recv_topk_idx, float* recv_topk_w,
                    int32_t* recv_src, int32_t* status) {
  if (T < 0 || H < 1 || k < 1 || W < 1 || W > 32 || cap < 0) return -1;
  if (quant != EP_REF_QUANT_BF16 && quant != EP_REF_QUANT_FP8) return -1;
  if (quant == EP_REF_QUANT_FP8 && H % 128 != 0) return -1;
  int nb = H / 128;
  int32_t st = 0;
  for (int64_t t = 0; t < T; ++t) {
    for (int r = 0; r < W; ++r) {
      int32_t s = slot[t * W + r];
      if (s < 0) continue;
      if ((int64_t)s >= cap) {
        st |= EP_REF_STATUS_CAPACITY;
        continue;
      }
      if (quant == EP_REF_QUANT_BF16) {
        uint16_t* dst = (uint16_t*)recv_x + (int64_t)s * H;
        for (int h = 0; h < H; ++h) dst[h] = x[t * H + h];
      } else {
        uint8_t* dst = (uint8_t*)recv_x + (int64_t)s * H;
        for (int b = 0; b < nb; ++b) {
          float amax = 0.0f;
          for (int i = 0; i < 128; ++i) {
            float a = fabsf(ep_ref_f32_from_bf16(x[t * H + b * 128 + i]));
            if (a > amax) amax = a;
          }
          float scale = amax / 448.0f;
          recv_scale[(int64_t)s * nb + b] = scale;
          for (int i = 0; i < 128; ++i) {
            float v = ep_ref_f32_from_bf16(x[t * H + b * 128 + i]);
            dst[b * 128 + i] = (scale == 0.0f) ? 0 : ep_ref_e4m3_from_f32(v / scale);
          }
        }
      }
      for (int j = 0; j < k; ++j) {
        recv_topk_idx[(int64_t)s * k + j] = topk_idx[t * k + j];
        recv_topk_w[(int64_t)s * k + j] = topk_w[t * k + j];
      }
      recv_src[s] = (int32_t)t;
    }
  }
  if (status) *status |= st;
  return 0;
}

/* ------------------------------------------------------------------ combine */

/* Combine: out[t][h] = bf16( ((+0 + y[s_0][h]) + y[s_1][h]) + ... ) over the
 * ranks r in ascending order with s_r = slot[t][r] >= 0; fp32 additions; a token
 * with no rows gives +0.  Rows s >= cap are skipped and flag
 * EP_REF_STATUS_CAPACITY. */
int ep_ref_combine(const uint16_t* y, const int32_t* slot, int64_t T, int H, int W, int64_t cap,
                   uint16_t* out, float* acc_scratch, int32_t* status) {
  if (T < 0 || H < 1 || W < 1 || W > 32 || cap < 0) return -1;
  int32_t st = 0;
  for (int64_t t = 0; t < T; ++t) {
    for (int h = 0; h < H; ++h) acc_scratch[h] = 0.0f;
    for (int r = 0; r < W; ++r) {
      int32_t s = slot[t * W + r];
      if (s < 0) continue;
      if ((int64_t)s >= cap) {
        st |= EP_REF_STATUS_CAPACITY;
        continue;
      }
      const uint16_t* row = y + (int64_t)s * H;
      for (int h = 0; h < H; ++h) acc_scratch[h] = acc_scratch[h] + ep_ref_f32_from_bf16(row[h]);
    }
    for (int h = 0; h < H; ++h) out[t * H + h] = ep_ref_bf16_from_f32(acc_scratch[h]);
  }
  if (status) *status |= st;
  return 0;
}

/* --------------------------------------------------------- local expert ids */

/* Local-id metadata (dispatch option): in receive row s of rank r (rows
 * rank_offset[r] <= s < rank_offset[r+1]), an expert id e of the row's token is
 * replaced by its index among rank r's experts, e - r * (E / W), when e is a
 * valid id hosted by rank r, and by -1 otherwise.  Applied in place to the
 * verbatim ids of rows [0, min(R, cap)). */
int ep_ref_localize_ids(int32_t* recv_topk_idx, int64_t cap, int k, int E, int W,
                        const int32_t* rank_offset) {
  if (k < 1 || E < 1 || W < 1 || W > 32 || E % W != 0 || cap < 0) return -1;
  int Er = E / W;
  for (int r = 0; r < W; ++r) {
    for (int64_t s = rank_offset[r]; s < rank_offset[r + 1] && s < cap; ++s) {
      for (int j = 0; j < k; ++j) {
        int32_t e = recv_topk_idx[s * k + j];
        int hosted = e >= 0 && e < E && e / Er == r;
        recv_topk_idx[s * k + j] = hosted ? e - r * Er : -1;
      }
    }
  }
  return 0;
}

/* ------------------------------------------------------ expert-major layout */

/* Expert-major layout: one receive row per valid (token, expert slot) pair,
 * grouped by expert.  counts per expert as in ep_ref_layout; expert_offset[0..E]
 * = exclusive prefix sum of the counts; slot[t][j] = expert_offset[e] + (number
 * of pairs (t', j') before (t, j) in (token, then j) order with the same expert
 * e = topk_idx[t][j]) for a valid e, else -1.  Rank r's experts r*Er..(r+1)*Er-1
 * are consecutive, so rank r's rows are one range as well.  This is the
 * per-expert receive layout of the recv kernel in "Optimizing Distributed
 * Inference Kernels for AMD DEVELOPER CHALLENGE 2025" (section 3.1, item 1:
 * rows of local expert e start at e times a per-expert maximum), with each
 * expert's rows packed by a scan of the counts instead of a fixed per-expert
 * capacity, and in token order. */
int ep_ref_layout_experts(const int32_t* topk_idx, int64_t T, int k, int E,
                          int32_t* num_tokens_per_expert, int32_t* expert_offset, int32_t* slot,
                          int32_t* next_scratch, int32_t* status) {
  if (T < 0 || k < 1 || E < 1) return -1;
  int32_t st = 0;
  for (int e = 0; e < E; ++e) num_tokens_per_expert[e] = 0;
  for (int64_t i = 0; i < T * k; ++i) {
    int32_t e = topk_idx[i];
    if (e < 0 || e >= E) {
      st |= EP_REF_STATUS_BAD_EXPERT;
      continue;
    }
    num_tokens_per_expert[e] += 1;
  }
  expert_offset[0] = 0;
  for (int e = 0; e < E; ++e) expert_offset[e + 1] = expert_offset[e] + num_tokens_per_expert[e];
  for (int e = 0; e < E; ++e) next_scratch[e] = expert_offset[e];
  for (int64_t t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      int32_t e = topk_idx[t * k + j];
      slot[t * k + j] = (e < 0 || e >= E) ? -1 : next_scratch[e]++;
    }
  }
  if (status) *status |= st;
  return 0;
}

/* ------------------------------------------------------- weighted combine */

/* Weighted combine over a slot table of C columns: out[t][h] =
 * bf16( fma(w[t][C-1], y[s_{C-1}][h], ... fma(w[t][0], y[s_0][h], +0)) ) over the
 * columns c in ascending order with s_c = slot[t][c] >= 0 (rows >= cap skipped
 * and flagged), each step one fused multiply-add rounded once (fmaf).  With the
 * expert-major slot table and w = topk_w this is the gate-weighted sum of the
 * token's expert outputs; with weights 1 it is the plain combine. */
int ep_ref_combine_weighted(const uint16_t* y, const int32_t* slot, const float* w, int64_t T,
                            int H, int C, int64_t cap, uint16_t* out, float* acc_scratch,
                            int32_t* status) {
  if (T < 0 || H < 1 || C < 1 || cap < 0) return -1;
  int32_t st = 0;
  for (int64_t t = 0; t < T; ++t) {
    for (int h = 0; h < H; ++h) acc_scratch[h] = 0.0f;
    for (int c = 0; c < C; ++c) {
      int32_t s = slot[t * C + c];
      if (s < 0) continue;
      if ((int64_t)s >= cap) {
        st |= EP_REF_STATUS_CAPACITY;
        continue;
      }
      const float wt = w[t * C + c];
      const uint16_t* row = y + (int64_t)s * H;
      for (int h = 0; h < H; ++h) acc_scratch[h] = fmaf(wt, ep_ref_f32_from_bf16(row[h]), acc_scratch[h]);
    }
    for (int h = 0; h < H; ++h) out[t * H + h] = ep_ref_bf16_from_f32(acc_scratch[h]);
  }
  if (status) *status |= st;
  return 0;
}

/* ------------------------------------------------- FP8 cast and transpose */

/* Cast and transposed cast of the expert-major rows ("Optimized rocm specific
 * multicast transpose kernel", ROCm/TransformerEngine pull 586: an FP8 cast and
 * an FP8 transposed cast of every expert's tensor in one launch, with the amax
 * fused).  Expert e owns rows off[e] .. off[e+1]-1 of y (n_e rows of H); with
 * the expert's scale s_e, every element gets code = e4m3(fl(x * s_e)) (fp32
 * product rounded to nearest even, then e4m3 round to nearest even with
 * saturation, as the dispatch encoder):
 *   out_c[row][h] = code            (row-major, rows as in y),
 *   out_t[tb_e + h * ld_e + i] = code of row off[e] + i, column h, where
 *     ld_e = n_e rounded up to a multiple of 16 and tb_e = H * (ld_0 + ... +
 *     ld_{e-1}); the padding bytes i >= n_e are 0,
 *   amax[e] = max(amax[e], max |x| over the expert's rows).
 * The caller zeroes amax for a fresh maximum. */
int ep_ref_cast_transpose(const uint16_t* y, const int32_t* off, int E, int H, const float* scale,
                          uint8_t* out_c, uint8_t* out_t, float* amax) {
  if (E < 1 || H < 1) return -1;
  int64_t tb = 0;
  for (int e = 0; e < E; ++e) {
    const int64_t r0 = off[e], n = (int64_t)off[e + 1] - off[e];
    if (n < 0) return -1;
    const int64_t ld = (n + 15) / 16 * 16;
    float m = amax[e];
    for (int64_t i = 0; i < ld; ++i) {
      for (int h = 0; h < H; ++h) {
        uint8_t code = 0;
        if (i < n) {
          const float x = ep_ref_f32_from_bf16(y[(r0 + i) * H + h]);
          const float q = x * scale[e];
          code = ep_ref_e4m3_from_f32(q);
          out_c[(r0 + i) * H + h] = code;
          const float a = fabsf(x);
          if (a > m) m = a;
        }
        out_t[tb + (int64_t)h * ld + i] = code;
      }
    }
    amax[e] = m;
    tb += (int64_t)H * ld;
  }
  return 0;
}
