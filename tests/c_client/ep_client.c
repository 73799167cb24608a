/*
 * A plain C client of libep_gb300: no Python and no PyTorch in the process,
 * only include/ep_gb300.h and the shared library.
 *
 *   query mode (no GPU): size queries, status strings, and host-side argument
 *     checks that reject a call before anything reaches a GPU;
 *   gpu mode (built with -DEP_CLIENT_GPU): a small batch through
 *     ep_dispatch_with_layout and ep_combine with identity experts (the
 *     combine reads the dispatched rows back), then the same rows through
 *     ep_dispatch_regions (and ep_dispatch_regions_with_layout) and
 *     ep_combine_regions with every rank's rows in a cudaMalloc of its own.
 *     Every output row must then be d_t * x_t exactly, with d_t the number
 *     of distinct destination ranks of token t: small integer inputs make the
 *     fp32 sum and the bf16 rounding exact, so this closed form needs no
 *     reference implementation.  Then the expert-major path
 *     (ep_dispatch_experts_with_layout, ep_combine_weighted with unit
 *     weights), whose rows must be k * x_t.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ep_gb300.h"
#ifdef EP_CLIENT_GPU
#include <cuda_runtime.h>
#endif

static int fail(const char* what) {
  fprintf(stderr, "FAIL: %s\n", what);
  return 1;
}

static int query_mode(void) {
  if (ep_max_recv_rows(4096, 8, 8) != 32768) return fail("ep_max_recv_rows");
  if (ep_layout_workspace_bytes(4096, 8, 256) < 4096 * 4) return fail("ep_layout_workspace_bytes");
  if (strncmp(ep_status_string(EP_OK), "EP_OK", 5) != 0) return fail("ep_status_string");
  if (ep_dispatch_with_layout_launches(4096, 7168, 8, 8, EP_QUANT_BF16) != 2)
    return fail("ep_dispatch_with_layout_launches");
  /* rejected on the host: more than 32 ranks, E not a multiple of W, H % 8 */
  if (ep_dispatch_layout(NULL, 10, 8, 256, 33, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL) !=
      EP_ERR_INVALID_ARG)
    return fail("reject W = 33");
  if (ep_dispatch_layout(NULL, 10, 8, 100, 8, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL) !=
      EP_ERR_INVALID_ARG)
    return fail("reject E % W");
  if (ep_dispatch(NULL, NULL, NULL, 10, 12, 8, 8, NULL, 80, EP_QUANT_BF16, NULL, NULL, NULL, NULL,
                  NULL, NULL, NULL) != EP_ERR_UNSUPPORTED)
    return fail("reject H = 12");
  /* per-rank regions: no table, or more than 32 ranks */
  if (ep_dispatch_regions(NULL, NULL, NULL, 10, 256, 8, 8, NULL, NULL, NULL, EP_QUANT_BF16, NULL,
                          NULL) != EP_ERR_INVALID_ARG)
    return fail("reject regions without a table");
  if (ep_combine_regions(NULL, NULL, NULL, NULL, 10, 256, 33, NULL, NULL, NULL) !=
      EP_ERR_INVALID_ARG)
    return fail("reject 33 ranks of regions");
  if (ep_dispatch_regions_with_layout(NULL, NULL, NULL, 10, 256, 8, 64, 8, NULL, NULL, NULL, NULL,
                                      NULL, 0, NULL, EP_QUANT_BF16, NULL,
                                      NULL) != EP_ERR_INVALID_ARG)
    return fail("reject the one-call regions dispatch without its arguments");
  printf("query mode ok\n");
  return 0;
}

#ifdef EP_CLIENT_GPU
/* bf16 bits of a small integer (exact: at most 8 significant bits) */
static uint16_t bf16_of_int(int v) {
  float f = (float)v;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

#define CK(call)                                              \
  do {                                                        \
    if ((call) != cudaSuccess) return fail(#call);            \
  } while (0)

/* The expert-major path from C: ep_dispatch_experts_with_layout (one row per
   (token, expert) pair, 2800 pairs: the chunked layout whose dispatch claims
   tokens, bulk-copy rows of 1 KB) and ep_combine_weighted with unit weights,
   so that every output row must be k * x_t exactly. */
static int expert_major(void) {
  enum { T = 700, H = 512, E = 32, K = 4 };
  static int32_t idx[T * K];
  static float ones[T * K];
  static uint16_t x[T * H], out[T * H];
  uint32_t lcg = 777u;
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < K; ++j) {
      int e, dup;
      do {
        lcg = lcg * 1664525u + 1013904223u;
        e = (int)((lcg >> 8) % E);
        dup = 0;
        for (int i = 0; i < j; ++i) dup |= idx[t * K + i] == e;
      } while (dup);
      idx[t * K + j] = e;
      ones[t * K + j] = 1.0f;
    }
    for (int h = 0; h < H; ++h) x[t * H + h] = bf16_of_int((t * 5 + h) % 13 - 6);
  }
  const int64_t cap = (int64_t)T * K;
  const size_t ws_bytes = ep_layout_experts_workspace_bytes(T, K, E);
  void *dx, *dy, *dout, *dws;
  int32_t *didx, *dne, *doff, *dslot, *dsrc, *dst;
  float* dw;
  CK(cudaMalloc((void**)&dx, sizeof x));
  CK(cudaMalloc((void**)&didx, sizeof idx));
  CK(cudaMalloc((void**)&dw, sizeof ones));
  CK(cudaMalloc((void**)&dne, E * 4));
  CK(cudaMalloc((void**)&doff, (E + 1) * 4));
  CK(cudaMalloc((void**)&dslot, T * K * 4));
  CK(cudaMalloc((void**)&dws, ws_bytes));
  CK(cudaMalloc((void**)&dy, (size_t)cap * H * 2));
  CK(cudaMalloc((void**)&dsrc, (size_t)cap * 4));
  CK(cudaMalloc((void**)&dout, sizeof out));
  CK(cudaMalloc((void**)&dst, 4));
  CK(cudaMemset(dst, 0, 4));
  CK(cudaMemcpy(dx, x, sizeof x, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(didx, idx, sizeof idx, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dw, ones, sizeof ones, cudaMemcpyHostToDevice));
  int rc = ep_dispatch_experts_with_layout(dx, didx, dw, T, H, K, E, dne, doff, dslot, dws,
                                           ws_bytes, cap, EP_QUANT_BF16, dy, NULL, NULL, NULL,
                                           dsrc, dst, NULL);
  if (rc != EP_OK) return fail(ep_status_string(rc));
  rc = ep_combine_weighted(dy, dslot, dw, T, H, K, cap, dout, dst, NULL);
  if (rc != EP_OK) return fail(ep_status_string(rc));
  CK(cudaDeviceSynchronize());
  int32_t status = -1, off[E + 1];
  CK(cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(off, doff, sizeof off, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&status, dst, 4, cudaMemcpyDeviceToHost));
  if (status != 0) return fail("status word (expert-major)");
  if (off[E] != T * K) return fail("expert_offset[E] != T * k");
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      if (out[t * H + h] != bf16_of_int(K * ((t * 5 + h) % 13 - 6))) {
        fprintf(stderr, "token %d column %d\n", t, h);
        return fail("weighted combine of the expert-major rows != k * x");
      }
  printf("gpu mode ok: expert-major T=%d H=%d E=%d k=%d\n", T, H, E, K);
  return 0;
}

static int gpu_mode(void) {
  enum { T = 300, H = 256, E = 64, K = 4, W = 8 };
  const int Er = E / W;
  static int32_t idx[T * K];
  static float wts[T * K];
  static uint16_t x[T * H], out[T * H];
  int d[T];
  uint32_t lcg = 12345u;
  for (int t = 0; t < T; ++t) { /* k distinct experts per token */
    for (int j = 0; j < K; ++j) {
      int e, dup;
      do {
        lcg = lcg * 1664525u + 1013904223u;
        e = (int)((lcg >> 8) % E);
        dup = 0;
        for (int i = 0; i < j; ++i) dup |= idx[t * K + i] == e;
      } while (dup);
      idx[t * K + j] = e;
      wts[t * K + j] = 1.0f / K;
    }
    unsigned ranks = 0;
    for (int j = 0; j < K; ++j) ranks |= 1u << (idx[t * K + j] / Er);
    d[t] = __builtin_popcount(ranks);
    for (int h = 0; h < H; ++h) x[t * H + h] = bf16_of_int((t * 7 + h * 3) % 17 - 8);
  }
  const int64_t cap = ep_max_recv_rows(T, K, W);
  const size_t ws_bytes = ep_layout_workspace_bytes(T, W, E);
  void *dx, *dy, *dout, *dws;
  int32_t *didx, *dne, *dnr, *doff, *dslot, *dri, *dsrc, *dst;
  float *dw, *drw;
  CK(cudaMalloc((void**)&dx, sizeof x));
  CK(cudaMalloc((void**)&didx, sizeof idx));
  CK(cudaMalloc((void**)&dw, sizeof wts));
  CK(cudaMalloc((void**)&dne, E * 4));
  CK(cudaMalloc((void**)&dnr, W * 4));
  CK(cudaMalloc((void**)&doff, (W + 1) * 4));
  CK(cudaMalloc((void**)&dslot, T * W * 4));
  CK(cudaMalloc((void**)&dws, ws_bytes));
  CK(cudaMalloc((void**)&dy, (size_t)cap * H * 2));
  CK(cudaMalloc((void**)&dri, (size_t)cap * K * 4));
  CK(cudaMalloc((void**)&drw, (size_t)cap * K * 4));
  CK(cudaMalloc((void**)&dsrc, (size_t)cap * 4));
  CK(cudaMalloc((void**)&dout, sizeof out));
  CK(cudaMalloc((void**)&dst, 4));
  CK(cudaMemset(dst, 0, 4));
  CK(cudaMemcpy(dx, x, sizeof x, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(didx, idx, sizeof idx, cudaMemcpyHostToDevice));
  CK(cudaMemcpy(dw, wts, sizeof wts, cudaMemcpyHostToDevice));
  int rc = ep_dispatch_with_layout(dx, didx, dw, T, H, K, E, W, dne, dnr, doff, dslot, dws,
                                   ws_bytes, cap, EP_QUANT_BF16, dy, NULL, dri, drw, dsrc, dst,
                                   NULL);
  if (rc != EP_OK) return fail(ep_status_string(rc));
  rc = ep_combine(dy, dslot, T, H, W, cap, dout, dst, NULL);
  if (rc != EP_OK) return fail(ep_status_string(rc));
  CK(cudaDeviceSynchronize());
  int32_t off[W + 1], status = -1;
  CK(cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(off, doff, sizeof off, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&status, dst, 4, cudaMemcpyDeviceToHost));
  if (status != 0) return fail("status word");
  int R = 0;
  for (int t = 0; t < T; ++t) R += d[t];
  if (off[W] != R) return fail("rank_offset[W] != sum of d_t");
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      if (out[t * H + h] != bf16_of_int(d[t] * ((t * 7 + h * 3) % 17 - 8))) {
        fprintf(stderr, "token %d column %d\n", t, h);
        return fail("combine(dispatch(x)) != d_t * x");
      }

  /* the same rows into per-rank regions: one allocation per rank, sized to
     its rows, the table passed from host memory */
  ep_rank_region_t regions[W];
  const void* yreg[W];
  int64_t yrows[W];
  for (int r = 0; r < W; ++r) {
    const int64_t n = off[r + 1] - off[r];
    memset(&regions[r], 0, sizeof regions[r]);
    regions[r].rows = n;
    CK(cudaMalloc(&regions[r].recv_x, (size_t)(n > 0 ? n : 1) * H * 2));
    CK(cudaMalloc((void**)&regions[r].recv_src, (size_t)(n > 0 ? n : 1) * 4));
    yreg[r] = regions[r].recv_x;
    yrows[r] = n;
  }
  CK(cudaMemset(dout, 0, sizeof out));
  rc = ep_dispatch_regions(dx, didx, dw, T, H, K, W, dslot, doff, regions, EP_QUANT_BF16, dst,
                           NULL);
  if (rc != EP_OK) return fail(ep_status_string(rc));
  rc = ep_combine_regions(yreg, yrows, dslot, doff, T, H, W, dout, dst, NULL);
  if (rc != EP_OK) return fail(ep_status_string(rc));
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&status, dst, 4, cudaMemcpyDeviceToHost));
  if (status != 0) return fail("status word (regions)");
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      if (out[t * H + h] != bf16_of_int(d[t] * ((t * 7 + h * 3) % 17 - 8))) {
        fprintf(stderr, "token %d column %d\n", t, h);
        return fail("combine_regions(dispatch_regions(x)) != d_t * x");
      }
  for (int r = 0; r < W; ++r) { /* region r's source tokens ascend */
    const int64_t n = yrows[r];
    static int32_t src[T];
    if (n == 0) continue;
    CK(cudaMemcpy(src, regions[r].recv_src, (size_t)n * 4, cudaMemcpyDeviceToHost));
    for (int64_t i = 1; i < n; ++i)
      if (src[i] <= src[i - 1]) return fail("region rows out of token order");
  }
  /* layout and dispatch into the regions in one call: the same rows */
  for (int r = 0; r < W; ++r)
    if (yrows[r] > 0) CK(cudaMemset(regions[r].recv_x, 0, (size_t)yrows[r] * H * 2));
  CK(cudaMemset(dslot, 0xff, T * W * 4));
  CK(cudaMemset(dout, 0, sizeof out));
  rc = ep_dispatch_regions_with_layout(dx, didx, dw, T, H, K, E, W, dne, dnr, doff, dslot, dws,
                                       ws_bytes, regions, EP_QUANT_BF16, dst, NULL);
  if (rc != EP_OK) return fail(ep_status_string(rc));
  rc = ep_combine_regions(yreg, yrows, dslot, doff, T, H, W, dout, dst, NULL);
  if (rc != EP_OK) return fail(ep_status_string(rc));
  CK(cudaDeviceSynchronize());
  CK(cudaMemcpy(out, dout, sizeof out, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(&status, dst, 4, cudaMemcpyDeviceToHost));
  if (status != 0) return fail("status word (regions, one call)");
  for (int t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      if (out[t * H + h] != bf16_of_int(d[t] * ((t * 7 + h * 3) % 17 - 8))) {
        fprintf(stderr, "token %d column %d\n", t, h);
        return fail("combine_regions(dispatch_regions_with_layout(x)) != d_t * x");
      }
  printf("gpu mode ok: T=%d H=%d E=%d k=%d W=%d R=%d (one buffer and per-rank regions)\n", T, H, E,
         K, W, R);
  return expert_major();
}
#endif

int main(void) {
  if (query_mode()) return 1;
#ifdef EP_CLIENT_GPU
  if (gpu_mode()) return 1;
#endif
  return 0;
}
