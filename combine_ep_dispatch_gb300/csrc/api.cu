// C ABI of the library: argument checks on the host, then kernel launches.
// Nothing here allocates, synchronises or keeps per-call state.
#include <stdint.h>

#include "dispatch_common.cuh"

namespace ep {

int device_sm_count() {
  static int cache[128];  // per device ordinal; 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 128) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace ep

namespace {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kMaxRows = 0x7fffffffLL;  // receive rows are int32

inline int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

int from_cuda(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

}  // namespace

extern "C" {

size_t ep_layout_workspace_bytes(int64_t T, int W, int E) {
  if (T < 0 || W < 1 || W > 32 || E < 1) return 0;
  return ep::layout_workspace_bytes(T, W, E);
}

int64_t ep_max_recv_rows(int64_t T, int k, int W) {
  if (T < 0 || k < 1 || W < 1) return -1;
  return T * min64(k, W);
}

namespace {

int check_layout(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                 const int32_t* num_tokens_per_expert, const int32_t* num_tokens_per_rank,
                 const int32_t* rank_offset, const int32_t* slot, const void* workspace,
                 size_t workspace_bytes, const int32_t* status) {
  if (T < 0 || k < 1 || W < 1 || W > 32 || E < 1 || E > 8192 || E % W != 0)
    return EP_ERR_INVALID_ARG;
  if (T * min64(k, W) > kMaxRows || T > kMaxRows / W) return EP_ERR_UNSUPPORTED;
  if (!num_tokens_per_expert || !num_tokens_per_rank || !rank_offset || !workspace)
    return EP_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !slot)) return EP_ERR_INVALID_ARG;
  if (workspace_bytes < ep::layout_workspace_bytes(T, W, E)) return EP_ERR_WORKSPACE;
  if (!aligned(topk_idx, 4) || !aligned(num_tokens_per_expert, 4) ||
      !aligned(num_tokens_per_rank, 4) || !aligned(rank_offset, 4) || !aligned(slot, 4) ||
      !aligned(workspace, 16) || !aligned(status, 4))
    return EP_ERR_MISALIGNED;
  return EP_OK;
}

int check_dispatch(const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T, int H,
                   int k, int W, const int32_t* slot, int64_t capacity_rows, int quant,
                   const void* recv_x, const float* recv_scale, const int32_t* recv_topk_idx,
                   const float* recv_topk_w, const int32_t* recv_src, const int32_t* status) {
  if (T < 0 || H < 1 || k < 1 || W < 1 || W > 32 || capacity_rows < 0 || capacity_rows > kMaxRows)
    return EP_ERR_INVALID_ARG;
  if (quant != EP_QUANT_BF16 && quant != EP_QUANT_FP8_E4M3_B128) return EP_ERR_INVALID_ARG;
  if (quant == EP_QUANT_BF16 && H % 8 != 0) return EP_ERR_UNSUPPORTED;
  if (quant == EP_QUANT_FP8_E4M3_B128 && H % 128 != 0) return EP_ERR_UNSUPPORTED;
  if (T > kMaxRows / W) return EP_ERR_UNSUPPORTED;
  if (T > 0 && (!x || !topk_idx || !topk_w || !slot)) return EP_ERR_INVALID_ARG;
  if (capacity_rows > 0 && !recv_x) return EP_ERR_INVALID_ARG;
  if (capacity_rows > 0 && quant == EP_QUANT_FP8_E4M3_B128 && !recv_scale)
    return EP_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv_x, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
      !aligned(slot, 4) || !aligned(recv_scale, 4) || !aligned(recv_topk_idx, 4) ||
      !aligned(recv_topk_w, 4) || !aligned(recv_src, 4) || !aligned(status, 4))
    return EP_ERR_MISALIGNED;
  return EP_OK;
}

}  // namespace

int ep_dispatch_layout(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                       int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                       int32_t* rank_offset, int32_t* slot, void* workspace,
                       size_t workspace_bytes, int32_t* status, ep_stream_t stream) {
  const int rc = check_layout(topk_idx, T, k, E, W, num_tokens_per_expert, num_tokens_per_rank,
                              rank_offset, slot, workspace, workspace_bytes, status);
  if (rc != EP_OK) return rc;
  return from_cuda(ep::launch_layout(topk_idx, T, k, E, W, num_tokens_per_expert,
                                     num_tokens_per_rank, rank_offset, slot, workspace, status,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

int ep_dispatch(const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T, int H,
                int k, int W, const int32_t* slot, int64_t capacity_rows, int quant, void* recv_x,
                float* recv_scale, int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                int32_t* status, ep_stream_t stream) {
  const int rc = check_dispatch(x, topk_idx, topk_w, T, H, k, W, slot, capacity_rows, quant,
                                recv_x, recv_scale, recv_topk_idx, recv_topk_w, recv_src, status);
  if (rc != EP_OK) return rc;
  return from_cuda(ep::launch_dispatch(x, topk_idx, topk_w, T, H, k, W, slot, capacity_rows, quant,
                                       recv_x, recv_scale, recv_topk_idx, recv_topk_w, recv_src,
                                       status, reinterpret_cast<cudaStream_t>(stream)));
}

int ep_dispatch_with_layout_launches(int64_t T, int H, int k, int W, int quant) {
  if (T < 0 || H < 1 || k < 1 || W < 1 || W > 32) return -1;
  if (quant != EP_QUANT_BF16 && quant != EP_QUANT_FP8_E4M3_B128) return -1;
  return ep::dispatch_with_layout_launches(T, H, k, W, quant);
}

int ep_dispatch_with_layout(const void* x, const int32_t* topk_idx, const float* topk_w,
                            int64_t T, int H, int k, int E, int W,
                            int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                            int32_t* rank_offset, int32_t* slot, void* workspace,
                            size_t workspace_bytes, int64_t capacity_rows, int quant,
                            void* recv_x, float* recv_scale, int32_t* recv_topk_idx,
                            float* recv_topk_w, int32_t* recv_src, int32_t* status,
                            ep_stream_t stream) {
  int rc = check_layout(topk_idx, T, k, E, W, num_tokens_per_expert, num_tokens_per_rank,
                        rank_offset, slot, workspace, workspace_bytes, status);
  if (rc != EP_OK) return rc;
  rc = check_dispatch(x, topk_idx, topk_w, T, H, k, W, slot, capacity_rows, quant, recv_x,
                      recv_scale, recv_topk_idx, recv_topk_w, recv_src, status);
  if (rc != EP_OK) return rc;
  return from_cuda(ep::launch_dispatch_with_layout(
      x, topk_idx, topk_w, T, H, k, E, W, num_tokens_per_expert, num_tokens_per_rank, rank_offset,
      slot, workspace, capacity_rows, quant, recv_x, recv_scale, recv_topk_idx, recv_topk_w,
      recv_src, status, reinterpret_cast<cudaStream_t>(stream)));
}

int ep_dispatch_fused(const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T,
                      int H, int k, int E, int W, int32_t* num_tokens_per_expert,
                      int32_t* num_tokens_per_rank, int32_t* rank_offset, int32_t* slot,
                      int64_t capacity_rows, void* recv_x, int32_t* recv_topk_idx,
                      float* recv_topk_w, int32_t* recv_src, int32_t* status, ep_stream_t stream) {
  if (T < 0 || H < 1 || k < 1 || W < 1 || W > 32 || E < 1 || E > 8192 || E % W != 0 ||
      capacity_rows < 0 || capacity_rows > kMaxRows)
    return EP_ERR_INVALID_ARG;
  if (T > ep::fused_max_tokens() || k > 16 || H % 8 != 0) return EP_ERR_UNSUPPORTED;
  if (!num_tokens_per_expert || !num_tokens_per_rank || !rank_offset) return EP_ERR_INVALID_ARG;
  if (T > 0 && (!x || !topk_idx || !topk_w || !slot)) return EP_ERR_INVALID_ARG;
  if (capacity_rows > 0 && !recv_x) return EP_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv_x, 16) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
      !aligned(slot, 4) || !aligned(num_tokens_per_expert, 4) || !aligned(num_tokens_per_rank, 4) ||
      !aligned(rank_offset, 4) || !aligned(recv_topk_idx, 4) || !aligned(recv_topk_w, 4) ||
      !aligned(recv_src, 4) || !aligned(status, 4))
    return EP_ERR_MISALIGNED;
  return from_cuda(ep::launch_dispatch_fused(x, topk_idx, topk_w, T, H, k, E, W,
                                             num_tokens_per_expert, num_tokens_per_rank,
                                             rank_offset, slot, capacity_rows, recv_x,
                                             recv_topk_idx, recv_topk_w, recv_src, status,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int ep_localize_expert_ids(int32_t* recv_topk_idx, const int32_t* rank_offset,
                           int64_t capacity_rows, int k, int E, int W, ep_stream_t stream) {
  if (k < 1 || W < 1 || W > 32 || E < 1 || E % W != 0 || capacity_rows < 0 ||
      capacity_rows > kMaxRows)
    return EP_ERR_INVALID_ARG;
  if (!rank_offset || (capacity_rows > 0 && !recv_topk_idx)) return EP_ERR_INVALID_ARG;
  if (!aligned(recv_topk_idx, 4) || !aligned(rank_offset, 4)) return EP_ERR_MISALIGNED;
  if (capacity_rows == 0) return EP_OK;
  return from_cuda(ep::launch_localize_ids(recv_topk_idx, rank_offset, capacity_rows, k, E, W,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int ep_combine(const void* y, const int32_t* slot, int64_t T, int H, int W, int64_t capacity_rows,
               void* out, int32_t* status, ep_stream_t stream) {
  if (T < 0 || H < 1 || W < 1 || W > 32 || capacity_rows < 0 || capacity_rows > kMaxRows)
    return EP_ERR_INVALID_ARG;
  if (H % 8 != 0) return EP_ERR_UNSUPPORTED;
  if (T > kMaxRows / W) return EP_ERR_UNSUPPORTED;
  if (T > 0 && (!slot || !out)) return EP_ERR_INVALID_ARG;
  if (T > 0 && capacity_rows > 0 && !y) return EP_ERR_INVALID_ARG;
  if (!aligned(y, 16) || !aligned(out, 16) || !aligned(slot, 4) || !aligned(status, 4))
    return EP_ERR_MISALIGNED;
  return from_cuda(ep::launch_combine(y, slot, T, H, W, capacity_rows, out, status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// The kernels' table of W receive regions, after checking each region.
int region_table(const ep_rank_region_t* regions, int W, int quant, const int32_t* rank_offset,
                 ep::RankRegions* rt) {
  if (W < 1 || W > 32 || !regions || !rank_offset) return EP_ERR_INVALID_ARG;
  const bool fp8 = quant == EP_QUANT_FP8_E4M3_B128;
  *rt = ep::RankRegions{};
  for (int r = 0; r < W; ++r) {
    const ep_rank_region_t& g = regions[r];
    if (g.rows < 0 || g.rows > kMaxRows) return EP_ERR_INVALID_ARG;
    if (g.rows > 0 && (!g.recv_x || (fp8 && !g.recv_scale))) return EP_ERR_INVALID_ARG;
    if (!aligned(g.recv_x, 16) || !aligned(g.recv_scale, 4) || !aligned(g.recv_topk_idx, 4) ||
        !aligned(g.recv_topk_w, 4) || !aligned(g.recv_src, 4))
      return EP_ERR_MISALIGNED;
    rt->x[r] = static_cast<uint8_t*>(g.recv_x);
    rt->scale[r] = g.recv_scale;
    rt->topk_idx[r] = g.recv_topk_idx;
    rt->topk_w[r] = g.recv_topk_w;
    rt->src[r] = g.recv_src;
    rt->rows[r] = g.rows;
  }
  rt->rank_offset = rank_offset;
  if (!aligned(rank_offset, 4)) return EP_ERR_MISALIGNED;
  return EP_OK;
}
}  // namespace

int ep_dispatch_regions(const void* x, const int32_t* topk_idx, const float* topk_w, int64_t T,
                        int H, int k, int W, const int32_t* slot, const int32_t* rank_offset,
                        const ep_rank_region_t* regions, int quant, int32_t* status,
                        ep_stream_t stream) {
  ep::RankRegions rt;
  int rc = region_table(regions, W, quant, rank_offset, &rt);
  if (rc != EP_OK) return rc;
  // the common checks of a dispatch (no single receive buffer: capacity 0)
  rc = check_dispatch(x, topk_idx, topk_w, T, H, k, W, slot, 0, quant, nullptr, nullptr, nullptr,
                      nullptr, nullptr, status);
  if (rc != EP_OK) return rc;
  return from_cuda(ep::launch_dispatch_regions(x, topk_idx, topk_w, T, H, k, W, slot, quant, rt,
                                               status, reinterpret_cast<cudaStream_t>(stream)));
}

int ep_dispatch_regions_with_layout(const void* x, const int32_t* topk_idx, const float* topk_w,
                                    int64_t T, int H, int k, int E, int W,
                                    int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                                    int32_t* rank_offset, int32_t* slot, void* workspace,
                                    size_t workspace_bytes, const ep_rank_region_t* regions,
                                    int quant, int32_t* status, ep_stream_t stream) {
  int rc = check_layout(topk_idx, T, k, E, W, num_tokens_per_expert, num_tokens_per_rank,
                        rank_offset, slot, workspace, workspace_bytes, status);
  if (rc != EP_OK) return rc;
  ep::RankRegions rt;
  rc = region_table(regions, W, quant, rank_offset, &rt);
  if (rc != EP_OK) return rc;
  rc = check_dispatch(x, topk_idx, topk_w, T, H, k, W, slot, 0, quant, nullptr, nullptr, nullptr,
                      nullptr, nullptr, status);
  if (rc != EP_OK) return rc;
  return from_cuda(ep::launch_dispatch_regions_with_layout(
      x, topk_idx, topk_w, T, H, k, E, W, num_tokens_per_expert, num_tokens_per_rank, rank_offset,
      slot, workspace, quant, rt, status, reinterpret_cast<cudaStream_t>(stream)));
}

int ep_combine_regions(const void* const* y_regions, const int64_t* y_rows, const int32_t* slot,
                       const int32_t* rank_offset, int64_t T, int H, int W, void* out,
                       int32_t* status, ep_stream_t stream) {
  if (T < 0 || H < 1 || W < 1 || W > 32 || !y_regions || !y_rows || !rank_offset)
    return EP_ERR_INVALID_ARG;
  if (H % 8 != 0) return EP_ERR_UNSUPPORTED;
  if (T > kMaxRows / W) return EP_ERR_UNSUPPORTED;
  if (T > 0 && (!slot || !out)) return EP_ERR_INVALID_ARG;
  ep::RankRegions rt{};
  for (int r = 0; r < W; ++r) {
    if (y_rows[r] < 0 || y_rows[r] > kMaxRows) return EP_ERR_INVALID_ARG;
    if (y_rows[r] > 0 && !y_regions[r]) return EP_ERR_INVALID_ARG;
    if (!aligned(y_regions[r], 16)) return EP_ERR_MISALIGNED;
    rt.x[r] = static_cast<uint8_t*>(const_cast<void*>(y_regions[r]));
    rt.rows[r] = y_rows[r];
  }
  rt.rank_offset = rank_offset;
  if (!aligned(out, 16) || !aligned(slot, 4) || !aligned(rank_offset, 4) || !aligned(status, 4))
    return EP_ERR_MISALIGNED;
  return from_cuda(ep::launch_combine_regions(rt, slot, T, H, W, out, status,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

size_t ep_layout_experts_workspace_bytes(int64_t T, int k, int E) {
  if (T < 0 || k < 1 || E < 1) return 0;
  return ep::layout_experts_workspace_bytes(T, k, E);
}

namespace {
int check_layout_experts(const int32_t* topk_idx, int64_t T, int k, int E,
                         const int32_t* num_tokens_per_expert, const int32_t* expert_offset,
                         const int32_t* slot, const void* workspace, size_t workspace_bytes,
                         const int32_t* status) {
  if (T < 0 || k < 1 || E < 1 || E > ep::layout_experts_max_experts()) return EP_ERR_INVALID_ARG;
  if (T > kMaxRows / k) return EP_ERR_UNSUPPORTED;
  if (!num_tokens_per_expert || !expert_offset || !workspace) return EP_ERR_INVALID_ARG;
  if (T > 0 && (!topk_idx || !slot)) return EP_ERR_INVALID_ARG;
  if (workspace_bytes < ep::layout_experts_workspace_bytes(T, k, E)) return EP_ERR_WORKSPACE;
  if (!aligned(topk_idx, 4) || !aligned(num_tokens_per_expert, 4) || !aligned(expert_offset, 4) ||
      !aligned(slot, 4) || !aligned(workspace, 16) || !aligned(status, 4))
    return EP_ERR_MISALIGNED;
  return EP_OK;
}
}  // namespace

int ep_dispatch_layout_experts(const int32_t* topk_idx, int64_t T, int k, int E,
                               int32_t* num_tokens_per_expert, int32_t* expert_offset,
                               int32_t* slot, void* workspace, size_t workspace_bytes,
                               int32_t* status, ep_stream_t stream) {
  const int rc = check_layout_experts(topk_idx, T, k, E, num_tokens_per_expert, expert_offset,
                                      slot, workspace, workspace_bytes, status);
  if (rc != EP_OK) return rc;
  return from_cuda(ep::launch_layout_experts(topk_idx, T, k, E, num_tokens_per_expert,
                                             expert_offset, slot, workspace, status,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

int ep_dispatch_experts_with_layout(const void* x, const int32_t* topk_idx, const float* topk_w,
                                    int64_t T, int H, int k, int E,
                                    int32_t* num_tokens_per_expert, int32_t* expert_offset,
                                    int32_t* slot, void* workspace, size_t workspace_bytes,
                                    int64_t capacity_rows, int quant, void* recv_x,
                                    float* recv_scale, int32_t* recv_topk_idx, float* recv_topk_w,
                                    int32_t* recv_src, int32_t* status, ep_stream_t stream) {
  int rc = check_layout_experts(topk_idx, T, k, E, num_tokens_per_expert, expert_offset, slot,
                                workspace, workspace_bytes, status);
  if (rc != EP_OK) return rc;
  // the dispatch of the [T, k] slot table: W = k columns
  if (k > 32) return EP_ERR_UNSUPPORTED;
  rc = check_dispatch(x, topk_idx, topk_w, T, H, k, k, slot, capacity_rows, quant, recv_x,
                      recv_scale, recv_topk_idx, recv_topk_w, recv_src, status);
  if (rc != EP_OK) return rc;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  rc = from_cuda(ep::launch_layout_experts(topk_idx, T, k, E, num_tokens_per_expert, expert_offset,
                                           slot, workspace, status, s));
  if (rc != EP_OK) return rc;
  // the dispatch follows the layout kernels directly: its first rows of x are
  // loaded while they run, and (bulk-copy rows) it takes its later tokens from
  // a counter the layout zeroed in the workspace
  return from_cuda(ep::launch_dispatch(x, topk_idx, topk_w, T, H, k, k, slot, capacity_rows, quant,
                                       recv_x, recv_scale, recv_topk_idx, recv_topk_w, recv_src,
                                       status, s, /*x_early=*/1,
                                       ep::layout_experts_claim(workspace, T, k, E)));
}

int ep_combine_weighted(const void* y, const int32_t* slot, const float* w, int64_t T, int H,
                        int C, int64_t capacity_rows, void* out, int32_t* status,
                        ep_stream_t stream) {
  if (T < 0 || H < 1 || C < 1 || C > 32 || capacity_rows < 0 || capacity_rows > kMaxRows)
    return EP_ERR_INVALID_ARG;
  if (H % 8 != 0) return EP_ERR_UNSUPPORTED;
  if (T > kMaxRows / C) return EP_ERR_UNSUPPORTED;
  if (T > 0 && (!slot || !w || !out)) return EP_ERR_INVALID_ARG;
  if (T > 0 && capacity_rows > 0 && !y) return EP_ERR_INVALID_ARG;
  if (!aligned(y, 16) || !aligned(out, 16) || !aligned(slot, 4) || !aligned(w, 4) ||
      !aligned(status, 4))
    return EP_ERR_MISALIGNED;
  return from_cuda(ep::launch_combine_weighted(y, slot, w, T, H, C, capacity_rows, out, status,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

size_t ep_cast_transpose_t_bytes(int64_t capacity_rows, int E, int H) {
  if (capacity_rows < 0 || E < 1 || H < 1) return 0;
  return ep::cast_transpose_t_bytes(capacity_rows, E, H);
}

int ep_cast_transpose_experts(const void* y, const int32_t* expert_offset, int E, int H,
                              const float* scale, int64_t capacity_rows, void* out_c, void* out_t,
                              float* amax, int32_t* status, ep_stream_t stream) {
  if (E < 1 || E > 8192 || H < 1 || capacity_rows < 0 || capacity_rows > kMaxRows)
    return EP_ERR_INVALID_ARG;
  if (H % 256 != 0) return EP_ERR_UNSUPPORTED;
  if (!expert_offset || !scale || !amax) return EP_ERR_INVALID_ARG;
  if (capacity_rows > 0 && (!y || !out_c || !out_t)) return EP_ERR_INVALID_ARG;
  if (!aligned(y, 16) || !aligned(out_c, 16) || !aligned(out_t, 16) ||
      !aligned(expert_offset, 4) || !aligned(scale, 4) || !aligned(amax, 4) || !aligned(status, 4))
    return EP_ERR_MISALIGNED;
  return from_cuda(ep::launch_cast_transpose(y, expert_offset, E, H, scale, capacity_rows,
                                             static_cast<uint8_t*>(out_c),
                                             static_cast<uint8_t*>(out_t), amax, status,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

const char* ep_status_string(int code) {
  switch (code) {
    case EP_OK:
      return "EP_OK";
    case EP_ERR_INVALID_ARG:
      return "EP_ERR_INVALID_ARG: a size or pointer argument is out of range or NULL";
    case EP_ERR_MISALIGNED:
      return "EP_ERR_MISALIGNED: payload pointers need 16-byte, index pointers 4-byte alignment";
    case EP_ERR_UNSUPPORTED:
      return "EP_ERR_UNSUPPORTED: shape outside the supported set";
    case EP_ERR_CUDA:
      return "EP_ERR_CUDA: the CUDA runtime refused a launch";
    case EP_ERR_WORKSPACE:
      return "EP_ERR_WORKSPACE: workspace smaller than ep_layout_workspace_bytes()";
    default:
      return "unknown ep status code";
  }
}

}  // extern "C"
