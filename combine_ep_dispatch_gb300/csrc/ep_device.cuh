// Device helpers and kernel launchers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ep_gb300.h"

namespace ep {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxRanks = 32;  // a token's destination ranks are one 32-bit mask

// ------------------------------------------------------------ dependent launch
// Every kernel of the library is launched with programmatic stream
// serialization and begins with pdl_wait(): the grid may become resident while
// the previous kernel on the stream drains, but touches no memory until that
// kernel has completed and its writes are visible.  Every CTA executes the wait
// before it can exit, so completion stays transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ memory access
// Read-once streaming load of 16 bytes: no L1 allocation.
__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 16-byte store of data that is not read again by this kernel.
__device__ __forceinline__ void st_v4(uint4* p, const uint4& v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_v2(uint2* p, const uint2& v) {
  asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// ------------------------------------------------------------ bulk copies (TMA)
// One-dimensional cp.async.bulk copies between global and shared memory.  Both
// addresses must be 16-byte aligned and the size a multiple of 16 bytes.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Test for completion of the barrier phase of the given parity
// (mbarrier.try_wait: may suspend the thread for a while).
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the barrier phase of the given parity to complete, for at most
// about one second; returns false when the limit ran out.
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr uint32_t kWaitCheckEvery = 512;  // polls between two reads of the timer
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (it % kWaitCheckEvery == 0 && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// shared -> global, tracked in the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes)
               : "memory");
}

// The same with an L2 eviction-priority hint (a policy from make_l2_policy).
__device__ __forceinline__ void bulk_store_hint(void* gdst, const void* smem_src, uint32_t bytes,
                                                uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(gdst),
               "r"(smem_u32(smem_src)), "r"(bytes), "l"(policy)
               : "memory");
}

// L2 policy: 1 = evict_first, 2 = evict_last, 3 = evict_unchanged (whole access).
template <int KIND>
__device__ __forceinline__ uint64_t make_l2_policy() {
  uint64_t p;
  if constexpr (KIND == 1)
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  else if constexpr (KIND == 2)
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  else
    asm volatile("createpolicy.fractional.L2::evict_unchanged.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ------------------------------------------------------------ warp helpers
__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Position of the (lane+1)-th set bit of `mask`, counting from bit 0 upwards:
// lane i < popc(mask) receives the rank of its i-th destination; the other
// lanes receive -1.
__device__ __forceinline__ int nth_set_bit_of_lane(unsigned mask, int lane) {
  return (int)__fns(mask, 0, lane + 1);
}

// ------------------------------------------------------------ launchers
int device_sm_count();  // cached per device; 0 on error

// Resident CTAs per SM of a kernel at a block size (no dynamic shared memory),
// queried once per device and kept in the caller's cache (one per call site).
template <typename K>
int occupancy_cached(K kernel, int threads, int (&cache)[128]) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) dev = -1;
  if (dev >= 0 && cache[dev] > 0) return cache[dev];
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  if (dev >= 0) cache[dev] = per_sm;  // a race only repeats the query
  return per_sm;
}

cudaError_t launch_layout(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                          int32_t* num_tokens_per_expert, int32_t* num_tokens_per_rank,
                          int32_t* rank_offset, int32_t* slot, void* workspace, int32_t* status,
                          cudaStream_t stream);
size_t layout_workspace_bytes(int64_t T, int W, int E);

// Per-chunk counts the layout's count kernel leaves in its workspace: chunk c
// holds tokens [c << shift, (c + 1) << shift).
struct LayoutChunks {
  const int32_t* chunk_rank;  // [C][W]  tokens of chunk c with r in D(t)
  const int32_t* chunk_exp;   // [C][E]  (t, j) entries of chunk c with expert e
  int64_t C;
  int shift;
  unsigned long long* claim;  // a counter the count kernel zeroes for the dispatch after it
};
// The count kernel alone; with local_slot non-null it also writes each
// (t, r)'s position p inside its chunk there as -2 - p (-1 when r is not in
// D(t)).
cudaError_t launch_layout_count(const int32_t* topk_idx, int64_t T, int k, int E, int W,
                                void* workspace, int32_t* local_slot, int32_t* status,
                                cudaStream_t stream, LayoutChunks* chunks);
// T up to which launch_layout uses its one-CTA kernel.
constexpr int64_t kLayoutSingleMaxT = 1024;
int64_t layout_num_chunks(int64_t T);
int dispatch_with_layout_launches(int64_t T, int H, int k, int W, int quant);
// ep_dispatch_with_layout: the layout, then the dispatch, launched so that the
// dispatch overlaps the layout (and, beyond 1024 tokens, finishes the layout
// itself in place of the scan kernel); small bf16 batches take the one-launch
// dispatch.
cudaError_t launch_dispatch_with_layout(const void* x, const int32_t* topk_idx, const float* topk_w,
                                        int64_t T, int H, int k, int E, int W,
                                        int32_t* num_tokens_per_expert,
                                        int32_t* num_tokens_per_rank, int32_t* rank_offset,
                                        int32_t* slot, void* workspace, int64_t capacity_rows,
                                        int quant, void* recv_x, float* recv_scale,
                                        int32_t* recv_topk_idx, float* recv_topk_w,
                                        int32_t* recv_src, int32_t* status, cudaStream_t stream);

cudaError_t launch_dispatch(const void* x, const int32_t* topk_idx, const float* topk_w,
                            int64_t T, int H, int k, int W, const int32_t* slot,
                            int64_t capacity_rows, int quant, void* recv_x, float* recv_scale,
                            int32_t* recv_topk_idx, float* recv_topk_w, int32_t* recv_src,
                            int32_t* status, cudaStream_t stream, int x_early = 0,
                            unsigned long long* claim = nullptr);

cudaError_t launch_localize_ids(int32_t* recv_topk_idx, const int32_t* rank_offset, int64_t cap,
                                int k, int E, int W, cudaStream_t stream);

int64_t fused_max_tokens();
cudaError_t launch_dispatch_fused(const void* x, const int32_t* topk_idx, const float* topk_w,
                                  int64_t T, int H, int k, int E, int W, int32_t* ne, int32_t* nr,
                                  int32_t* off, int32_t* slot, int64_t cap, void* recv_x,
                                  int32_t* ridx, float* rw, int32_t* rsrc, int32_t* status,
                                  cudaStream_t stream);

cudaError_t launch_combine(const void* y, const int32_t* slot, int64_t T, int H, int W,
                           int64_t capacity_rows, void* out, int32_t* status, cudaStream_t stream);
cudaError_t launch_combine_weighted(const void* y, const int32_t* slot, const float* w, int64_t T,
                                    int H, int C, int64_t capacity_rows, void* out,
                                    int32_t* status, cudaStream_t stream);

size_t cast_transpose_t_bytes(int64_t R, int E, int H);
cudaError_t launch_cast_transpose(const void* y, const int32_t* expert_offset, int E, int H,
                                  const float* scale, int64_t capacity_rows, uint8_t* out_c,
                                  uint8_t* out_t, float* amax, int32_t* status,
                                  cudaStream_t stream);

int layout_experts_max_experts();
size_t layout_experts_workspace_bytes(int64_t T, int k, int E);
// The token counter that launch_layout_experts zeroes in its workspace for the
// dispatch that follows it (null when its one-CTA path runs, which has none).
unsigned long long* layout_experts_claim(void* workspace, int64_t T, int k, int E);
cudaError_t launch_layout_experts(const int32_t* topk_idx, int64_t T, int k, int E,
                                  int32_t* num_tokens_per_expert, int32_t* expert_offset,
                                  int32_t* slot, void* workspace, int32_t* status,
                                  cudaStream_t stream);

// cudaLaunchKernelEx with the programmatic-stream-serialization attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace ep
