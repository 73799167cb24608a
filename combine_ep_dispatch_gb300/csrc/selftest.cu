// Self-test of the bounded on-chip waits.  Every wait in the library's
// kernels (bulk-copy completions on mbarriers) gives up after about one second
// and reports EP_STATUS_TIMEOUT instead of hanging.  This kernel waits, with
// the same helper, on an mbarrier that nothing ever completes, so the limit
// must run out: the call returns normally, the status word carries
// EP_STATUS_TIMEOUT and the CUDA context stays usable.
#include "ep_device.cuh"

namespace ep {
namespace {

__global__ void __launch_bounds__(32) selftest_wait_kernel(int32_t* __restrict__ status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // one arrival expected; none will come
    fence_barrier_init();
    const bool completed = mbar_wait_bounded(&bar, 0);
    if (!completed && status != nullptr) atomicOr(status, EP_STATUS_TIMEOUT);
  }
  __syncwarp();
}

}  // namespace
}  // namespace ep

extern "C" EP_API int ep_selftest_wait_timeout(int32_t* status, ep_stream_t stream) {
  if (status == nullptr || (reinterpret_cast<uintptr_t>(status) & 3) != 0) return EP_ERR_INVALID_ARG;
  ep::selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
  return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
