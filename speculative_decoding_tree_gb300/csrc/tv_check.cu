// tv_check_bounded_wait: the library's bounded mbarrier wait (mbar_wait in
// tc_ptx.cuh, used by every tensor-core kernel) run against a barrier that
// nothing completes, so that the timeout path is exercised: the wait gives
// up after the limit, raises the abort flag, and the kernel reports
// TV_DEV_TIMEOUT and ends normally.
#include <cstdint>

#include "tc_ptx.cuh"
#include "tv_internal.cuh"

namespace tv {
namespace {

__global__ void bounded_wait_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&bar), 1);          // one arrival expected; none ever comes
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  dep_wait();
  dep_launch();
  if (threadIdx.x == 0) {
    const bool done = tc::mbar_wait(tc::smem_u32(&bar), 0, &abort_flag, limit_ns);
    if (!done) set_status(status, TV_DEV_TIMEOUT);
  }
}

}  // namespace
}  // namespace tv

extern "C" int tv_check_bounded_wait(int64_t limit_ns, int32_t* d_status, void* stream) {
  if (limit_ns < 1000000 || limit_ns > 10000000000ll) return TV_ERR_SHAPE;
  if (!d_status) return TV_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(d_status) & 15u) return TV_ERR_ALIGN;
  const cudaError_t e = tv::launch_dep(tv::bounded_wait_kernel, dim3(1), dim3(32), 0,
                                       static_cast<cudaStream_t>(stream), (uint64_t)limit_ns, d_status);
  return e == cudaSuccess ? TV_OK : TV_ERR_CUDA;
}
