// Self-test of the failure-detection path of the kernels' bounded waits.
//
// Every mbarrier wait in the library's pipelines is bounded: a wait that
// runs out raises an abort flag in shared memory (so the CTA's other roles
// stop waiting too), records DEV_TIMEOUT and the waiting site in the status
// words of the workspace, and the kernel returns.  This entry point runs a
// kernel built from the same wait routine in which nothing ever arrives on
// the barriers: warp 0 waits with the caller's short limit and must time out
// and report `site`; warp 1 waits on a second barrier with the library's
// default limit and must give up early because of warp 0's abort flag.  The
// kernel then returns normally and leaves the CUDA context usable.
#include "moe.h"

#include <cuda_runtime.h>

#include <cstdint>

#include "sm100_ptx.cuh"

namespace {

__global__ void __launch_bounds__(64) wait_timeout_kernel(int32_t* status, uint64_t limit_ns, int32_t site) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    moe::mbar_init(&bars[0], 1);
    moe::mbar_init(&bars[1], 1);
    abort_flag = 0;
    moe::fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    // phase 0 of a barrier nobody arrives on never completes
    if (warp == 0) moe::mbar_wait_bounded(&bars[0], 0, &abort_flag, status, site, limit_ns);
    else moe::mbar_wait_bounded(&bars[1], 0, &abort_flag, status, site + 1);
  }
  __syncwarp();
}

}  // namespace

extern "C" moe_status_t moe_selftest_wait_timeout(void* ws, size_t ws_bytes, uint64_t limit_ns, int32_t site,
                                                  void* stream) {
  if (!ws || ws_bytes < 2 * sizeof(int32_t) || (reinterpret_cast<uintptr_t>(ws) & 15u) != 0)
    return MOE_ERR_WORKSPACE;
  if (limit_ns == 0 || limit_ns > 1000000000ull) return MOE_ERR_INVALID_ARG;   // at most 1 s
  wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int32_t*>(ws), limit_ns, site);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
