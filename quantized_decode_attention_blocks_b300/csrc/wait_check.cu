// wait_check.cu -- diagnosis of the bounded waits every kernel of the library
// takes on its mbarriers: one warp waits on a barrier of its own, which
// either receives its one arrival first or none at all, with the library's
// bounded wait (mbar_wait_warp).  With no arrival the wait runs out, the
// kernel reports KVARN_STATUS_TIMEOUT and returns, and the context stays
// usable: the path every kernel takes when a copy or an MMA never completes,
// exercised without any fault.
#include "kvarn_internal.cuh"
#include "ptx.cuh"

namespace kvarn {
namespace {

using namespace ptx;

__global__ void __launch_bounds__(32) wait_check_kernel(int32_t* status, uint64_t limit_ns,
                                                        int arrive) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
  __syncwarp();
  if (!mbar_wait_warp(&bar, 0, limit_ns) && threadIdx.x == 0) report(status, KVARN_STATUS_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_check(int32_t* status, uint64_t limit_ns, int arrive, cudaStream_t s) {
  wait_check_kernel<<<1, 32, 0, s>>>(status, limit_ns, arrive);
  return cudaGetLastError();
}

}  // namespace kvarn
