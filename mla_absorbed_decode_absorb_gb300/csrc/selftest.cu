// Self-test of the bounded-wait path every kernel of this library relies on:
// one warp waits, through the same mbarrier wait, on a barrier that nothing
// completes.  After `limit_ns` the wait gives up, records MLA_ERR_TIMEOUT in the
// device status word and the kernel returns, so the context stays usable and
// the host sees the code through mla_get_device_status.  Nothing faults,
// traps or hangs.  (No counterpart on the MLA pages: failure reporting.)
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected; none comes
    fence_mbar_init();
  }
  __syncwarp();
  grid_dep_wait();
  grid_dep_launch();
  if (threadIdx.x == 0) mbar_wait_impl<false>(smem_u32(&bar), 0, status, nullptr, limit_ns);
  __syncwarp();
}

}  // namespace

cudaError_t launch_wait_timeout(int* status, uint64_t limit_ns, cudaStream_t stream) {
  return launch_kernel(wait_timeout_kernel, dim3(1), dim3(32), 0, stream, status, limit_ns);
}

}  // namespace mla
