// Self-test of the device failure path: one warp waits on an mbarrier that nothing ever
// arrives on, with a short cycle budget.  The bounded wait gives up, records
// FGE_ERR_DEVICE_TIMEOUT in the status word and the kernel returns normally, which is how
// every pipeline wait in the library reports a protocol failure instead of hanging.
#include "fge_device.cuh"

namespace fge {

__global__ void wait_timeout_kernel(int32_t* status, long long budget) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, budget);
}

}  // namespace fge

extern "C" fge_status fge_selftest_wait_timeout(void* workspace, int64_t budget_cycles,
                                                fge_stream_t stream) {
  if (!workspace || budget_cycles <= 0 || budget_cycles > (1LL << 32)) return FGE_ERR_INVALID_ARG;
  fge::wait_timeout_kernel<<<1, 32, 0, stream>>>(static_cast<int32_t*>(workspace), budget_cycles);
  return cudaGetLastError() == cudaSuccess ? FGE_OK : FGE_ERR_CUDA;
}
