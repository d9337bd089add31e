// Failure-detection check: the bounded waits of the pipelines, made to run
// out on purpose without faulting or hanging the GPU.  One thread waits on a
// shared-memory mbarrier that nothing arrives on (the wait every GEMM stage
// uses), then on a device counter that nothing increments (the ring
// dispatch's wait); each gives up after the 2 s budget and records
// MOK_ERR_TIMEOUT | SITE_CHECK in the status word, as a stalled pipeline
// would, and the kernel returns normally.
#include "common.cuh"
#include "kernels.h"

namespace mok {
namespace {

__device__ int32_t g_check_counter;  // never incremented

__global__ void wait_timeout_kernel(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  mbar_wait(&bar, 0, &abort_flag, status, SITE_CHECK);
  abort_flag = 0;
  wait_count(&g_check_counter, 1, &abort_flag, status, SITE_CHECK);
}

}  // namespace
}  // namespace mok

extern "C" mok_status mok_check_wait_timeout(void* stream) {
  int* status = mok::status_ptr();
  if (!status) return MOK_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* counter = nullptr;
  if (cudaGetSymbolAddress(&counter, mok::g_check_counter) != cudaSuccess ||
      cudaMemsetAsync(counter, 0, sizeof(int32_t), st) != cudaSuccess)
    return MOK_ERR_CUDA;
  mok::wait_timeout_kernel<<<1, 32, 0, st>>>(status);
  MOK_CHECK_LAUNCH();
  return MOK_OK;
}
