// hstu_attn_test_wait_timeout: exercises the failure path of the kernels'
// bounded waits on the GPU without faulting or hanging it. One CTA waits,
// with the same mbar_wait the attention kernels use, on an mbarrier that
// nothing ever arrives at; after the given limit the wait gives up, raises
// the CTA's abort flag, and the CTA records the timeout in the workspace's
// error word exactly as a timed-out attention kernel does. The context stays
// usable, and the next plan clears the error word.
#include "../../include/hstu_attn.h"
#include "common.cuh"

namespace hstu {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int32_t* header, uint64_t limit_ns) {
  __shared__ alignas(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    volatile int* flag = &abort_flag;
    const bool arrived = mbar_wait(smem_u32(&bar), 0, flag, limit_ns);  // nothing arrives
    if (!arrived && *flag) atomicOr(header + kHdrErr, kErrTimeout);
  }
}

}  // namespace hstu

extern "C" HSTU_API hstu_status_t hstu_attn_test_wait_timeout(void* ws, int32_t limit_ms, void* stream) {
  if (!ws || reinterpret_cast<uintptr_t>(ws) % 256 != 0) return HSTU_ERR_WORKSPACE;
  if (limit_ms < 1 || limit_ms > 2000) return HSTU_ERR_INVALID_ARG;
  hstu::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int32_t*>(ws), static_cast<uint64_t>(limit_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}
