// Host-side launchers of the CUDA path (C++ linkage, not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"

namespace hstu {

// Raises `kernel`'s dynamic shared-memory limit to `smem` bytes on the
// current device, once per device (the attribute belongs to the device's
// context, so a process that drives several GPUs sets it on each).
// `done` holds one bit per device already set up.
template <typename Kernel>
cudaError_t ensure_smem_limit(Kernel kernel, int smem, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);
// grid_items: upper bound on the number of work items (CTAs = items * heads).
// One translation unit per input type keeps the many kernel variants
// compiling in parallel.
cudaError_t launch_fwd_bf16(const AttnParams& p, int nint, int grid_items, cudaStream_t stream);
cudaError_t launch_fwd_f16(const AttnParams& p, int nint, int grid_items, cudaStream_t stream);
cudaError_t launch_bwd_bf16(const AttnParams& p, int nint, int grid_items, cudaStream_t stream);
cudaError_t launch_bwd_f16(const AttnParams& p, int nint, int grid_items, cudaStream_t stream);
inline cudaError_t launch_fwd(const AttnParams& p, int nint, int dtype, int grid_items, cudaStream_t stream) {
  return dtype == kDtypeF16 ? launch_fwd_f16(p, nint, grid_items, stream)
                            : launch_fwd_bf16(p, nint, grid_items, stream);
}
inline cudaError_t launch_bwd(const AttnParams& p, int nint, int dtype, int grid_items, cudaStream_t stream) {
  return dtype == kDtypeF16 ? launch_bwd_f16(p, nint, grid_items, stream)
                            : launch_bwd_bf16(p, nint, grid_items, stream);
}
cudaError_t launch_targets_fwd(const TgtParams& p, int dtype, cudaStream_t stream);
cudaError_t launch_targets_bwd(const TgtParams& p, int dtype, cudaStream_t stream);

}  // namespace hstu
