// Host-side launchers of the CUDA path (C++ linkage, not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace hstu {

cudaError_t launch_plan(const PlanParams& p, cudaStream_t stream);
// grid_items: upper bound on the number of work items (CTAs = items * heads).
cudaError_t launch_fwd(const AttnParams& p, int nint, int grid_items, cudaStream_t stream);
cudaError_t launch_bwd(const AttnParams& p, int nint, int grid_items, cudaStream_t stream);
cudaError_t launch_targets_fwd(const TgtParams& p, cudaStream_t stream);
cudaError_t launch_targets_bwd(const TgtParams& p, cudaStream_t stream);

}  // namespace hstu
