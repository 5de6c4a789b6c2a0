// Backward kernels for bf16 inputs (every head-dim and interval-count variant);
// the kernel itself is in attn_bwd.cuh.
#include "attn_bwd.cuh"

namespace hstu {

cudaError_t launch_bwd_bf16(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  return launch_bwd_typed<__nv_bfloat16>(p, nint, grid_items, stream);
}

}  // namespace hstu
