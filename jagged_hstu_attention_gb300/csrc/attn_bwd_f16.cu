// Backward kernels for f16 inputs (every head-dim and interval-count variant);
// the kernel itself is in attn_bwd.cuh.
#include "attn_bwd.cuh"

namespace hstu {

cudaError_t launch_bwd_f16(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  return launch_bwd_typed<__half>(p, nint, grid_items, stream);
}

}  // namespace hstu
