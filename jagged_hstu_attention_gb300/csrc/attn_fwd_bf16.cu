// Forward kernels for bf16 inputs (every head-dim and interval-count variant);
// the kernel itself is in attn_fwd.cuh.
#include "attn_fwd.cuh"

namespace hstu {

cudaError_t launch_fwd_bf16(const AttnParams& p, int nint, int grid_items, cudaStream_t stream) {
  return launch_fwd_typed<__nv_bfloat16>(p, nint, grid_items, stream);
}

}  // namespace hstu
