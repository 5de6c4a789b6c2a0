// hstu_attn_fwd_noalloc: the forward pass for callers that cannot allocate
// device memory -- for example a serving runtime or a host framework that
// reserves all device memory up front and hands out none on the request path,
// or any caller for whom a cudaMalloc (which may synchronise the device or
// simply fail once memory is fully reserved) is not an option. The caller
// still owns q, k, v, o, seq_offsets, func and row_counts; only the scratch
// the forward needs for its plan (tile classes, work lists, error word) comes
// from a fixed array compiled into this library.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes.
// Every GPU that loads the library holds it until the process exits. All
// calls on a device share it and it keeps the last call's contents; the plan
// clears the parts that must start at zero at the beginning of every call.
// Calls whose work overlaps on the GPU (two streams at once) race on it.
#include <mutex>

#include "../../include/hstu_attn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = HSTU_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device. Host code only
// sees a host-side stand-in under the array's name, so the address is looked
// up once per device, with that device current, and cached.
hstu_status_t scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HSTU_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return HSTU_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return HSTU_OK;
}

}  // namespace

extern "C" HSTU_API hstu_status_t hstu_attn_fwd_noalloc(const void* q, const void* k, const void* v,
                                                        void* o, const int32_t* seq_offsets,
                                                        const int32_t* func,
                                                        const hstu_attn_shape_t* shape,
                                                        int32_t* row_counts, void* stream) {
  const size_t need = hstu_attn_workspace_size(shape, HSTU_WS_FULL);
  if (need == 0) {
    // Invalid or unsupported shape: let the regular checks name the reason.
    return hstu_attn_fwd(q, k, v, o, seq_offsets, func, shape, row_counts, nullptr, 0,
                         HSTU_FLAG_NONE, stream);
  }
  if (need > kNoAllocScratchBytes) return HSTU_ERR_WORKSPACE;  // beyond the built-in maximum
  void* scratch = nullptr;
  const hstu_status_t st = scratch_for_current_device(&scratch);
  if (st != HSTU_OK) return st;
  return hstu_attn_fwd(q, k, v, o, seq_offsets, func, shape, row_counts, scratch,
                       kNoAllocScratchBytes, HSTU_FLAG_NONE, stream);
}
