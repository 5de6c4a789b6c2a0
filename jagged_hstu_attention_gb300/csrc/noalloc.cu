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
#include <cudaTypedefs.h>

#include <mutex>

#include "../../include/hstu_attn.h"

namespace {

constexpr size_t kNoAllocScratchBytes = HSTU_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address, looked up once per CUDA context of a device.
// A context has a unique id for the life of the process; a device whose
// context was torn down and rebuilt (cudaDeviceReset) gets a new one, in
// which the module is loaded again and the array may sit elsewhere, so the
// cached address is only reused while the current context's id matches.
struct ScratchSlot {
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
std::mutex g_setup_mutex;
ScratchSlot g_scratch[kMaxDevices];

struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};
const CtxFns& ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
  });
  return fns;
}

// Unique id of the current context (0 if none can be read).
unsigned long long current_ctx_id() {
  const CtxFns& fns = ctx_fns();
  if (!fns.get_current || !fns.get_id) return 0;
  CUcontext ctx = nullptr;
  if (fns.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (fns.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current device's context. Host
// code only sees a host-side stand-in under the array's name, so the address
// is looked up with cudaGetSymbolAddress, with that device current, on the
// first call in each context, and cached.
hstu_status_t scratch_for_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return HSTU_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchSlot& slot = g_scratch[dev];
  unsigned long long id = current_ctx_id();
  if (!slot.ptr || id == 0 || id != slot.ctx_id) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) return HSTU_ERR_CUDA;
    if (id == 0) id = current_ctx_id();  // the lookup may have made the context current
    slot.ptr = ptr;
    slot.ctx_id = id;  // 0: not cacheable, looked up again next call
    *out = ptr;
    return HSTU_OK;
  }
  *out = slot.ptr;
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
