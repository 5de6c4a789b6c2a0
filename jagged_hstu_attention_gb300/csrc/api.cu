// C ABI of the library (declared in include/hstu_attn.h): host-side argument
// checks, workspace layout, TMA tensor-map encoding and kernel dispatch.
// Nothing here allocates device memory or synchronises, except
// hstu_attn_get_device_status.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/hstu_attn.h"
#include "common.cuh"
#include "internal.h"

namespace {

using hstu::kBlock;

// NVTX range around one entry point's host work (checks, tensor maps and the
// launches it enqueues), so a profiler timeline shows which call issued
// which kernels. NVTX is header-only and does nothing unless a tool is
// attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

bool aligned(const void* ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

hstu_status_t check_shape(const hstu_attn_shape_t* s) {
  if (!s) return HSTU_ERR_INVALID_ARG;
  if (s->batch < 1 || s->total < 0 || s->num_heads < 1 || s->max_seqlen < 1)
    return HSTU_ERR_INVALID_ARG;
  if (s->total > INT32_MAX) return HSTU_ERR_INVALID_ARG;  // offsets are int32
  if (s->max_seqlen > hstu::kMaxSeqlen) return HSTU_ERR_UNSUPPORTED;
  if (s->batch > (1 << 22) - 1) return HSTU_ERR_UNSUPPORTED;  // work-list encoding
  if (!hstu_attn_nfunc_supported(s->nfunc)) return HSTU_ERR_UNSUPPORTED;
  if (!dim_ok(s->head_dim) || (s->head_dim_v != 0 && !dim_ok(s->head_dim_v))) return HSTU_ERR_UNSUPPORTED;
  if (s->dtype != HSTU_DTYPE_BF16 && s->dtype != HSTU_DTYPE_F16) return HSTU_ERR_UNSUPPORTED;
  if (!(s->alpha == s->alpha)) return HSTU_ERR_INVALID_ARG;  // NaN
  // The kernels number their work (list entry x heads + head) in int32, and
  // their counters run past the end by up to a grid: keep it below 2^30. The
  // backward list has 2 sum_b ceil(L_b / 128) <= 2 min(B NT, T / 128 + B)
  // entries.
  const int64_t nt = (static_cast<int64_t>(s->max_seqlen) + hstu::kBlock - 1) / hstu::kBlock;
  const int64_t entries =
      2 * std::min<int64_t>(static_cast<int64_t>(s->batch) * nt, s->total / hstu::kBlock + s->batch);
  if (entries * s->num_heads >= (int64_t{1} << 30)) return HSTU_ERR_UNSUPPORTED;
  return HSTU_OK;
}

// D_v of a shape (0 stands for D_v = D_qk).
int dim_v(const hstu_attn_shape_t* s) { return s->head_dim_v != 0 ? s->head_dim_v : s->head_dim; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// (tokens, H, D) 16-bit elements viewed as a 4-D tensor {64 columns, tokens, H, D / 64
// chunks} with the chunk stride (128 B) below the row stride. One box of
// 64 columns x box_rows rows x 1 head x all chunks, with 128-byte swizzle,
// lands in shared memory as [chunk][row][128 B]: the K-major layout of the
// kernels' UMMA descriptors, in one TMA instruction per tile. For D = 32 the
// box is wider than the tensor and TMA fills the missing columns with zeros.
bool make_map(CUtensorMap* m, const void* ptr, int64_t tokens, int heads, int dim, int dtype,
              int box_rows = kBlock) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t chunks = dim > 64 ? static_cast<cuuint64_t>(dim / 64) : 1;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(dim < 64 ? dim : 64), static_cast<cuuint64_t>(tokens),
                        static_cast<cuuint64_t>(heads), chunks};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(heads) * dim * 2, static_cast<cuuint64_t>(dim) * 2, 128};
  cuuint32_t box[4] = {64, static_cast<cuuint32_t>(box_rows), 1, static_cast<cuuint32_t>(chunks)};
  cuuint32_t es[4] = {1, 1, 1, 1};
  const CUtensorMapDataType type =
      dtype == HSTU_DTYPE_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  return fn(m, type, 4, const_cast<void*>(ptr), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

hstu_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA; }

// Limit of the attention kernels' accumulator hand-off wait; 0 = the
// kernels' normal limit. Only hstu_attn_test_set_handoff_limit changes it.
std::atomic<uint64_t> g_handoff_limit_ns{0};

uint64_t handoff_limit() {
  const uint64_t v = g_handoff_limit_ns.load(std::memory_order_relaxed);
  return v != 0 ? v : hstu::kWaitLimitNs;
}

// Upper bound on the number of (sequence, tile) work items.
int grid_items(const hstu_attn_shape_t* s, int nt) {
  const int64_t by_tokens = (s->total + kBlock - 1) / kBlock + s->batch;
  const int64_t by_batch = static_cast<int64_t>(s->batch) * nt;
  return static_cast<int>(by_tokens < by_batch ? by_tokens : by_batch);
}

hstu_status_t check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (!ws || !aligned(ws, 256) || ws_bytes < need) return HSTU_ERR_WORKSPACE;
  return HSTU_OK;
}

hstu::PlanParams plan_params(const int32_t* seq_offsets, const int32_t* func,
                             const hstu_attn_shape_t* s, int32_t* row_counts, void* ws,
                             const hstu::FullLayout& l) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  hstu::PlanParams p{};
  p.seq_offsets = seq_offsets;
  p.func = func;
  p.row_counts = row_counts;
  p.header = reinterpret_cast<int32_t*>(base + l.header);
  p.fwd_list = reinterpret_cast<int32_t*>(base + l.fwd_list);
  p.bwd_list = reinterpret_cast<int32_t*>(base + l.bwd_list);
  p.ivmask = base + l.ivmask;
  p.cls = base + l.cls;
  p.total = s->total;
  p.batch = s->batch;
  p.nfunc = s->nfunc;
  p.nt = l.nt;
  p.max_seqlen = s->max_seqlen;
  p.role_window = hstu::role_window(s->num_heads, s->head_dim, dim_v(s));
  return p;
}

hstu_status_t check_common(const int32_t* seq_offsets, const int32_t* func,
                           const hstu_attn_shape_t* s, const void* ws, size_t ws_bytes) {
  hstu_status_t st = check_shape(s);
  if (st != HSTU_OK) return st;
  if (!seq_offsets || (s->total > 0 && !func)) return HSTU_ERR_INVALID_ARG;
  if (!aligned(seq_offsets, 4) || !aligned(func, 4)) return HSTU_ERR_INVALID_ARG;
  return check_ws(ws, ws_bytes, hstu_attn_workspace_size(s, HSTU_WS_FULL));
}

bool tensor_ok(const void* p) { return p && aligned(p, 16); }

hstu_status_t run_plan(const int32_t* seq_offsets, const int32_t* func, const hstu_attn_shape_t* s,
                       int32_t* row_counts, void* ws, cudaStream_t stream) {
  const hstu::FullLayout l = hstu::full_layout(s->batch, s->max_seqlen);
  return from_cuda(hstu::launch_plan(plan_params(seq_offsets, func, s, row_counts, ws, l), stream));
}

}  // namespace

extern "C" {

int hstu_attn_nfunc_supported(int32_t nfunc) {
  return (nfunc >= 1 && nfunc <= 2 * hstu::kMaxIntervals - 1 && nfunc % 2 == 1) ? 1 : 0;
}

size_t hstu_attn_workspace_size(const hstu_attn_shape_t* shape, int32_t mode) {
  if (check_shape(shape) != HSTU_OK) return 0;
  if (mode == HSTU_WS_FULL) return hstu::full_layout(shape->batch, shape->max_seqlen).total;
  if (mode == HSTU_WS_TARGETS) return hstu_attn_targets_workspace_size(shape, shape->batch);
  return 0;
}

hstu_status_t hstu_attn_plan(const int32_t* seq_offsets, const int32_t* func,
                             const hstu_attn_shape_t* shape, int32_t* row_counts, void* ws,
                             size_t ws_bytes, void* stream) {
  NvtxRange nvtx("hstu_attn_plan");
  hstu_status_t st = check_common(seq_offsets, func, shape, ws, ws_bytes);
  if (st != HSTU_OK) return st;
  if (row_counts && !aligned(row_counts, 4)) return HSTU_ERR_INVALID_ARG;
  return run_plan(seq_offsets, func, shape, row_counts, ws, static_cast<cudaStream_t>(stream));
}

hstu_status_t hstu_attn_fwd(const void* q, const void* k, const void* v, void* o,
                            const int32_t* seq_offsets, const int32_t* func,
                            const hstu_attn_shape_t* shape, int32_t* row_counts, void* ws,
                            size_t ws_bytes, uint32_t flags, void* stream) {
  NvtxRange nvtx("hstu_attn_fwd");
  hstu_status_t st = check_common(seq_offsets, func, shape, ws, ws_bytes);
  if (st != HSTU_OK) return st;
  if (shape->total > 0 && !(tensor_ok(q) && tensor_ok(k) && tensor_ok(v) && tensor_ok(o)))
    return HSTU_ERR_INVALID_ARG;
  if (row_counts && !aligned(row_counts, 4)) return HSTU_ERR_INVALID_ARG;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (!(flags & HSTU_FLAG_REUSE_PLAN)) {
    st = run_plan(seq_offsets, func, shape, row_counts, ws, cs);
    if (st != HSTU_OK) return st;
  }
  if (shape->total == 0) return HSTU_OK;
  const hstu::FullLayout l = hstu::full_layout(shape->batch, shape->max_seqlen);
  uint8_t* base = static_cast<uint8_t*>(ws);
  hstu::AttnParams p{};
  const int T = static_cast<int>(shape->total), H = shape->num_heads, Dq = shape->head_dim, Dv = dim_v(shape);
  const int dt = shape->dtype;
  if (!make_map(&p.tm_q, q, T, H, Dq, dt) || !make_map(&p.tm_k, k, T, H, Dq, dt) ||
      !make_map(&p.tm_v, v, T, H, Dv, dt))
    return HSTU_ERR_CUDA;
  p.tm_do = p.tm_q;
  p.seq_offsets = seq_offsets;
  p.func = func;
  p.out0 = o;
  p.cls = base + l.cls;
  p.ivmask = base + l.ivmask;
  p.list = reinterpret_cast<const int32_t*>(base + l.fwd_list);
  p.header = reinterpret_cast<int32_t*>(base + l.header);
  p.total = shape->total;
  p.batch = shape->batch;
  p.heads = shape->num_heads;
  p.dim = Dq;
  p.dim_v = Dv;
  p.nt = l.nt;
  p.max_seqlen = shape->max_seqlen;
  p.alpha = shape->alpha;
  p.inv_n = 1.0f / static_cast<float>(shape->max_seqlen);
  p.handoff_limit_ns = handoff_limit();
  return from_cuda(hstu::launch_fwd(p, (shape->nfunc + 1) / 2, dt, grid_items(shape, l.nt), cs));
}

hstu_status_t hstu_attn_bwd(const void* dout, const void* q, const void* k, const void* v,
                            void* dq, void* dk, void* dv, const int32_t* seq_offsets,
                            const int32_t* func, const hstu_attn_shape_t* shape, void* ws,
                            size_t ws_bytes, uint32_t flags, void* stream) {
  NvtxRange nvtx("hstu_attn_bwd");
  hstu_status_t st = check_common(seq_offsets, func, shape, ws, ws_bytes);
  if (st != HSTU_OK) return st;
  if (shape->total > 0 && !(tensor_ok(dout) && tensor_ok(q) && tensor_ok(k) && tensor_ok(v) &&
                            tensor_ok(dq) && tensor_ok(dk) && tensor_ok(dv)))
    return HSTU_ERR_INVALID_ARG;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (!(flags & HSTU_FLAG_REUSE_PLAN)) {
    st = run_plan(seq_offsets, func, shape, nullptr, ws, cs);
    if (st != HSTU_OK) return st;
  }
  if (shape->total == 0) return HSTU_OK;
  const hstu::FullLayout l = hstu::full_layout(shape->batch, shape->max_seqlen);
  uint8_t* base = static_cast<uint8_t*>(ws);
  hstu::AttnParams p{};
  const int T = static_cast<int>(shape->total), H = shape->num_heads, Dq = shape->head_dim, Dv = dim_v(shape);
  const int dt = shape->dtype;
  // q, k (and dq, dk) are D_qk wide; v and dout (and dv) D_v wide.
  if (!make_map(&p.tm_q, q, T, H, Dq, dt) || !make_map(&p.tm_k, k, T, H, Dq, dt) ||
      !make_map(&p.tm_v, v, T, H, Dv, dt) || !make_map(&p.tm_do, dout, T, H, Dv, dt) ||
      !make_map(&p.tm_q64, q, T, H, Dq, dt, kBlock / 2) || !make_map(&p.tm_k64, k, T, H, Dq, dt, kBlock / 2) ||
      !make_map(&p.tm_v64, v, T, H, Dv, dt, kBlock / 2) || !make_map(&p.tm_do64, dout, T, H, Dv, dt, kBlock / 2))
    return HSTU_ERR_CUDA;
  p.seq_offsets = seq_offsets;
  p.func = func;
  p.out0 = dq;
  p.out1 = dk;
  p.out2 = dv;
  p.cls = base + l.cls;
  p.ivmask = base + l.ivmask;
  p.list = reinterpret_cast<const int32_t*>(base + l.bwd_list);
  p.header = reinterpret_cast<int32_t*>(base + l.header);
  p.total = shape->total;
  p.batch = shape->batch;
  p.heads = shape->num_heads;
  p.dim = Dq;
  p.dim_v = Dv;
  p.nt = l.nt;
  p.max_seqlen = shape->max_seqlen;
  p.alpha = shape->alpha;
  p.inv_n = 1.0f / static_cast<float>(shape->max_seqlen);
  p.handoff_limit_ns = handoff_limit();
  return from_cuda(hstu::launch_bwd(p, (shape->nfunc + 1) / 2, dt, grid_items(shape, l.nt), cs));
}

static hstu_status_t targets_common(const void* q_c, const void* k, const void* v,
                                    const int32_t* seq_offsets, const int32_t* cand_offsets, int64_t num_cand,
                                    const int32_t* func_c, const hstu_attn_shape_t* shape, void* ws,
                                    size_t ws_bytes, hstu::TgtParams* p) {
  hstu_status_t st = check_shape(shape);
  if (st != HSTU_OK) return st;
  if (num_cand < 0 || num_cand > INT32_MAX) return HSTU_ERR_INVALID_ARG;
  if (!seq_offsets || (num_cand > 0 && !func_c) || !aligned(seq_offsets, 4) || !aligned(func_c, 4) ||
      !aligned(cand_offsets, 4))
    return HSTU_ERR_INVALID_ARG;
  if ((num_cand > 0 && !tensor_ok(q_c)) || (shape->total > 0 && !(tensor_ok(k) && tensor_ok(v))))
    return HSTU_ERR_INVALID_ARG;
  st = check_ws(ws, ws_bytes, hstu_attn_targets_workspace_size(shape, num_cand));
  if (st != HSTU_OK) return st;
  const hstu::TargetsLayout l = hstu::targets_layout(static_cast<int>(num_cand), shape->num_heads,
                                                     std::max(shape->head_dim, dim_v(shape)), shape->max_seqlen);
  uint8_t* base = static_cast<uint8_t*>(ws);
  *p = hstu::TgtParams{};
  p->q_c = q_c;
  p->k = k;
  p->v = v;
  p->seq_offsets = seq_offsets;
  p->cand_offsets = cand_offsets;
  p->func_c = func_c;
  p->partial = reinterpret_cast<float*>(base + l.partial);
  p->header = reinterpret_cast<int32_t*>(base + l.header);
  p->total = shape->total;
  p->batch = shape->batch;
  p->num_cand = static_cast<int32_t>(num_cand);
  p->heads = shape->num_heads;
  p->dim = shape->head_dim;
  p->dim_v = dim_v(shape);
  p->nfunc = shape->nfunc;
  p->nc = l.nc;
  p->max_seqlen = shape->max_seqlen;
  p->alpha = shape->alpha;
  p->inv_n = 1.0f / static_cast<float>(shape->max_seqlen);
  return HSTU_OK;
}

static hstu_status_t targets_fwd(const void* q_c, const void* k, const void* v, void* o_c,
                                 const int32_t* seq_offsets, const int32_t* cand_offsets, int64_t num_cand,
                                 const int32_t* func_c, const hstu_attn_shape_t* shape, void* ws, size_t ws_bytes,
                                 void* stream) {
  hstu::TgtParams p;
  hstu_status_t st = targets_common(q_c, k, v, seq_offsets, cand_offsets, num_cand, func_c, shape, ws, ws_bytes, &p);
  if (st != HSTU_OK) return st;
  if (num_cand > 0 && !tensor_ok(o_c)) return HSTU_ERR_INVALID_ARG;
  p.o_c = o_c;
  return from_cuda(hstu::launch_targets_fwd(p, shape->dtype, static_cast<cudaStream_t>(stream)));
}

static hstu_status_t targets_bwd(const void* dout_c, const void* q_c, const void* k, const void* v, void* dq_c,
                                 void* dk, void* dv, const int32_t* seq_offsets, const int32_t* cand_offsets,
                                 int64_t num_cand, const int32_t* func_c, const hstu_attn_shape_t* shape, void* ws,
                                 size_t ws_bytes, void* stream) {
  hstu::TgtParams p;
  hstu_status_t st = targets_common(q_c, k, v, seq_offsets, cand_offsets, num_cand, func_c, shape, ws, ws_bytes, &p);
  if (st != HSTU_OK) return st;
  if ((num_cand > 0 && !(tensor_ok(dout_c) && tensor_ok(dq_c))) ||
      (shape->total > 0 && !(tensor_ok(dk) && tensor_ok(dv))))
    return HSTU_ERR_INVALID_ARG;
  p.do_c = dout_c;
  p.dq_c = dq_c;
  p.dk = dk;
  p.dv = dv;
  return from_cuda(hstu::launch_targets_bwd(p, shape->dtype, static_cast<cudaStream_t>(stream)));
}

size_t hstu_attn_targets_workspace_size(const hstu_attn_shape_t* shape, int64_t num_candidates) {
  if (check_shape(shape) != HSTU_OK || num_candidates < 0 || num_candidates > INT32_MAX) return 0;
  return hstu::targets_layout(static_cast<int>(num_candidates), shape->num_heads,
                              std::max(shape->head_dim, dim_v(shape)), shape->max_seqlen)
      .total;
}

hstu_status_t hstu_attn_fwd_targets_only(const void* q_c, const void* k, const void* v, void* o_c,
                                         const int32_t* seq_offsets, const int32_t* func_c,
                                         const hstu_attn_shape_t* shape, void* ws,
                                         size_t ws_bytes, void* stream) {
  NvtxRange nvtx("hstu_attn_fwd_targets_only");
  if (!shape) return HSTU_ERR_INVALID_ARG;
  if (!q_c || !func_c) return HSTU_ERR_INVALID_ARG;
  return targets_fwd(q_c, k, v, o_c, seq_offsets, nullptr, shape->batch, func_c, shape, ws, ws_bytes, stream);
}

hstu_status_t hstu_attn_bwd_targets_only(const void* dout_c, const void* q_c, const void* k,
                                         const void* v, void* dq_c, void* dk, void* dv,
                                         const int32_t* seq_offsets, const int32_t* func_c,
                                         const hstu_attn_shape_t* shape, void* ws,
                                         size_t ws_bytes, void* stream) {
  NvtxRange nvtx("hstu_attn_bwd_targets_only");
  if (!shape) return HSTU_ERR_INVALID_ARG;
  if (!q_c || !func_c) return HSTU_ERR_INVALID_ARG;
  return targets_bwd(dout_c, q_c, k, v, dq_c, dk, dv, seq_offsets, nullptr, shape->batch, func_c, shape, ws,
                     ws_bytes, stream);
}

hstu_status_t hstu_attn_fwd_targets(const void* q_c, const void* k, const void* v, void* o_c,
                                    const int32_t* seq_offsets, const int32_t* cand_offsets, int64_t num_candidates,
                                    const int32_t* func_c, const hstu_attn_shape_t* shape, void* ws,
                                    size_t ws_bytes, void* stream) {
  NvtxRange nvtx("hstu_attn_fwd_targets");
  if (!cand_offsets) return HSTU_ERR_INVALID_ARG;
  return targets_fwd(q_c, k, v, o_c, seq_offsets, cand_offsets, num_candidates, func_c, shape, ws, ws_bytes,
                     stream);
}

hstu_status_t hstu_attn_bwd_targets(const void* dout_c, const void* q_c, const void* k, const void* v, void* dq_c,
                                    void* dk, void* dv, const int32_t* seq_offsets, const int32_t* cand_offsets,
                                    int64_t num_candidates, const int32_t* func_c, const hstu_attn_shape_t* shape,
                                    void* ws, size_t ws_bytes, void* stream) {
  NvtxRange nvtx("hstu_attn_bwd_targets");
  if (!cand_offsets) return HSTU_ERR_INVALID_ARG;
  return targets_bwd(dout_c, q_c, k, v, dq_c, dk, dv, seq_offsets, cand_offsets, num_candidates, func_c, shape,
                     ws, ws_bytes, stream);
}

hstu_status_t hstu_attn_test_set_handoff_limit(uint64_t limit_ns) {
  if (limit_ns > hstu::kWaitLimitNs) return HSTU_ERR_INVALID_ARG;
  g_handoff_limit_ns.store(limit_ns, std::memory_order_relaxed);
  return HSTU_OK;
}

hstu_status_t hstu_attn_get_device_status(const void* ws, void* stream) {
  if (!ws || !aligned(ws, 256)) return HSTU_ERR_WORKSPACE;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(cs) != cudaSuccess) return HSTU_ERR_CUDA;
  int32_t err = 0;
  if (cudaMemcpy(&err, ws, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return HSTU_ERR_CUDA;
  if (err & hstu::kErrInput) return HSTU_ERR_DEVICE_INPUT;
  if (err & hstu::kErrTimeout) return HSTU_ERR_TIMEOUT;
  if (err & hstu::kErrCheck) return HSTU_ERR_DEVICE_CHECK;
  return HSTU_OK;
}

const char* hstu_status_string(hstu_status_t status) {
  switch (status) {
    case HSTU_OK: return "ok";
    case HSTU_ERR_INVALID_ARG: return "invalid argument";
    case HSTU_ERR_UNSUPPORTED: return "unsupported nfunc, head dims, dtype or size";
    case HSTU_ERR_WORKSPACE: return "workspace null, misaligned or too small";
    case HSTU_ERR_CUDA: return "CUDA runtime error";
    case HSTU_ERR_DEVICE_INPUT: return "device-side input check failed (seq_offsets)";
    case HSTU_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
    case HSTU_ERR_DEVICE_CHECK: return "index check of the checked build failed";
  }
  return "unknown status";
}

}  // extern "C"
