// Shared definitions of the CUDA path: workspace layout, kernel parameter
// blocks, the func-interval decode and the SiLU arithmetic used by the
// epilogues.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sm103_primitives.cuh"

namespace hstu {

constexpr int kBlock = 128;        // q-tile rows = kv-tile rows
constexpr int kMaxSeqlen = 32768;  // => at most 256 tiles per sequence
constexpr int kMaxTiles = kMaxSeqlen / kBlock;
constexpr int kMaxIntervals = 5;   // nfunc <= 9

// Workspace header (int32 words).
constexpr int kHdrErr = 0;     // error bits (kErrInput | kErrTimeout | kErrCheck)
constexpr int kHdrNFwd = 1;    // entries of the forward work list
constexpr int kHdrNBwd = 2;    // entries of the backward work list
// Dynamic work distribution of the persistent attention kernels: the next
// work index to hand out and the CTAs that have finished. The last CTA of a
// launch puts both back to zero, so that a reused plan starts clean.
constexpr int kHdrFwdNext = 4;
constexpr int kHdrFwdDone = 5;
constexpr int kHdrBwdNext = 6;
constexpr int kHdrBwdDone = 7;
// 1 when every sequence has the same tile count. Then striding the list by
// the grid size already hands every CTA the same mix of items, and the
// persistent kernels use that fixed assignment; otherwise they take items
// from the counters above, which balances ragged batches.
constexpr int kHdrUniform = 8;
constexpr int kHdrWords = 64;  // 256 bytes
constexpr int kErrInput = 1;
constexpr int kErrTimeout = 2;
constexpr int kErrCheck = 4;  // an index check of the checked build failed

// The checked build (compiled with HSTU_CHECKED) validates every work-list
// entry before anything is read or written through it; the release build
// compiles the checks away.
#ifdef HSTU_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// Tile classes written by the plan (bits 0-1), with the dead 64-wide halves
// of a partial pair: kv columns 0..63 / 64..127 seen by no row, q rows
// 0..63 / 64..127 seeing no column of the tile.
constexpr uint8_t kSkip = 0, kPartial = 1, kFull = 2, kClassMask = 3;
constexpr uint8_t kLoKvDead = 4, kHiKvDead = 8, kLoQDead = 16, kHiQDead = 32;

// Backward work-list entries: bit 30 = role (1: dK/dV for a kv tile,
// 0: dQ for a q tile), bits 8..29 = sequence, bits 0..7 = tile.
constexpr int kRoleDkdv = 1 << 30;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Layout of the HSTU_WS_FULL workspace. The plan writes every header word
// the kernels read; every other region is fully written before it is read.
struct FullLayout {
  int nt = 0;  // tiles per sequence at max_seqlen
  size_t header = 0, header_bytes = 0, fwd_list = 0, bwd_list = 0, ivmask = 0, cls = 0, total = 0;
};
inline FullLayout full_layout(int batch, int max_seqlen) {
  FullLayout l;
  l.nt = (max_seqlen + kBlock - 1) / kBlock;
  const size_t items = static_cast<size_t>(batch) * l.nt;
  l.header = 0;
  l.header_bytes = kHdrWords * 4;
  l.fwd_list = l.header_bytes;
  l.bwd_list = l.fwd_list + align_up(items * 4, 256);
  l.ivmask = l.bwd_list + align_up(2 * items * 4, 256);
  l.cls = l.ivmask + align_up(items, 256);
  l.total = l.cls + align_up(items * l.nt, 256);
  return l;
}

// Hands out the next work index of a persistent kernel (one thread).
__device__ __forceinline__ int fetch_work(int32_t* header, int next_word) {
  return atomicAdd(header + next_word, 1);
}
// Called once per CTA after all its roles have finished; the last CTA of the
// launch resets the counters for the next launch on the same plan.
__device__ __forceinline__ void finish_work(int32_t* header, int next_word, int done_word) {
  __threadfence();
  if (atomicAdd(header + done_word, 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(header + next_word, 0);
    atomicExch(header + done_word, 0);
  }
}

// Targets-only: keys per CTA chunk and the workspace of fp32 partials.
constexpr int kTgtChunk = 256;
struct TargetsLayout {
  int nc = 0;
  size_t header = 0, partial = 0, total = 0;
};
// dim: the wider of D_qk and D_v (the partials hold O rows or dQ rows).
inline TargetsLayout targets_layout(int batch, int heads, int dim, int max_seqlen) {
  TargetsLayout l;
  l.nc = (max_seqlen + kTgtChunk - 1) / kTgtChunk;
  l.header = 0;
  l.partial = kHdrWords * 4;
  l.total = l.partial + align_up(static_cast<size_t>(batch) * heads * l.nc * dim * 4, 256);
  return l;
}

struct PlanParams {
  const int32_t* seq_offsets;
  const int32_t* func;
  int32_t* row_counts;  // nullable
  int32_t* header;
  int32_t* fwd_list;
  int32_t* bwd_list;
  uint8_t* ivmask;     // per q tile: bit t set iff interval t is non-empty for some row
  uint8_t* cls;
  int64_t total;
  int32_t batch, nfunc, nt, max_seqlen;
  int32_t role_window;  // backward list entries per role window (role_window())
};

// Backward list entries per role window: as many as keep a window's q, k, v
// and dO rows (128 rows an entry, every head) within 32 MB, a quarter of L2,
// at most 128 and at least 16. (With 64 MB the SLA B=16 S=2048 H=8 backward
// re-read its tiles from HBM and ran 6% slower; with 32 MB every workload
// measured here ran at least as fast as without windows.)
inline int role_window(int heads, int dim, int dim_v) {
  const long long per_entry = 128LL * heads * (2LL * dim + 2LL * dim_v) * 2;
  const long long w = (32LL << 20) / (per_entry > 0 ? per_entry : 1);
  return static_cast<int>(w < 16 ? 16 : (w > 128 ? 128 : w));
}

// Element types of q, k, v, dO and the outputs (one type for all of them).
constexpr int kDtypeBf16 = 0, kDtypeF16 = 1;

struct AttnParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;          // 128-row boxes
  CUtensorMap tm_q64, tm_k64, tm_v64, tm_do64;  // 64-row boxes (backward streams)
  const int32_t* seq_offsets;
  const int32_t* func;
  void* out0;  // fwd: o (T, H, dim_v); bwd: dq (T, H, dim)
  void* out1;  // bwd: dk (T, H, dim)
  void* out2;  // bwd: dv (T, H, dim_v)
  const uint8_t* cls;
  const uint8_t* ivmask;
  const int32_t* list;
  int32_t* header;
  int64_t total;
  int32_t batch, heads, dim, dim_v, nt, max_seqlen;  // dim = D_qk, dim_v = D_v
  float alpha, inv_n;
  // Limit of the MMA thread's wait for the epilogue to have read out the
  // previous item's accumulators (kWaitLimitNs unless a test shortens it to
  // make that wait run out with copies and MMAs in flight).
  uint64_t handoff_limit_ns;
};

// Checked builds only: a work-list entry must name a sequence of the batch
// (and only the role bit besides it), and a tile inside that sequence. A bad
// entry sets kErrCheck; the caller then ends its work as if the list had run
// out. Every lane of the calling warp gets the same answer.
__device__ __forceinline__ bool list_entry_ok(const AttnParams& p, int code, bool bwd) {
  if (!kChecked) return true;
  const int payload = bwd ? (code & ~kRoleDkdv) : code;
  bool ok = payload >= 0 && (payload >> 8) < p.batch;
  if (ok) {
    const int b = payload >> 8;
    const int L = p.seq_offsets[b + 1] - p.seq_offsets[b];
    ok = (payload & 255) * kBlock < L;
  }
  if (!ok) atomicOr(p.header + kHdrErr, kErrCheck);
  return ok;
}

struct TgtParams {
  const void* q_c;   // (C, H, dim), C = num_cand candidate rows
  const void* k;     // (T, H, dim)
  const void* v;     // (T, H, dim_v)
  const void* do_c;  // (C, H, dim_v)
  void* o_c;         // fwd output (C, H, dim_v)
  void* dq_c;        // bwd outputs: (C, H, dim)
  void* dk;          // (T, H, dim)
  void* dv;          // (T, H, dim_v)
  const int32_t* seq_offsets;
  const int32_t* cand_offsets;  // (batch + 1) or null: one candidate per sequence
  const int32_t* func_c;        // (nfunc, num_cand)
  float* partial;
  int32_t* header;
  int64_t total;
  int32_t batch, num_cand, heads, dim, dim_v, nfunc, nc, max_seqlen;
  float alpha, inv_n;
};

// ---------------------------------------------------------------- func decode
// Clamped intervals of one row; an empty interval becomes [0, 0) so that it
// can never widen a bound or pass a membership test. Intervals whose bit is
// clear in `active` (empty for every row of the tile, as the plan found) are
// not read at all.
template <int NINT>
__device__ __forceinline__ void load_row_intervals(const int32_t* __restrict__ func, int64_t total,
                                                   int64_t row, int L, bool valid, int (&lo)[NINT],
                                                   int (&hi)[NINT], uint32_t active = 0xffu) {
#pragma unroll
  for (int t = 0; t < NINT; ++t) {
    int a = 0, e = 0;
    if (valid && ((active >> t) & 1u)) {
      a = (t == 0) ? 0 : __ldg(func + static_cast<int64_t>(2 * t - 1) * total + row);
      e = __ldg(func + static_cast<int64_t>(2 * t) * total + row);
      a = min(max(a, 0), L);
      e = min(max(e, 0), L);
      if (e <= a) a = e = 0;
    }
    lo[t] = a;
    hi[t] = e;
  }
}

// Bit k set iff column (base + k) lies in one of the row's intervals, k < 32.
template <int NINT>
__device__ __forceinline__ uint32_t row_mask_word(const int (&lo)[NINT], const int (&hi)[NINT],
                                                  int base) {
  uint32_t w = 0;
#pragma unroll
  for (int t = 0; t < NINT; ++t) {
    const int a = max(lo[t] - base, 0);
    const int e = min(hi[t] - base, 32);
    if (e > a) w |= static_cast<uint32_t>(((1ull << e) - 1ull) ^ ((1ull << a) - 1ull));
  }
  return w;
}

// ---------------------------------------------------------------- SiLU math
__device__ __forceinline__ float sigmoidf_fast(float x) {
  return __fdividef(1.0f, 1.0f + __expf(-x));
}

// Hardware tanh (one MUFU op, max relative error about 2^-11).
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Epilogue arithmetic on one S element s, with t = tanh(alpha s / 2) so that
// sigmoid(alpha s) = (1 + t) / 2 (one MUFU op per element). The common factor
// hc = alpha / (2N) is left out of every element and applied once to the fp32
// accumulators at their store:
//   silu(alpha s) / N  = hc * s (1 + t)                           -> P' = s (1 + t)
//   silu'(alpha s)     = (1 + t) / 2 + (alpha s / 4)(1 - t^2)
//                      = (1 + t)(1 + h (1 - t)) / 2,  h = alpha s / 2
//   dP silu'(alpha s) alpha / N = hc * dP (1 + t)(1 + h (1 - t))   -> G' = dP (1 + t)(1 + h - h t)
// so O = hc sum P' V, dV = hc sum P'^T dO, dK = hc sum G'^T Q, dQ = hc sum G' K.
__device__ __forceinline__ float silu_pu(float s, float half_alpha) {
  const float t = tanh_approx(half_alpha * s);
  return fmaf(s, t, s);
}
__device__ __forceinline__ void silu_pu_gu(float s, float dp, float half_alpha, float& p, float& g) {
  const float h = half_alpha * s;
  const float t = tanh_approx(h);
  p = fmaf(s, t, s);                      // s (1 + t)
  const float u = fmaf(dp, t, dp);        // dP (1 + t)
  const float f = fmaf(-h, t, h + 1.0f);  // 1 + h - h t
  g = u * f;
}
__device__ __forceinline__ float silu_gu(float s, float dp, float half_alpha) {
  const float h = half_alpha * s;
  const float t = tanh_approx(h);
  const float u = fmaf(dp, t, dp);
  const float f = fmaf(-h, t, h + 1.0f);
  return u * f;
}

// Stores 32 fp32 accumulator columns of one row, times `scale`, as T (bf16
// or fp16):
// 64 bytes as two 32-byte stores when `wide` (a 32-byte aligned row), else
// as four 16-byte stores. Each thread writes its own row, so every store
// instruction of a warp touches 32 rows; wider stores halve their number.
// The stores skip L1 allocation: nothing reads the rows back, and the
// read-out of a tile's accumulators measured about 20% faster that way.
template <typename T>
__device__ __forceinline__ void store_row32(T* dst, const uint32_t (&a)[32], float scale, bool wide) {
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e)
    pk[e] = Elem<T>::pack2(scale * __uint_as_float(a[2 * e]), scale * __uint_as_float(a[2 * e + 1]));
  if (wide) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
      asm volatile("st.global.L1::no_allocate.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(
                       dst + 16 * e),
                   "r"(pk[8 * e]), "r"(pk[8 * e + 1]), "r"(pk[8 * e + 2]), "r"(pk[8 * e + 3]),
                   "r"(pk[8 * e + 4]), "r"(pk[8 * e + 5]), "r"(pk[8 * e + 6]), "r"(pk[8 * e + 7])
                   : "memory");
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 8 * e),
                   "r"(pk[4 * e]), "r"(pk[4 * e + 1]), "r"(pk[4 * e + 2]), "r"(pk[4 * e + 3])
                   : "memory");
  }
}

// True when 32-byte stores of output rows of `dim` 16-bit elements from
// these bases stay aligned.
__device__ __forceinline__ bool wide_rows_ok(const void* a, const void* b, const void* c, int dim, int dim2) {
  return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b) | reinterpret_cast<uintptr_t>(c)) &
          31u) == 0 &&
         (dim % 16) == 0 && (dim2 % 16) == 0;
}

}  // namespace hstu
