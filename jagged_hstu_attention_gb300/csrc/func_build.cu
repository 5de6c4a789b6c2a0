// Device-side builders of the func interval tensor for the mask families the
// pages name, so that a caller never assembles func on the host and uploads
// it. Each thread writes one row: its nfunc values, one per func row, at
// stride `total` (rows of a sequence are consecutive, so the stores of a warp
// are coalesced).
//
//   causal   -- every row i: [0, i+1) (MLCommons training PR #903, the DLRMv4
//               last layer: causal, one candidate at the end); every further
//               interval repeats i+1 and is empty.
//   sla      -- TorchEasyRec PR #670 (build_sla_func_tensor, PR body): a global
//               prefix of k1 columns clipped causally, [0, min(k1, i+1)), and a
//               causal local window of k2 columns, [max(0, i-k2+1), i+1); the
//               padded third interval repeats the window end (empty).
//   onerank  -- TorchEasyRec PR #670 (the OneRank commit: history prefix,
//               candidate, task token). `groups` groups of 1 + `task_tokens`
//               tokens close each sequence after a history of Lp = L -
//               groups (1 + task_tokens) rows. Group g starts with its
//               candidate e_g = Lp + g (1 + task_tokens), followed by its task
//               tokens. A history row i sees [0, i+1), the candidate
//               e_(i mod groups) and the task token e + 1 + (i mod task_tokens)
//               of that group; a group row sees [0, Lp), its group's candidate
//               and itself. Sequences with Lp <= 0 get the causal row.
//   candidates (targets-only func_c) -- the candidate row of sequence b (its
//               last row) sees [0, L_b); every further interval is empty.
//
// Rows of a sequence longer than max_seqlen are not written; the plan rejects
// such offsets anyway. Offsets are read as given: a sequence whose offsets
// are out of order or out of [0, total] is skipped.
#include "../../include/hstu_attn.h"
#include "common.cuh"

namespace hstu {

constexpr int kBuildRows = 256;

// The func values of local row i of a sequence of length L, for the kinds
// above, written to v[0..nfunc).
__device__ __forceinline__ void func_row(const hstu_func_spec_t& spec, int i, int L, int nfunc, int (&v)[9]) {
  int a[5];
  int n = 0;
  if (spec.kind == HSTU_FUNC_SLA) {
    a[0] = min(spec.k1, i + 1);
    a[1] = max(0, i - spec.k2 + 1);
    a[2] = i + 1;
    n = 3;
  } else if (spec.kind == HSTU_FUNC_ONERANK) {
    const int gsize = spec.task_tokens + 1;
    const int lp = L - spec.groups * gsize;
    if (lp <= 0) {
      a[0] = i + 1;
      n = 1;
    } else if (i < lp) {
      const int e = lp + (i % spec.groups) * gsize;
      const int t = e + 1 + (i % spec.task_tokens);
      a[0] = i + 1; a[1] = e; a[2] = e + 1; a[3] = t; a[4] = t + 1;
      n = 5;
    } else {
      const int e = lp + ((i - lp) / gsize) * gsize;
      a[0] = lp; a[1] = e; a[2] = e + 1; a[3] = i; a[4] = i + 1;  // i == e: {e} twice
      n = 5;
    }
  } else {  // causal
    a[0] = i + 1;
    n = 1;
  }
  // Rows past the family's own repeat its last bound: empty intervals.
#pragma unroll
  for (int t = 0; t < 9; ++t) v[t] = t < n ? a[t < 5 ? t : 4] : a[n - 1];
  (void)nfunc;
}

__global__ void __launch_bounds__(kBuildRows) build_func_kernel(const int32_t* __restrict__ seq_offsets,
                                                                int32_t batch, int64_t total, int32_t nfunc,
                                                                int32_t chunks, hstu_func_spec_t spec,
                                                                int32_t* __restrict__ func) {
  const int b = blockIdx.x / chunks;
  const int chunk = blockIdx.x - b * chunks;
  if (b >= batch) return;
  const int o0 = seq_offsets[b], o1 = seq_offsets[b + 1];
  if (o0 < 0 || o1 < o0 || static_cast<int64_t>(o1) > total) return;
  const int L = o1 - o0;
  const int i = chunk * kBuildRows + threadIdx.x;
  if (i >= L) return;
  int v[9];
  func_row(spec, i, L, nfunc, v);
  const int64_t row = static_cast<int64_t>(o0) + i;
#pragma unroll
  for (int t = 0; t < 9; ++t)
    if (t < nfunc) func[static_cast<int64_t>(t) * total + row] = v[t];
}

__global__ void __launch_bounds__(256) build_func_candidates_kernel(const int32_t* __restrict__ seq_offsets,
                                                                    int32_t batch, int32_t nfunc,
                                                                    int32_t* __restrict__ func_c) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= batch) return;
  const int L = max(seq_offsets[b + 1] - seq_offsets[b], 0);
  for (int t = 0; t < nfunc; ++t) func_c[static_cast<int64_t>(t) * batch + b] = L;
}

}  // namespace hstu

extern "C" {

HSTU_API hstu_status_t hstu_attn_build_func(const hstu_func_spec_t* spec, const int32_t* seq_offsets,
                                            int32_t batch, int64_t total, int32_t max_seqlen, int32_t nfunc,
                                            int32_t* func, void* stream) {
  if (!spec || !seq_offsets || batch < 1 || total < 0 || total > INT32_MAX || max_seqlen < 1)
    return HSTU_ERR_INVALID_ARG;
  if (!hstu_attn_nfunc_supported(nfunc)) return HSTU_ERR_UNSUPPORTED;
  if (total > 0 && !func) return HSTU_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seq_offsets) | reinterpret_cast<uintptr_t>(func)) % 4 != 0)
    return HSTU_ERR_INVALID_ARG;
  switch (spec->kind) {
    case HSTU_FUNC_CAUSAL: break;
    case HSTU_FUNC_SLA:
      if (spec->k1 < 0 || spec->k2 < 0) return HSTU_ERR_INVALID_ARG;
      if (nfunc < 3) return HSTU_ERR_UNSUPPORTED;  // prefix and window need two intervals
      break;
    case HSTU_FUNC_ONERANK:
      if (spec->groups < 1 || spec->task_tokens < 1) return HSTU_ERR_INVALID_ARG;
      if (nfunc < 5) return HSTU_ERR_UNSUPPORTED;  // three intervals
      break;
    default: return HSTU_ERR_INVALID_ARG;
  }
  if (total == 0) return HSTU_OK;
  const int chunks = (max_seqlen + hstu::kBuildRows - 1) / hstu::kBuildRows;
  const long long blocks = static_cast<long long>(batch) * chunks;
  if (blocks > 0x7fffffffLL) return HSTU_ERR_UNSUPPORTED;
  hstu::build_func_kernel<<<static_cast<unsigned>(blocks), hstu::kBuildRows, 0, static_cast<cudaStream_t>(stream)>>>(
      seq_offsets, batch, total, nfunc, chunks, *spec, func);
  return cudaGetLastError() == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

HSTU_API hstu_status_t hstu_attn_build_func_candidates(const int32_t* seq_offsets, int32_t batch, int32_t nfunc,
                                                       int32_t* func_c, void* stream) {
  if (!seq_offsets || !func_c || batch < 1) return HSTU_ERR_INVALID_ARG;
  if (!hstu_attn_nfunc_supported(nfunc)) return HSTU_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(seq_offsets) | reinterpret_cast<uintptr_t>(func_c)) % 4 != 0)
    return HSTU_ERR_INVALID_ARG;
  const unsigned blocks = static_cast<unsigned>((batch + 255) / 256);
  hstu::build_func_candidates_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(seq_offsets, batch, nfunc,
                                                                                           func_c);
  return cudaGetLastError() == cudaSuccess ? HSTU_OK : HSTU_ERR_CUDA;
}

}  // extern "C"
