/*
 * hstu_attn.h -- C ABI of the GB300 (sm_103a) jagged HSTU attention library.
 *
 * Operation (MLCommons training PR #903 and TorchEasyRec PR #670 describe the
 * op; the formula below is the pointwise-SiLU attention those pages run):
 *
 *   For every sequence b (rows [seq_offsets[b], seq_offsets[b+1]) of the
 *   jagged tensors, length L_b), every head h and every query row i < L_b:
 *     O[i] = sum over visible columns j of  silu(alpha * q_i . k_j) / N * v_j
 *   with silu(x) = x * sigmoid(x) and N = max_seqlen (one N for the batch).
 *
 *   Visible columns (TorchEasyRec PR #670, "move the HSTU arbitrary-mask path
 *   to NFUNC=5", PR body): row i reads (nfunc+1)/2 half-open column intervals
 *   from func[:, row] -- interval 0 is [0, func[0]), interval t >= 1 is
 *   [func[2t-1], func[2t]) -- in the sequence's local column coordinates.
 *   Bounds are clamped to [0, L_b]; an interval whose end <= start is empty
 *   and skipped; the visible set is the union of the intervals. func values
 *   are never an error.
 *
 *   Targets-only mode (MLCommons training PR #903, "compute the last HSTU
 *   layer only for the rows the loss reads"): one query row per sequence (its
 *   candidate) against the full-length K/V of that sequence; the result is
 *   that row of the full op.
 *
 * Conventions (all entry points):
 *   - q, k, v, o, dout, dq, dk, dv: DEVICE pointers, all bf16 or all fp16
 *     (shape->dtype), contiguous (tokens, num_heads, width): q, k, dq, dk are
 *     head_dim (D_qk) wide, v, o, dout, dv head_dim_v (D_v) wide. Products run
 *     on the tensor cores in the input type with fp32 accumulation; P and dS
 *     are rounded to the input type before their MMAs. Base addresses must be
 *     16-byte aligned.
 *   - seq_offsets: DEVICE int32 (batch+1), seq_offsets[0] = 0, non-decreasing,
 *     seq_offsets[batch] = total, every length <= max_seqlen.
 *   - func: DEVICE int32 (nfunc, total), shared by all heads (read once per
 *     row). func_c (targets-only): DEVICE int32 (nfunc, batch).
 *   - ws: DEVICE workspace of at least hstu_attn_workspace_size() bytes,
 *     256-byte aligned, owned by the caller. The library allocates nothing.
 *   - stream: a cudaStream_t passed as void*. Work is only enqueued on it; no
 *     entry point synchronises except hstu_attn_get_device_status.
 *   - Host-checkable errors (null pointers, unsupported nfunc or head_dim,
 *     misalignment, workspace too small, bad sizes) return a status before
 *     anything is enqueued. Errors only visible on the device (offsets that
 *     are not monotone, a length above max_seqlen, a wrong first or last
 *     offset) set the workspace error word; every later kernel that reads
 *     that workspace then writes nothing. Read it with
 *     hstu_attn_get_device_status. (The full path checks the offsets in the
 *     plan, before any output is written; the targets-only kernels check
 *     them as they go, so dk/dv rows of other sequences may already be
 *     written, but o_c and dq_c are not.)
 *   - No C++ exception crosses this boundary.
 */
#ifndef HSTU_ATTN_H_
#define HSTU_ATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define HSTU_API __attribute__((visibility("default")))
#else
#define HSTU_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HSTU_OK = 0,
  HSTU_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned pointer */
  HSTU_ERR_UNSUPPORTED = 2,  /* nfunc, head dims or dtype the library has no kernel for */
  HSTU_ERR_WORKSPACE = 3,    /* workspace null, too small or misaligned */
  HSTU_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, sync) */
  HSTU_ERR_DEVICE_INPUT = 5, /* device-side input check failed (offsets) */
  HSTU_ERR_TIMEOUT = 6,      /* a bounded in-kernel wait gave up */
  HSTU_ERR_DEVICE_CHECK = 7  /* checked build only: a work-list index check failed */
} hstu_status_t;

/* Input and output element types (all tensors of a call share one). */
#define HSTU_DTYPE_BF16 0
#define HSTU_DTYPE_F16 1

/* Size limits of a shape:
 *   - T < 2^31, since seq_offsets are int32 (else HSTU_ERR_INVALID_ARG);
 *   - B < 2^22, since the work lists pack the sequence index in 22 bits
 *     (else HSTU_ERR_UNSUPPORTED);
 *   - 2 min(B ceil(N/128), T/128 + B) H < 2^30: the backward's work items,
 *     which the kernels number in int32 (else HSTU_ERR_UNSUPPORTED). */
typedef struct {
  int32_t batch;      /* B, number of sequences (>= 1) */
  int64_t total;      /* T = seq_offsets[B], rows of k and v (and of q, o) */
  int32_t num_heads;  /* H >= 1 */
  int32_t head_dim;   /* D_qk, width of q and k rows (and dq, dk): 32, 64 or 128 */
  int32_t nfunc;      /* rows of func: odd, 1 to 9 */
  int32_t max_seqlen; /* N: >= every L_b, <= 32768; also the 1/N scale */
  float alpha;        /* scale on q.k, usually 1/sqrt(head_dim) */
  int32_t head_dim_v; /* D_v, width of v, o, dout and dv rows: 32, 64 or 128;
                         0 means D_v = D_qk (the attention dim and the linear
                         dim of an HSTU layer may differ) */
  int32_t dtype;      /* HSTU_DTYPE_BF16 (0) or HSTU_DTYPE_F16 (1) */
} hstu_attn_shape_t;

/* Workspace modes for hstu_attn_workspace_size. */
#define HSTU_WS_FULL 0    /* plan + hstu_attn_fwd + hstu_attn_bwd */
#define HSTU_WS_TARGETS 1 /* hstu_attn_{fwd,bwd}_targets_only */

/* Flags for hstu_attn_fwd / hstu_attn_bwd. */
#define HSTU_FLAG_NONE 0
/* The workspace already holds the plan that hstu_attn_plan (or an earlier
 * fwd/bwd call without this flag) built for the same seq_offsets, func and
 * shape; skip rebuilding it. The caller guarantees that none changed. */
#define HSTU_FLAG_REUSE_PLAN 1

/* 1 if the library has kernels for that nfunc (1, 3, 5, 7, 9), else 0. The pages'
 * wheel bakes NFUNC in at compile time (TorchEasyRec PR #670 review thread on
 * exposing it at runtime); here it is a runtime argument dispatched to
 * compiled variants, and this query exposes which ones exist. */
HSTU_API int hstu_attn_nfunc_supported(int32_t nfunc);

/* Bytes of workspace the given mode needs for that shape; 0 if the shape is
 * invalid or unsupported. */
HSTU_API size_t hstu_attn_workspace_size(const hstu_attn_shape_t* shape, int32_t mode);

/* Builds the plan in ws: validates seq_offsets on the device, classifies
 * every (q-tile, kv-tile) pair of 128x128 as skipped / partial / full from
 * func, and writes the longest-first work lists of the forward and backward
 * kernels. row_counts (nullable, DEVICE int32 (total)) receives the number of
 * visible columns of every row -- a debug output, head independent. */
HSTU_API hstu_status_t hstu_attn_plan(const int32_t* seq_offsets, const int32_t* func,
                             const hstu_attn_shape_t* shape, int32_t* row_counts, void* ws,
                             size_t ws_bytes, void* stream);

/* Forward: o = attention(q, k, v) over the full jagged batch. Rows with no
 * visible column get 0. Builds the plan first unless HSTU_FLAG_REUSE_PLAN. */
HSTU_API hstu_status_t hstu_attn_fwd(const void* q, const void* k, const void* v, void* o,
                            const int32_t* seq_offsets, const int32_t* func,
                            const hstu_attn_shape_t* shape, int32_t* row_counts, void* ws,
                            size_t ws_bytes, uint32_t flags, void* stream);

/* Backward of sum(o * dout): writes dq, dk, dv (all rows; zero where a row or
 * column takes part in no visible pair). dk/dv accumulate per kv tile in
 * tensor memory and dq per q tile, each output element written once by one
 * CTA: no atomics, bitwise repeatable. */
HSTU_API hstu_status_t hstu_attn_bwd(const void* dout, const void* q, const void* k, const void* v,
                            void* dq, void* dk, void* dv, const int32_t* seq_offsets,
                            const int32_t* func, const hstu_attn_shape_t* shape, void* ws,
                            size_t ws_bytes, uint32_t flags, void* stream);

/* Targets-only forward: q_c (batch, H, D) holds one candidate row per
 * sequence, func_c (nfunc, batch) its intervals; k, v are full length
 * (total, H, D). o_c (batch, H, D). */
HSTU_API hstu_status_t hstu_attn_fwd_targets_only(const void* q_c, const void* k, const void* v, void* o_c,
                                         const int32_t* seq_offsets, const int32_t* func_c,
                                         const hstu_attn_shape_t* shape, void* ws,
                                         size_t ws_bytes, void* stream);

/* Targets-only backward of sum(o_c * dout_c): dq_c (batch, H, D); dk, dv
 * (total, H, D), every row written (zero where not visible to its
 * sequence's candidate). */
HSTU_API hstu_status_t hstu_attn_bwd_targets_only(const void* dout_c, const void* q_c, const void* k,
                                         const void* v, void* dq_c, void* dk, void* dv,
                                         const int32_t* seq_offsets, const int32_t* func_c,
                                         const hstu_attn_shape_t* shape, void* ws,
                                         size_t ws_bytes, void* stream);

/* Several candidates per sequence (MLCommons training PR #903, Gating: the
 * targets-only rewrite must cope with batches that are not exactly one target
 * per sequence). Candidates cand_offsets[b] .. cand_offsets[b+1] of q_c belong
 * to sequence b; each has its own func column and sees the full-length K/V of
 * its sequence. A sequence may have none.
 *   q_c      DEVICE (num_candidates, H, D_qk); o_c (num_candidates, H, D_v)
 *   cand_offsets  DEVICE int32 (batch+1): 0, non-decreasing, last =
 *            num_candidates (checked on the device: HSTU_ERR_DEVICE_INPUT)
 *   func_c   DEVICE int32 (nfunc, num_candidates)
 *   ws       at least hstu_attn_targets_workspace_size(shape, num_candidates)
 * The backward writes dq_c (num_candidates, H, D_qk) and every row of dk, dv
 * (total, H, ...): each key row sums its sequence's candidates in candidate
 * order, once, without atomics (bitwise repeatable); rows no candidate sees
 * are zero. */
HSTU_API size_t hstu_attn_targets_workspace_size(const hstu_attn_shape_t* shape, int64_t num_candidates);
HSTU_API hstu_status_t hstu_attn_fwd_targets(const void* q_c, const void* k, const void* v, void* o_c,
                                             const int32_t* seq_offsets, const int32_t* cand_offsets,
                                             int64_t num_candidates, const int32_t* func_c,
                                             const hstu_attn_shape_t* shape, void* ws, size_t ws_bytes,
                                             void* stream);
HSTU_API hstu_status_t hstu_attn_bwd_targets(const void* dout_c, const void* q_c, const void* k, const void* v,
                                             void* dq_c, void* dk, void* dv, const int32_t* seq_offsets,
                                             const int32_t* cand_offsets, int64_t num_candidates,
                                             const int32_t* func_c, const hstu_attn_shape_t* shape, void* ws,
                                             size_t ws_bytes, void* stream);

/* Candidate-row projection of the targets-only layer (MLCommons training PR
 * #903, Summary: the last layer computes U and Q for the candidate rows
 * alone; K and V stay full length). The pages leave the projection itself
 * open; it is read as the layer's pointwise-SiLU input projection of a row,
 *     y = silu(x w^T + bias),  z = x w^T + bias,
 * evaluated on the listed rows of x only. GEMMs run on the tensor cores in
 * the input type with fp32 accumulation; y, z and the gradients are rounded
 * to the input type.
 *   x      DEVICE (x_rows, d_in); rows DEVICE int32 (num_rows) row indices
 *          into x, or NULL for all rows in order (num_rows = x_rows)
 *   w      DEVICE (d_out, d_in) (out features, in features); bias DEVICE
 *          (d_out) or NULL
 *   y, z   DEVICE (num_rows, d_out), written; z may be NULL (the backward
 *          needs it)
 *   d_in, d_out  multiples of 64; dtype HSTU_DTYPE_BF16 or HSTU_DTYPE_F16
 *          for every tensor
 *   ws     DEVICE, hstu_attn_project_workspace_size(rows ? num_rows : 0,
 *          d_in, d_out, 0) bytes, 256-byte aligned
 * x, w, bias, y and z must be 16-byte aligned (else HSTU_ERR_INVALID_ARG).
 * A row index outside [0, x_rows) sets HSTU_ERR_DEVICE_INPUT in ws's error
 * word (read with hstu_attn_get_device_status) and gives a zero input row. */
HSTU_API size_t hstu_attn_project_workspace_size(int64_t num_rows, int32_t d_in, int32_t d_out, int32_t backward);
HSTU_API hstu_status_t hstu_attn_project_rows(const void* x, int64_t x_rows, const int32_t* rows, int64_t num_rows,
                                              const void* w, const void* bias, int32_t d_in, int32_t d_out,
                                              int32_t dtype, void* y, void* z, void* ws, size_t ws_bytes,
                                              void* stream);
/* Backward of sum(y * dy) for hstu_attn_project_rows: dx_rows (num_rows,
 * d_in) is the gradient of each listed row of x (a caller adds it into its
 * dx at those rows), dw (d_out, d_in) and dbias (d_out, nullable) are
 * written. z is the forward's pre-activation. dbias sums the rows in a fixed
 * order (deterministic). ws: hstu_attn_project_workspace_size(num_rows, d_in,
 * d_out, 1) bytes. */
HSTU_API hstu_status_t hstu_attn_project_rows_bwd(const void* dy, const void* z, const void* x, int64_t x_rows,
                                                  const int32_t* rows, int64_t num_rows, const void* w,
                                                  int32_t d_in, int32_t d_out, int32_t dtype, void* dx_rows,
                                                  void* dw, void* dbias, void* ws, size_t ws_bytes, void* stream);

/* Scratch capacity of hstu_attn_fwd_noalloc, in bytes (8 MiB). */
#define HSTU_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/* Forward pass that allocates nothing and takes no workspace. The pages have
 * no counterpart: it is an addition of this library for callers that cannot
 * allocate device memory -- a serving runtime or host framework that reserves
 * all device memory up front and forbids allocation on the request path, or
 * a caller for whom cudaMalloc would synchronise the device or fail because
 * the memory is already spoken for. Arguments and result are those of
 * hstu_attn_fwd (the plan is always rebuilt). The plan's scratch is a fixed
 * array of HSTU_NOALLOC_SCRATCH_BYTES compiled into the library; every GPU
 * that loads the library holds it until the process exits.
 *   - A shape whose plan needs more than HSTU_NOALLOC_SCRATCH_BYTES (see
 *     hstu_attn_workspace_size with HSTU_WS_FULL) returns HSTU_ERR_WORKSPACE
 *     and enqueues nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and caches it for that
 *     device's current CUDA context; make that first call before any stream
 *     capture. A context rebuilt later (after cudaDeviceReset) is a new one:
 *     its first call looks the address up again, so make it outside a
 *     capture too.
 *   - No cudaMalloc, cudaFree or allocating library routine is called.
 *   - All calls on a device share the array, which keeps the last call's
 *     contents; each call clears what must start at zero. Calls whose work
 *     overlaps on the GPU (for example on two streams at once) race on it.
 *   - Errors found on the device (bad seq_offsets, a timed-out wait) are
 *     recorded in the array's error word, which a caller cannot read: there
 *     is no handle to it. On such an error o is left unwritten. This entry
 *     point is for callers that validate seq_offsets themselves; one that
 *     needs the device status uses hstu_attn_fwd with its own workspace. */
HSTU_API hstu_status_t hstu_attn_fwd_noalloc(const void* q, const void* k, const void* v, void* o,
                                             const int32_t* seq_offsets, const int32_t* func,
                                             const hstu_attn_shape_t* shape, int32_t* row_counts,
                                             void* stream);

/* Mask families whose func the library can build on the device. */
typedef enum {
  HSTU_FUNC_CAUSAL = 0,  /* row i: [0, i+1) (MLCommons training PR #903: causal,
                            one candidate at the end of each sequence) */
  HSTU_FUNC_SLA = 1,     /* TorchEasyRec PR #670, build_sla_func_tensor: a global
                            prefix [0, min(k1, i+1)) and a causal window
                            [max(0, i-k2+1), i+1) */
  HSTU_FUNC_ONERANK = 2  /* TorchEasyRec PR #670, OneRank: history prefix,
                            candidate and task-token intervals (see below) */
} hstu_func_kind_t;

typedef struct {
  int32_t kind;        /* hstu_func_kind_t */
  int32_t k1, k2;      /* SLA: prefix and window widths, >= 0 */
  int32_t groups;      /* OneRank: candidate groups at the end of a sequence, >= 1 */
  int32_t task_tokens; /* OneRank: task tokens per group, >= 1 */
} hstu_func_spec_t;

/* Builds func (nfunc, total) on the device for a mask family, so that it is
 * never assembled on the host (the pages build it on the host and, in the
 * reference wheel, once per head; TorchEasyRec PR #670, PR body). One thread
 * writes one row; the values are local column bounds as func expects.
 *   - CAUSAL:  row i -> [i+1, i+1, ...]: interval 0 = [0, i+1), the rest empty.
 *   - SLA:     row i -> [min(k1, i+1), max(0, i-k2+1), i+1, i+1, ...]; the
 *              padded intervals repeat the window end (empty). nfunc >= 3.
 *   - ONERANK: each sequence ends in `groups` groups of 1 + task_tokens rows
 *              after a history of Lp = L - groups (1 + task_tokens) rows. Group
 *              g opens with its candidate e_g = Lp + g (1 + task_tokens). A
 *              history row i -> [i+1, e, e+1, t, t+1] with e = e_(i mod groups)
 *              and t = e + 1 + (i mod task_tokens) (its prefix, a candidate and
 *              one of that candidate's task tokens); a group row r of group g
 *              -> [Lp, e_g, e_g+1, r, r+1] (the history, its candidate, itself).
 *              Sequences with Lp <= 0 get causal rows. nfunc >= 5; rows past
 *              the fifth repeat the fifth (empty).
 * Arguments: seq_offsets DEVICE int32 (batch+1); total = seq_offsets[batch];
 * max_seqlen >= every length (rows of a longer sequence past max_seqlen are
 * not written); func DEVICE int32 (nfunc, total), written. A sequence whose
 * offsets are out of order or out of [0, total] is skipped (the plan reports
 * such offsets). Returns HSTU_ERR_INVALID_ARG for null or misaligned
 * pointers, bad sizes or spec values, HSTU_ERR_UNSUPPORTED for an nfunc the
 * family cannot fill; nothing is enqueued then. */
HSTU_API hstu_status_t hstu_attn_build_func(const hstu_func_spec_t* spec, const int32_t* seq_offsets,
                                            int32_t batch, int64_t total, int32_t max_seqlen, int32_t nfunc,
                                            int32_t* func, void* stream);

/* Builds func_c (nfunc, batch) for the targets-only entry points on the
 * device: the candidate of sequence b is its last row and sees [0, L_b);
 * every further interval repeats L_b (empty). seq_offsets DEVICE int32
 * (batch+1); func_c DEVICE int32, written. */
HSTU_API hstu_status_t hstu_attn_build_func_candidates(const int32_t* seq_offsets, int32_t batch, int32_t nfunc,
                                                       int32_t* func_c, void* stream);

/* Synchronises the stream, then returns the status recorded in the
 * workspace error word (HSTU_OK, HSTU_ERR_DEVICE_INPUT, HSTU_ERR_TIMEOUT,
 * and in the checked build HSTU_ERR_DEVICE_CHECK) or HSTU_ERR_CUDA if the
 * synchronisation failed.
 *
 * Checked build: libhstu_attn_checked.so exports the same entry points,
 * compiled with HSTU_CHECKED. Its attention kernels validate each entry of
 * the plan's work lists (sequence inside the batch, tile inside the
 * sequence) before any load or store goes through it; a bad entry ends that
 * CTA's work and records HSTU_ERR_DEVICE_CHECK, and the workspace must be
 * planned again. It is a debugging aid: results equal the release build's
 * bit for bit. */
HSTU_API hstu_status_t hstu_attn_get_device_status(const void* ws, void* stream);

/* Static description of a status code. */
HSTU_API const char* hstu_status_string(hstu_status_t status);

/* Test hook for the failure path of the kernels' bounded in-kernel waits.
 * Enqueues one small kernel that waits, with the same bounded wait the
 * attention kernels use, on a barrier that nothing arrives at. After
 * limit_ms milliseconds the wait gives up, and the kernel records
 * HSTU_ERR_TIMEOUT in ws's error word, as a timed-out attention kernel does;
 * hstu_attn_get_device_status then returns it. Nothing faults and the
 * context stays usable. The next plan clears the error word.
 *   ws:       DEVICE workspace of either mode, 256-byte aligned.
 *   limit_ms: 1 to 2000.
 * Returns HSTU_ERR_WORKSPACE for a null or misaligned ws and
 * HSTU_ERR_INVALID_ARG for a limit out of range; nothing is enqueued then. */
HSTU_API hstu_status_t hstu_attn_test_wait_timeout(void* ws, int32_t limit_ms, void* stream);

/* Test hook for the abort path inside the attention kernels. Sets the limit
 * of one bounded wait of hstu_attn_fwd and hstu_attn_bwd launched after the
 * call: the MMA-issuing thread's wait for the epilogue to have read out the
 * previous work item's accumulators. A limit of 1 ns makes that wait give up
 * at once, while the next item's copies and MMAs are in flight; the kernel
 * then raises its abort flag, every role drains what it issued (bounded
 * waits), TMEM is freed and the workspace error word gets HSTU_ERR_TIMEOUT --
 * no fault, no hang, the context stays usable.
 *   limit_ns: 1 .. 2e9; 0 restores the kernels' normal limit (2 s).
 * Process-wide and meant for tests only; returns HSTU_ERR_INVALID_ARG above
 * 2e9. */
HSTU_API hstu_status_t hstu_attn_test_set_handoff_limit(uint64_t limit_ns);

/* Splits a batch over `world` data-parallel ranks, by whole sequences. Every
 * (sequence, head) unit of the op is independent in the forward and the
 * backward pass, so the ranks need no exchange; each runs the op on its own
 * sequences with the same max_seqlen N (N is the 1/N scale, so it must be the
 * one of the whole batch for results to match an unsplit run). The pages give
 * no partitioning; this is the greedy longest-processing-time rule: sequences
 * in descending cost (equal costs: lower index first) each go to the rank with
 * the smallest load so far (equal loads: lower rank).
 *   cost:      HOST int64 (batch), >= 0, the caller's work estimate of each
 *              sequence (its visible pairs, or L_b^2 for causal masks).
 *   owner:     HOST int32 (batch), written: the rank of each sequence.
 *   rank_load: HOST int64 (world), nullable, written: each rank's total cost.
 * Deterministic, so every rank computes the same split from the same costs.
 * Host-only: touches no GPU. Returns HSTU_ERR_INVALID_ARG (writing nothing)
 * for batch < 0, world < 1, a null cost or owner with batch > 0, a negative
 * cost, or costs whose sum overflows int64. */
HSTU_API hstu_status_t hstu_attn_shard_sequences(const int64_t* cost, int32_t batch, int32_t world,
                                                 int32_t* owner, int64_t* rank_load);

#ifdef __cplusplus
}
#endif

#endif /* HSTU_ATTN_H_ */
