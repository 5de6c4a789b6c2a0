"""CPU fp64 oracle for jagged HSTU attention with per-row interval masks.

TEST INFRASTRUCTURE ONLY. This module is the reference the CUDA kernels are
checked against. Only the test suite, the smoke check and the benchmark's CPU
baseline leg may import it; the library's own code path never does. It shares
no code with the CUDA path.

What it computes (the plain definition; the GPU method reaches it exactly up
to rounding, its speed coming only from skipping work):

* Mask (TorchEasyRec PR #670, "move the HSTU arbitrary-mask path to NFUNC=5",
  PR body and the CPU decode-coverage review thread): each query row r of a
  sequence of length L reads ``(nfunc + 1) // 2`` half-open column intervals
  from ``func[:, r]``: interval 0 is ``[0, func[0, r])``, interval t >= 1 is
  ``[func[2t-1, r], func[2t, r])``. Columns are local to the sequence. An
  interval with end <= start is skipped (empty); the row's visible set is the
  union (OR) of the remaining intervals. Bounds are clamped to ``[0, L]``
  (reading: the pages never let a bound leave the sequence; clamping is the
  plainest way to keep a row inside it).
* Forward: ``s_ij = alpha * q_i . k_j``; ``p_ij = silu(s_ij) / N`` with
  ``silu(x) = x * sigmoid(x)`` and N the batch's max sequence length;
  ``O_i = sum_{j visible} p_ij v_j`` (pointwise SiLU attention, no softmax).
* Backward of ``sum(O * dO)``: ``dV_j = sum_i p_ij dO_i``;
  ``g_ij = (dO_i . v_j) * silu'(s_ij) / N`` with
  ``silu'(x) = sigmoid(x) * (1 + x * (1 - sigmoid(x)))``;
  ``dQ_i = alpha * sum_j g_ij k_j``; ``dK_j = alpha * sum_i g_ij q_i``, all sums
  over visible pairs only.
* Targets-only (MLCommons training PR #903, "compute the last HSTU layer only
  for the rows the loss reads", Summary and Read First): one query row per
  sequence, evaluated against the full-length K/V of its sequence; it is the
  same function of the same inputs as that row of the full path, so it calls
  the same row-block routine with a one-row block. Several candidates per
  sequence (the page's "not exactly one target per sequence" batches) form a
  row block of their sequence (``fwd_targets`` / ``bwd_targets``).
* Candidate-row projection (the same page, Summary: U and Q are computed for
  the candidate rows alone): ``silu(x[rows] W^T + b)`` and its gradients
  (``project_rows`` / ``project_rows_backward``).

Two independent formulations are provided so that they can pin each other on
tiny inputs: a per-pair pure-Python loop (``*_loop``) and a dense per-sequence
mask-matrix formulation (``*_dense``, numpy fp64 matmuls).
"""
from __future__ import annotations

import math
from typing import List, Sequence, Tuple

import numpy as np

Interval = Tuple[int, int]


# ----------------------------------------------------------------------------
# Mask decode (TorchEasyRec PR #670: interleaved [max0, min0, max1, min1, ...]
# row layout, (NFUNC+1)/2 intervals, "max <= min" intervals skipped, OR).
# ----------------------------------------------------------------------------
def decode_intervals(func_col: Sequence[int], nfunc: int, L: int) -> List[Interval]:
    """Non-empty, clamped intervals of one query row."""
    if nfunc < 1 or nfunc % 2 == 0:
        raise ValueError("nfunc must be odd and >= 1")
    out: List[Interval] = []
    for t in range((nfunc + 1) // 2):
        if t == 0:
            lo, hi = 0, int(func_col[0])
        else:
            lo, hi = int(func_col[2 * t - 1]), int(func_col[2 * t])
        lo = min(max(lo, 0), L)
        hi = min(max(hi, 0), L)
        if hi <= lo:
            continue
        out.append((lo, hi))
    return out


def visible_row(func_col: Sequence[int], nfunc: int, L: int) -> np.ndarray:
    """Boolean (L,) visibility of one query row: the OR of its intervals."""
    m = np.zeros(L, dtype=bool)
    for lo, hi in decode_intervals(func_col, nfunc, L):
        m[lo:hi] = True
    return m


def mask_block(func_cols: np.ndarray, nfunc: int, L: int) -> np.ndarray:
    """(rows, L) boolean mask for a block of query rows; func_cols is
    (nfunc, rows)."""
    rows = func_cols.shape[1]
    M = np.zeros((rows, L), dtype=bool)
    for r in range(rows):
        M[r] = visible_row(func_cols[:, r], nfunc, L)
    return M


def visible_counts(seq_offsets: np.ndarray, func: np.ndarray, nfunc: int, seqs=None) -> np.ndarray:
    """Per-row visible column count |union of intervals| (head independent).
    ``seqs`` restricts the work to those sequence indices (other rows: 0)."""
    T = int(seq_offsets[-1])
    out = np.zeros(T, dtype=np.int64)
    for b in range(len(seq_offsets) - 1):
        if seqs is not None and b not in seqs:
            continue
        o0, o1 = int(seq_offsets[b]), int(seq_offsets[b + 1])
        L = o1 - o0
        for r in range(o0, o1):
            out[r] = int(visible_row(func[:, r], nfunc, L).sum())
    return out


# ----------------------------------------------------------------------------
# Scalar pieces (plain definitions, fp64).
# ----------------------------------------------------------------------------
def _sigmoid(x):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-x))


def _silu(x):
    return x * _sigmoid(x)


def _silu_grad(x):
    s = _sigmoid(x)
    return s * (1.0 + x * (1.0 - s))


# ----------------------------------------------------------------------------
# Per-pair loop formulation (tiny inputs only).
# ----------------------------------------------------------------------------
def fwd_loop(q, k, v, seq_offsets, func, nfunc, max_seqlen, alpha):
    """O (T, H, D) by the per-pair definition."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, H, D = q.shape
    o = np.zeros((T, H, v.shape[2]))
    N = float(max_seqlen)
    for b in range(len(seq_offsets) - 1):
        o0, o1 = int(seq_offsets[b]), int(seq_offsets[b + 1])
        L = o1 - o0
        for i in range(L):
            vis = visible_row(func[:, o0 + i], nfunc, L)
            for h in range(H):
                acc = np.zeros(v.shape[2])
                for j in range(L):
                    if not vis[j]:
                        continue
                    s = alpha * float(np.dot(q[o0 + i, h], k[o0 + j, h]))
                    acc += (s / (1.0 + math.exp(-s)) / N) * v[o0 + j, h]
                o[o0 + i, h] = acc
    return o


def bwd_loop(do, q, k, v, seq_offsets, func, nfunc, max_seqlen, alpha):
    """(dq, dk, dv) by the per-pair definition."""
    do = np.asarray(do, np.float64)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    T, H, D = q.shape
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    N = float(max_seqlen)
    for b in range(len(seq_offsets) - 1):
        o0, o1 = int(seq_offsets[b]), int(seq_offsets[b + 1])
        L = o1 - o0
        for i in range(L):
            vis = visible_row(func[:, o0 + i], nfunc, L)
            for j in range(L):
                if not vis[j]:
                    continue
                for h in range(H):
                    s = alpha * float(np.dot(q[o0 + i, h], k[o0 + j, h]))
                    sg = 1.0 / (1.0 + math.exp(-s))
                    p = s * sg / N
                    dv[o0 + j, h] += p * do[o0 + i, h]
                    g = float(np.dot(do[o0 + i, h], v[o0 + j, h])) * sg * (1.0 + s * (1.0 - sg)) / N
                    dq[o0 + i, h] += alpha * g * k[o0 + j, h]
                    dk[o0 + j, h] += alpha * g * q[o0 + i, h]
    return dq, dk, dv


# ----------------------------------------------------------------------------
# Dense per-sequence formulation: one (rows x L) block per sequence and head.
# ----------------------------------------------------------------------------
def _heads_first(x):
    return np.ascontiguousarray(np.transpose(x, (1, 0, 2)))


def block_forward(Qb, Kb, Vb, M, alpha, N):
    """Qb (m, H, D), Kb/Vb (L, H, D), M (m, L) bool -> (m, H, Dv)."""
    Qh, Kh, Vh = _heads_first(Qb), _heads_first(Kb), _heads_first(Vb)
    S = alpha * (Qh @ np.transpose(Kh, (0, 2, 1)))  # (H, m, L)
    with np.errstate(over="ignore"):
        P = _silu(S) / N * M[None]
    return np.transpose(P @ Vh, (1, 0, 2))


def block_backward(dOb, Qb, Kb, Vb, M, alpha, N):
    """Gradients of sum(O * dO) for one block -> (dQb, dKb, dVb)."""
    Qh, Kh, Vh, dOh = (_heads_first(x) for x in (Qb, Kb, Vb, dOb))
    S = alpha * (Qh @ np.transpose(Kh, (0, 2, 1)))
    Mf = M[None].astype(np.float64)
    with np.errstate(over="ignore"):
        P = _silu(S) / N * Mf
        G = (dOh @ np.transpose(Vh, (0, 2, 1))) * _silu_grad(S) / N * Mf
    dVh = np.transpose(P, (0, 2, 1)) @ dOh
    dQh = alpha * (G @ Kh)
    dKh = alpha * (np.transpose(G, (0, 2, 1)) @ Qh)
    back = lambda x: np.transpose(x, (1, 0, 2))
    return back(dQh), back(dKh), back(dVh)


def _seq_iter(seq_offsets):
    for b in range(len(seq_offsets) - 1):
        yield b, int(seq_offsets[b]), int(seq_offsets[b + 1])


def fwd_dense(q, k, v, seq_offsets, func, nfunc, max_seqlen, alpha, seqs=None):
    """O (T, H, D). ``seqs`` restricts the work to those sequence indices
    (other rows stay zero)."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    o = np.zeros((q.shape[0], q.shape[1], v.shape[2]))
    for b, o0, o1 in _seq_iter(seq_offsets):
        if seqs is not None and b not in seqs:
            continue
        L = o1 - o0
        M = mask_block(func[:, o0:o1], nfunc, L)
        o[o0:o1] = block_forward(q[o0:o1], k[o0:o1], v[o0:o1], M, alpha, float(max_seqlen))
    return o


def bwd_dense(do, q, k, v, seq_offsets, func, nfunc, max_seqlen, alpha, seqs=None):
    do = np.asarray(do, np.float64)
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b, o0, o1 in _seq_iter(seq_offsets):
        if seqs is not None and b not in seqs:
            continue
        L = o1 - o0
        M = mask_block(func[:, o0:o1], nfunc, L)
        dq[o0:o1], dk[o0:o1], dv[o0:o1] = block_backward(
            do[o0:o1], q[o0:o1], k[o0:o1], v[o0:o1], M, alpha, float(max_seqlen))
    return dq, dk, dv


# ----------------------------------------------------------------------------
# Targets-only: one candidate row per sequence against full-length K/V.
# ----------------------------------------------------------------------------
def fwd_targets_only(q_c, k, v, seq_offsets, func_c, nfunc, max_seqlen, alpha):
    """q_c (B, H, D), func_c (nfunc, B) -> o_c (B, H, Dv)."""
    q_c = np.asarray(q_c, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    B = q_c.shape[0]
    o_c = np.zeros((B, q_c.shape[1], v.shape[2]))
    for b, o0, o1 in _seq_iter(seq_offsets):
        L = o1 - o0
        M = mask_block(func_c[:, b:b + 1], nfunc, L)
        o_c[b:b + 1] = block_forward(q_c[b:b + 1], k[o0:o1], v[o0:o1], M, alpha, float(max_seqlen))
    return o_c


def bwd_targets_only(do_c, q_c, k, v, seq_offsets, func_c, nfunc, max_seqlen, alpha):
    """-> (dq_c (B, H, D), dk (T, H, D), dv (T, H, D))."""
    do_c = np.asarray(do_c, np.float64)
    q_c = np.asarray(q_c, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dq_c = np.zeros_like(q_c)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b, o0, o1 in _seq_iter(seq_offsets):
        L = o1 - o0
        M = mask_block(func_c[:, b:b + 1], nfunc, L)
        dq_c[b:b + 1], dk[o0:o1], dv[o0:o1] = block_backward(
            do_c[b:b + 1], q_c[b:b + 1], k[o0:o1], v[o0:o1], M, alpha, float(max_seqlen))
    return dq_c, dk, dv


# ----------------------------------------------------------------------------
# Several candidates per sequence (MLCommons training PR #903, Gating: a batch
# that is not exactly one target per sequence). Reading: each candidate row is
# the same function of its own q row and func column against its sequence's
# full K/V, so the candidates of a sequence form one row block of that
# sequence. Candidates cand_offsets[b] .. cand_offsets[b+1] of q_c belong to
# sequence b.
# ----------------------------------------------------------------------------
def fwd_targets(q_c, k, v, seq_offsets, cand_offsets, func_c, nfunc, max_seqlen, alpha):
    """q_c (C, H, D), func_c (nfunc, C) -> o_c (C, H, Dv)."""
    q_c = np.asarray(q_c, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    o_c = np.zeros((q_c.shape[0], q_c.shape[1], v.shape[2]))
    for b, o0, o1 in _seq_iter(seq_offsets):
        c0, c1 = int(cand_offsets[b]), int(cand_offsets[b + 1])
        if c1 <= c0:
            continue
        M = mask_block(func_c[:, c0:c1], nfunc, o1 - o0)
        o_c[c0:c1] = block_forward(q_c[c0:c1], k[o0:o1], v[o0:o1], M, alpha, float(max_seqlen))
    return o_c


def bwd_targets(do_c, q_c, k, v, seq_offsets, cand_offsets, func_c, nfunc, max_seqlen, alpha):
    """-> (dq_c (C, H, D), dk (T, H, D), dv (T, H, Dv)); dk, dv sum over the
    candidates of each sequence."""
    do_c = np.asarray(do_c, np.float64)
    q_c = np.asarray(q_c, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    dq_c = np.zeros_like(q_c)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b, o0, o1 in _seq_iter(seq_offsets):
        c0, c1 = int(cand_offsets[b]), int(cand_offsets[b + 1])
        if c1 <= c0:
            continue
        M = mask_block(func_c[:, c0:c1], nfunc, o1 - o0)
        dq_c[c0:c1], dk[o0:o1], dv[o0:o1] = block_backward(
            do_c[c0:c1], q_c[c0:c1], k[o0:o1], v[o0:o1], M, alpha, float(max_seqlen))
    return dq_c, dk, dv


# ----------------------------------------------------------------------------
# Candidate-row projection of the targets-only layer (MLCommons training PR
# #903, Summary: the last layer computes U and Q for the candidate row alone,
# K and V stay full length). The pages do not spell the projection out;
# reading: U and Q of a row come from that row of the layer input through the
# layer's pointwise-SiLU input projection, y = silu(x W^T + b) with W laid
# out (out features, in features), so the targets-only layer evaluates it on
# the candidate rows only.
# ----------------------------------------------------------------------------
def project_rows(x, rows, w, bias):
    """x (T, d_in), rows (C,) int, w (d_out, d_in), bias (d_out,) or None ->
    (y (C, d_out), z (C, d_out)) with z = x[rows] w^T + bias, y = silu(z)."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    z = x[np.asarray(rows, dtype=np.int64)] @ w.T
    if bias is not None:
        z = z + np.asarray(bias, np.float64)[None, :]
    with np.errstate(over="ignore"):
        return _silu(z), z


def project_rows_backward(dy, x, rows, w, bias):
    """Gradients of sum(y * dy) -> (dx (T, d_in): zero on rows not selected,
    dw (d_out, d_in), db (d_out,))."""
    dy = np.asarray(dy, np.float64)
    x = np.asarray(x, np.float64)
    w = np.asarray(w, np.float64)
    rows = np.asarray(rows, dtype=np.int64)
    _, z = project_rows(x, rows, w, bias)
    g = dy * _silu_grad(z)
    dx = np.zeros_like(x)
    np.add.at(dx, rows, g @ w)
    return dx, g.T @ x[rows], g.sum(axis=0)


def useful_pairs(seq_offsets, func, nfunc) -> int:
    """Number of visible (row, column) pairs per head."""
    return int(visible_counts(seq_offsets, func, nfunc).sum())
