"""Pins for the CPU fp64 oracle (no GPU).

Each test ties the oracle to something other than itself: the worked example
printed on the pages, closed forms, special cases that reduce to a textbook
routine (causal HSTU through torch's own SiLU and autograd), invariants the
pages state (inert padding, union over intervals, targets-only equals the
full path's row), brute-force loop vs dense formulation, and central finite
differences. Mutation tests plant a mistake in the oracle and check that a
pin catches it.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle.hstu_oracle as orc
from jagged_hstu_attention_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np64(t):
    return t.float().numpy().astype(np.float64)


def _small_batch(seed, lens, H=2, D=16):
    lens = np.asarray(lens, dtype=np.int64)
    off = wl.offsets_from_lengths(lens)
    T = int(off[-1])
    g = torch.Generator().manual_seed(seed)
    q, k, v, do = (_np64(wl.randn_bf16((T, H, D), g)) for _ in range(4))
    return lens, off, q, k, v, do


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ---------------------------------------------------------------- golden
def test_partition_worked_example_rows():
    """TorchEasyRec PR #670 decode-coverage example: [s1,s1,s2,s2,q+1] covers
    exactly the causal row [0, q+1)."""
    rows = np.loadtxt(os.path.join(GOLDEN, "partition_rows.txt"), dtype=np.int64, comments="#")
    assert rows.shape[0] >= 8
    L = 64
    for row in rows:
        q, f, lo, hi, cnt = row[0], row[1:6], row[6], row[7], row[8]
        vis = orc.visible_row(f, 5, L)
        expect = np.zeros(L, dtype=bool)
        expect[lo:hi] = True
        assert np.array_equal(vis, expect), q
        assert vis.sum() == cnt == q + 1


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_loop_matches_dense_tiny(seed):
    cfg = wl.CONFIGS["tiny"]
    lens = wl.lengths(cfg, seed)[:2] // 2 + 3  # keep the loop small
    off = wl.offsets_from_lengths(lens)
    func = wl.build_func(cfg, lens)
    _, _, q, k, v, do = _small_batch(seed, lens, H=2, D=8)
    N, alpha = int(lens.max()), 1.0 / math.sqrt(8)
    o_loop = orc.fwd_loop(q, k, v, off, func, 5, N, alpha)
    o_dense = orc.fwd_dense(q, k, v, off, func, 5, N, alpha)
    assert _rel(o_loop, o_dense) < 1e-12
    gl = orc.bwd_loop(do, q, k, v, off, func, 5, N, alpha)
    gd = orc.bwd_dense(do, q, k, v, off, func, 5, N, alpha)
    for a, b in zip(gl, gd):
        assert _rel(a, b) < 1e-12


# ---------------------------------------------------------------- causal textbook
def _textbook_causal(q, k, v, off, N, alpha):
    """Causal HSTU written with torch's tril and torch's SiLU (fp64)."""
    out = torch.zeros(q.shape, dtype=torch.float64)
    for b in range(len(off) - 1):
        o0, o1 = int(off[b]), int(off[b + 1])
        Q, K, V = (x[o0:o1].transpose(0, 1) for x in (q, k, v))  # (H, L, D)
        A = torch.nn.functional.silu(alpha * Q @ K.transpose(1, 2)) / N
        A = torch.tril(A)
        out[o0:o1] = (A @ V).transpose(0, 1)
    return out


@pytest.mark.parametrize("nfunc", [1, 3, 5, 7, 9])
def test_causal_special_case_matches_textbook(nfunc):
    lens, off, q, k, v, do = _small_batch(3, [37, 5, 64, 20], H=2, D=16)
    cfg = wl.Config("c", 4, 0, 0, 2, 16, "causal", nfunc)
    func = wl.build_func(cfg, lens, nfunc)
    N, alpha = 64, 0.25
    o = orc.fwd_dense(q, k, v, off, func, nfunc, N, alpha)
    qt, kt, vt = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    ref = _textbook_causal(qt, kt, vt, off, N, alpha)
    assert _rel(o, ref.detach().numpy()) < 1e-13
    # gradients of sum(O * dO) through torch autograd
    (ref * torch.tensor(do)).sum().backward()
    dq, dk, dv = orc.bwd_dense(do, q, k, v, off, func, nfunc, N, alpha)
    assert _rel(dq, qt.grad.numpy()) < 1e-12
    assert _rel(dk, kt.grad.numpy()) < 1e-12
    assert _rel(dv, vt.grad.numpy()) < 1e-12


# ---------------------------------------------------------------- invariants
def test_padding_is_inert_exactly():
    """NFUNC=5 with the third interval padded empty equals NFUNC=3 bitwise
    (TorchEasyRec PR #670: pad rows repeat col_max1, max <= min is skipped)."""
    cfg = wl.Config("s", 3, 0, 0, 2, 16, "sla", 5, k1=20, k2=6)
    lens, off, q, k, v, do = _small_batch(4, [50, 33, 70])
    f5 = wl.build_func(cfg, lens, 5)
    f3 = wl.build_func(cfg, lens, 3)
    assert np.array_equal(f5[:3], f3)
    assert np.all(f5[4] <= f5[3])  # pad interval is empty
    N, alpha = 70, 0.25
    assert np.array_equal(orc.fwd_dense(q, k, v, off, f5, 5, N, alpha),
                          orc.fwd_dense(q, k, v, off, f3, 3, N, alpha))
    for a, b in zip(orc.bwd_dense(do, q, k, v, off, f5, 5, N, alpha),
                    orc.bwd_dense(do, q, k, v, off, f3, 3, N, alpha)):
        assert np.array_equal(a, b)


def _partition_func(lens):
    cols = []
    for L in lens:
        i = np.arange(L)
        s1 = np.minimum(2, i + 1)
        s2 = np.minimum(5, i + 1)
        cols.append(np.stack([s1, s1, s2, s2, i + 1]))
    return np.concatenate(cols, axis=1).astype(np.int32)


def test_partition_chunks_equal_causal():
    lens, off, q, k, v, do = _small_batch(5, [12, 30, 7])
    f = _partition_func(lens)
    fc = wl.build_func(wl.Config("c", 3, 0, 0, 2, 16, "causal", 1), lens, 1)
    N, alpha = 30, 0.25
    np.testing.assert_allclose(orc.fwd_dense(q, k, v, off, f, 5, N, alpha),
                               orc.fwd_dense(q, k, v, off, fc, 1, N, alpha), rtol=0, atol=1e-15)


def test_sla_equals_causal_when_the_prefix_spans_every_row():
    """SLA with a global prefix K1 at least as long as the sequence sees
    [0, i+1) on every row (the prefix clipped causally covers the window):
    the same function as plain causal, forward and backward."""
    lens, off, q, k, v, do = _small_batch(9, [20, 33, 5])
    sla = wl.Config("s", 3, 0, 0, 2, 16, "sla", 5, k1=40, k2=6)
    fs = wl.build_func(sla, lens, 5)
    fc = wl.build_func(wl.Config("c", 3, 0, 0, 2, 16, "causal", 1), lens, 1)
    N, alpha = 33, 0.3
    np.testing.assert_array_equal(orc.visible_counts(off, fs, 5), orc.visible_counts(off, fc, 1))
    np.testing.assert_allclose(orc.fwd_dense(q, k, v, off, fs, 5, N, alpha),
                               orc.fwd_dense(q, k, v, off, fc, 1, N, alpha), rtol=0, atol=1e-15)
    for a, b in zip(orc.bwd_dense(do, q, k, v, off, fs, 5, N, alpha),
                    orc.bwd_dense(do, q, k, v, off, fc, 1, N, alpha)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-15)
    # a shorter prefix is not causal: rows past K1 + K2 lose columns
    short = wl.build_func(wl.Config("s", 3, 0, 0, 2, 16, "sla", 5, k1=8, k2=6), lens, 5)
    assert orc.visible_counts(off, short, 5).sum() < orc.visible_counts(off, fc, 1).sum()


@pytest.mark.parametrize("mask", ["tiny", "sla", "onerank", "causal"])
@pytest.mark.parametrize("nfunc", [5, 7, 9])
def test_func_width_matches_nfunc_and_padding_is_empty(mask, nfunc):
    """Contract of the func builders: nfunc rows per token, and every interval
    past the ones the mask uses is empty (max <= min) on every row."""
    lens = np.array([40, 100] if mask == "onerank" else [40, 9])
    cfg = wl.Config("w", 2, 0, 0, 2, 16, mask, nfunc)
    f = wl.build_func(cfg, lens, nfunc)
    assert f.shape == (nfunc, int(lens.sum()))
    used = {"tiny": 3, "sla": 3, "onerank": 5, "causal": 1}[mask]
    for t in range((used + 1) // 2, (nfunc + 1) // 2):
        assert np.all(f[2 * t] <= f[2 * t - 1]), t


def test_mutation_dropping_last_interval_is_caught(monkeypatch):
    """Plant the mistake the pages describe (decode loop drops the last
    interval) in the oracle: the partition pin must then fail."""
    lens, off, q, k, v, do = _small_batch(5, [12, 30, 7])
    f = _partition_func(lens)
    fc = wl.build_func(wl.Config("c", 3, 0, 0, 2, 16, "causal", 1), lens, 1)
    N, alpha = 30, 0.25
    good = orc.fwd_dense(q, k, v, off, fc, 1, N, alpha)
    real = orc.decode_intervals

    def dropped(func_col, nfunc, L):
        if nfunc == 1:
            return real(func_col, nfunc, L)
        return real(func_col, nfunc - 2, L)

    monkeypatch.setattr(orc, "decode_intervals", dropped)
    bad = orc.fwd_dense(q, k, v, off, f, 5, N, alpha)
    assert not np.allclose(bad, good, atol=1e-6)


def test_mutation_double_counting_overlap_is_caught(monkeypatch):
    """Union, not sum: the tiny mask overlaps prefix and window on purpose; a
    mask that counts overlapping columns twice must break the count pin."""
    cfg = wl.CONFIGS["tiny"]
    lens = np.array([20, 9])
    off = wl.offsets_from_lengths(lens)
    func = wl.build_func(cfg, lens)
    good = orc.visible_counts(off, func, 5)

    def summed(func_col, nfunc, L):
        m = np.zeros(L, dtype=np.int64)
        for lo, hi in orc.decode_intervals(func_col, nfunc, L):
            m[lo:hi] += 1
        return m

    monkeypatch.setattr(orc, "visible_row", summed)
    bad = orc.visible_counts(off, func, 5)
    assert not np.array_equal(bad, good)
    assert np.array_equal(good, _tiny_closed_form(lens))


# ---------------------------------------------------------------- closed forms
def _tiny_closed_form(lens):
    out = []
    for L in lens:
        for i in range(L):
            a = min(8, L)                  # |[0, a)|
            b0, b1 = max(0, i - 7), i + 1  # window
            inter = max(0, min(a, b1) - b0)
            out.append(a + (b1 - b0) - inter)
    return np.array(out)


def test_counts_closed_forms():
    cfg = wl.CONFIGS["tiny"]
    lens = wl.lengths(cfg, 0)
    off = wl.offsets_from_lengths(lens)
    assert np.array_equal(orc.visible_counts(off, wl.build_func(cfg, lens), 5), _tiny_closed_form(lens))
    # SLA K1=256, K2=32: count_i = min(i+1, 288)
    sla = wl.CONFIGS["sla_b32_s1024"]
    lens = np.array([1024, 300])
    off = wl.offsets_from_lengths(lens)
    got = orc.visible_counts(off, wl.build_func(sla, lens), 5)
    exp = np.concatenate([np.minimum(np.arange(L) + 1, 288) for L in lens])
    assert np.array_equal(got, exp)
    # causal: i+1
    c = wl.CONFIGS["dlrm_b1024"]
    lens = np.array([17, 130])
    off = wl.offsets_from_lengths(lens)
    got = orc.visible_counts(off, wl.build_func(c, lens), 1)
    assert np.array_equal(got, np.concatenate([np.arange(L) + 1 for L in lens]))


def test_clamping_and_empty_encodings():
    L = 10
    # negative / beyond-L bounds are clamped; any end <= start is empty
    assert orc.decode_intervals([15, -4, 3, 7, 7], 5, L) == [(0, 10), (0, 3)]
    assert orc.decode_intervals([0, 0, 0, 0, 0], 5, L) == []
    assert orc.decode_intervals([-1, 5, 2, 9, 1], 5, L) == []
    assert orc.visible_row([3, 2, 6, 5, 8], 5, L).sum() == 8  # [0,3) u [2,6) u [5,8) = [0,8)


def test_constant_inputs_closed_form():
    """q = 0.75, k = 0.5 per component (D = 4), v = 1: s = alpha * 1.5 and
    O_i = count_i * silu(s) / N in every component."""
    cfg = wl.CONFIGS["tiny"]
    lens = np.array([23, 11])
    off = wl.offsets_from_lengths(lens)
    func = wl.build_func(cfg, lens)
    T, H, D = int(off[-1]), 2, 4
    q = np.full((T, H, D), 0.75)
    k = np.full((T, H, D), 0.5)
    v = np.ones((T, H, D))
    N, alpha = 23, 0.5
    s = alpha * 1.5
    silu = s / (1.0 + math.exp(-s))
    counts = orc.visible_counts(off, func, 5)
    o = orc.fwd_dense(q, k, v, off, func, 5, N, alpha)
    np.testing.assert_allclose(o, (counts * silu / N)[:, None, None] * np.ones((1, H, D)), rtol=1e-14)


# ---------------------------------------------------------------- targets-only
def test_targets_only_equals_full_candidate_row():
    """MLCommons training PR #903: the candidate row is the same function of
    the same inputs; its gradients equal the full path's when dO is zero off
    the candidate rows."""
    cfg = wl.CONFIGS["dlrm_b1024"]
    lens, off, q, k, v, do = _small_batch(6, [40, 17, 64, 3], H=2, D=16)
    func = wl.build_func(cfg, lens, 1)
    cand = off[1:] - 1
    fc = wl.build_func_candidates(lens, 1)
    assert np.array_equal(fc, func[:, cand])
    N, alpha = 64, 0.25
    o = orc.fwd_dense(q, k, v, off, func, 1, N, alpha)
    oc = orc.fwd_targets_only(q[cand], k, v, off, fc, 1, N, alpha)
    np.testing.assert_allclose(oc, o[cand], rtol=1e-13, atol=1e-15)
    do_full = np.zeros_like(do)
    do_full[cand] = do[cand]
    dq, dk, dv = orc.bwd_dense(do_full, q, k, v, off, func, 1, N, alpha)
    dqc, dkc, dvc = orc.bwd_targets_only(do[cand], q[cand], k, v, off, fc, 1, N, alpha)
    np.testing.assert_allclose(dqc, dq[cand], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dkc, dk, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dvc, dv, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- finite differences
def test_gradients_match_central_differences():
    cfg = wl.CONFIGS["tiny"]
    lens = np.array([13, 6])
    off = wl.offsets_from_lengths(lens)
    func = wl.build_func(cfg, lens)
    _, _, q, k, v, do = _small_batch(7, lens, H=2, D=4)
    N, alpha, h = 13, 0.5, 1e-6

    def loss(q_, k_, v_):
        return float((orc.fwd_dense(q_, k_, v_, off, func, 5, N, alpha) * do).sum())

    dq, dk, dv = orc.bwd_dense(do, q, k, v, off, func, 5, N, alpha)
    rng = np.random.default_rng(0)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, s)) for s in q.shape)
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])) + 1e-9, (which, idx)


def test_rows_with_no_visible_column_are_zero():
    lens, off, q, k, v, do = _small_batch(8, [9, 5])
    func = np.zeros((3, 14), dtype=np.int32)  # every interval empty
    o = orc.fwd_dense(q, k, v, off, func, 3, 9, 0.25)
    assert not o.any()
    dq, dk, dv = orc.bwd_dense(do, q, k, v, off, func, 3, 9, 0.25)
    assert not dq.any() and not dk.any() and not dv.any()


# ---------------------------------------------------------------- several candidates per sequence
def test_multi_candidates_equal_the_full_paths_rows():
    """Candidate rows taken from inside each sequence (any rows, any number,
    none for one sequence) give exactly the full path's rows; the gradients
    equal the full path's when dO is zero off those rows."""
    cfg = wl.CONFIGS["tiny"]
    lens, off, q, k, v, do = _small_batch(12, [40, 17, 64, 3], H=2, D=16)
    func = wl.build_func(cfg, lens, 5)
    picks = [[0, 7, 39], [], [5, 6, 63, 20], [2]]
    rows = np.array([off[b] + i for b, p in enumerate(picks) for i in p])
    cand_off = np.concatenate([[0], np.cumsum([len(p) for p in picks])])
    N, alpha = 64, 0.25
    o = orc.fwd_dense(q, k, v, off, func, 5, N, alpha)
    oc = orc.fwd_targets(q[rows], k, v, off, cand_off, func[:, rows], 5, N, alpha)
    np.testing.assert_allclose(oc, o[rows], rtol=1e-13, atol=1e-15)
    do_full = np.zeros_like(do)
    do_full[rows] = do[rows]
    dq, dk, dv = orc.bwd_dense(do_full, q, k, v, off, func, 5, N, alpha)
    dqc, dkc, dvc = orc.bwd_targets(do[rows], q[rows], k, v, off, cand_off, func[:, rows], 5, N, alpha)
    np.testing.assert_allclose(dqc, dq[rows], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dkc, dk, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(dvc, dv, rtol=1e-12, atol=1e-15)


def test_one_candidate_per_sequence_is_the_targets_only_form():
    cfg = wl.CONFIGS["dlrm_b1024"]
    lens, off, q, k, v, do = _small_batch(13, [30, 9, 50], H=2, D=8)
    fc = wl.build_func_candidates(lens, 3)
    g = torch.Generator().manual_seed(2)
    q_c, do_c = (_np64(wl.randn_bf16((3, 2, 8), g)) for _ in range(2))
    one = np.arange(4)
    np.testing.assert_array_equal(orc.fwd_targets(q_c, k, v, off, one, fc, 3, 50, 0.3),
                                  orc.fwd_targets_only(q_c, k, v, off, fc, 3, 50, 0.3))
    for a, b in zip(orc.bwd_targets(do_c, q_c, k, v, off, one, fc, 3, 50, 0.3),
                    orc.bwd_targets_only(do_c, q_c, k, v, off, fc, 3, 50, 0.3)):
        np.testing.assert_array_equal(a, b)


def test_multi_candidate_gradients_match_central_differences():
    lens = np.array([11, 7])
    off = wl.offsets_from_lengths(lens)
    _, _, _, k, v, _ = _small_batch(14, lens, H=1, D=4)
    g = torch.Generator().manual_seed(5)
    q_c, do_c = (_np64(wl.randn_bf16((5, 1, 4), g)) for _ in range(2))
    cand_off = np.array([0, 3, 5])
    fc = np.array([[11, 4, 6, 7, 2], [2, 0, 1, 3, 0], [9, 11, 3, 7, 7]], dtype=np.int32)  # NFUNC=3
    N, alpha, h = 11, 0.7, 1e-6

    def loss(q_, k_, v_):
        return float((orc.fwd_targets(q_, k_, v_, off, cand_off, fc, 3, N, alpha) * do_c).sum())

    grads = orc.bwd_targets(do_c, q_c, k, v, off, cand_off, fc, 3, N, alpha)
    rng = np.random.default_rng(1)
    for which, grad in enumerate(grads):
        base = (q_c, k, v)[which]
        for _ in range(10):
            idx = tuple(int(rng.integers(0, s_)) for s_ in base.shape)
            args = [q_c.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])) + 1e-9, (which, idx)


# ---------------------------------------------------------------- candidate-row projection
def test_projection_matches_a_per_element_loop():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((9, 5))
    w = rng.standard_normal((4, 5))
    b = rng.standard_normal(4)
    rows = np.array([7, 0, 3])
    y, z = orc.project_rows(x, rows, w, b)
    for i, r in enumerate(rows):
        for o in range(4):
            zz = b[o]
            for d in range(5):
                zz += x[r, d] * w[o, d]
            assert abs(z[i, o] - zz) < 1e-12
            assert abs(y[i, o] - zz / (1.0 + math.exp(-zz))) < 1e-12


def test_projection_identity_weights_give_silu_of_the_rows():
    x = np.linspace(-6, 6, 30).reshape(6, 5)
    rows = np.array([5, 2])
    y, _ = orc.project_rows(x, rows, np.eye(5), None)
    np.testing.assert_allclose(y, x[rows] * torch.sigmoid(torch.tensor(x[rows])).numpy(), rtol=1e-14)


def test_projection_gradients_match_central_differences():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((8, 6))
    w = rng.standard_normal((5, 6))
    b = rng.standard_normal(5)
    rows = np.array([1, 6, 1, 3])  # a repeated row accumulates
    dy = rng.standard_normal((4, 5))
    dx, dw, db = orc.project_rows_backward(dy, x, rows, w, b)
    assert not dx[[0, 2, 4, 5, 7]].any()
    h = 1e-6

    def loss(x_, w_, b_):
        return float((orc.project_rows(x_, rows, w_, b_)[0] * dy).sum())

    for which, grad in ((0, dx), (1, dw), (2, db)):
        for _ in range(8):
            base = (x, w, b)[which]
            idx = tuple(int(rng.integers(0, s_)) for s_ in base.shape)
            args = [x.copy(), w.copy(), b.copy()]
            args[which][idx] += h
            lp = loss(*args)
            args[which][idx] -= 2 * h
            lm = loss(*args)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(grad[idx])) + 1e-9, (which, idx)
