"""Targets-only mode with any number of candidates per sequence
(hstu_attn_fwd_targets / hstu_attn_bwd_targets) against the oracle, and
against the one-candidate entry points."""
import numpy as np
import pytest
import torch

import oracle.hstu_oracle as orc
from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl
from hstu_testutil import check_grad, check_o, np64

pytestmark = pytest.mark.gpu


def _setup(lens, counts, H, dq, dv, nfunc, seed, dtype=torch.bfloat16):
    lens = np.asarray(lens)
    off = wl.offsets_from_lengths(lens)
    T, C = int(off[-1]), int(np.sum(counts))
    g = torch.Generator().manual_seed(seed)
    k = wl.randn((T, H, dq), g, dtype=dtype).cuda()
    v = wl.randn((T, H, dv), g, dtype=dtype).cuda()
    q_c = wl.randn((C, H, dq), g, dtype=dtype).cuda()
    do_c = wl.randn((C, H, dv), g, dtype=dtype).cuda()
    cand_off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    rng = np.random.default_rng(seed)
    # per candidate: a causal row somewhere in its sequence, with extra random intervals
    func_c = np.zeros((nfunc, C), dtype=np.int32)
    for b, L in enumerate(lens):
        for c in range(cand_off[b], cand_off[b + 1]):
            func_c[0, c] = int(rng.integers(0, L + 1))
            for t in range(1, nfunc):
                func_c[t, c] = int(rng.integers(-5, L + 6))
    return off, cand_off, k, v, q_c, do_c, func_c


def _run(off, cand_off, k, v, q_c, do_c, func_c, N, alpha):
    d_off = torch.tensor(off, dtype=torch.int32, device="cuda")
    d_coff = torch.tensor(cand_off, dtype=torch.int32, device="cuda")
    d_fc = torch.tensor(func_c, dtype=torch.int32, device="cuda")
    o_c = hb.fwd_targets(q_c, k, v, d_off, d_coff, d_fc, N, alpha)
    grads = hb.bwd_targets(do_c, q_c, k, v, d_off, d_coff, d_fc, N, alpha)
    torch.cuda.synchronize()
    return o_c, grads


def _check(off, cand_off, k, v, q_c, do_c, func_c, nfunc, N, alpha, o_c, grads):
    hk, hv, hq, hdo = np64(k), np64(v), np64(q_c), np64(do_c)
    check_o(np64(o_c), orc.fwd_targets(hq, hk, hv, off, cand_off, func_c, nfunc, N, alpha))
    ref = orc.bwd_targets(hdo, hq, hk, hv, off, cand_off, func_c, nfunc, N, alpha)
    for got, r, n in zip(grads, ref, ("dq_c", "dk", "dv")):
        check_grad(np64(got), r, n)


@pytest.mark.parametrize("dq,dv", [(128, 128), (64, 128), (128, 32)])
def test_several_candidates_per_sequence(dq, dv):
    lens, counts = [700, 33, 260, 1, 513], [10, 0, 3, 1, 25]
    off, cand_off, k, v, q_c, do_c, func_c = _setup(lens, counts, 2, dq, dv, 5, seed=dq + dv)
    N, alpha = 700, 1.0 / np.sqrt(dq)
    o_c, grads = _run(off, cand_off, k, v, q_c, do_c, func_c, N, alpha)
    _check(off, cand_off, k, v, q_c, do_c, func_c, 5, N, alpha, o_c, grads)


def test_fp16_several_candidates():
    lens, counts = [300, 129, 64], [4, 7, 2]
    off, cand_off, k, v, q_c, do_c, func_c = _setup(lens, counts, 3, 128, 128, 3, seed=4, dtype=torch.float16)
    o_c, grads = _run(off, cand_off, k, v, q_c, do_c, func_c, 300, 0.088)
    _check(off, cand_off, k, v, q_c, do_c, func_c, 3, 300, 0.088, o_c, grads)


def test_one_candidate_each_equals_the_single_target_entry_points():
    lens, counts = [400, 77, 256], [1, 1, 1]
    off, cand_off, k, v, q_c, do_c, func_c = _setup(lens, counts, 2, 128, 128, 1, seed=8)
    N, alpha = 400, 0.088
    o_c, grads = _run(off, cand_off, k, v, q_c, do_c, func_c, N, alpha)
    d_off = torch.tensor(off, dtype=torch.int32, device="cuda")
    d_fc = torch.tensor(func_c, dtype=torch.int32, device="cuda")
    o1 = hb.fwd_targets_only(q_c, k, v, d_off, d_fc, N, alpha)
    g1 = hb.bwd_targets_only(do_c, q_c, k, v, d_off, d_fc, N, alpha)
    assert torch.equal(o_c, o1)
    assert torch.equal(grads[0], g1[0])
    # dk/dv: one candidate's rank-1 rows in both forms (same arithmetic order)
    assert torch.equal(grads[1], g1[1]) and torch.equal(grads[2], g1[2])


def test_candidates_at_the_full_paths_rows_match_the_full_path():
    """Candidates taken from real rows of each sequence (with their own func
    columns) give the full path's outputs at those rows."""
    cfg = wl.CONFIGS["onerank_b64"]
    lens = np.array([600, 129, 900])
    T = int(lens.sum())
    off = wl.offsets_from_lengths(lens)
    func = wl.build_func(cfg, lens)
    g = torch.Generator().manual_seed(6)
    q, k, v = (wl.randn_bf16((T, 2, 128), g).cuda() for _ in range(3))
    picks = [[599, 598, 10], [128], [899, 450, 0, 1, 2]]
    rows = np.array([off[b] + i for b, p in enumerate(picks) for i in p])
    cand_off = np.concatenate([[0], np.cumsum([len(p) for p in picks])])
    d_off = torch.tensor(off, dtype=torch.int32, device="cuda")
    d_func = torch.tensor(func, dtype=torch.int32, device="cuda")
    N, alpha = 900, 0.088
    o_full = hb.fwd(q, k, v, d_off, d_func, N, alpha)
    ridx = torch.as_tensor(rows, device="cuda")
    o_c = hb.fwd_targets(q.index_select(0, ridx).contiguous(), k, v, d_off,
                         torch.tensor(cand_off, dtype=torch.int32, device="cuda"),
                         torch.tensor(np.ascontiguousarray(func[:, rows]), dtype=torch.int32, device="cuda"), N,
                         alpha)
    check_o(np64(o_c), np64(o_full.index_select(0, ridx)), "candidates vs full rows")


def test_no_candidates_at_all_writes_zero_key_gradients():
    lens, counts = [50, 70], [0, 0]
    off, cand_off, k, v, q_c, do_c, func_c = _setup(lens, counts, 2, 64, 64, 1, seed=2)
    o_c, (dq_c, dk, dv) = _run(off, cand_off, k, v, q_c, do_c, func_c, 70, 0.125)
    assert o_c.numel() == 0 and dq_c.numel() == 0
    assert not dk.any() and not dv.any()


def test_bad_candidate_offsets_are_reported():
    lens, counts = [50, 70], [2, 3]
    off, cand_off, k, v, q_c, do_c, func_c = _setup(lens, counts, 2, 64, 64, 1, seed=3)
    d_off = torch.tensor(off, dtype=torch.int32, device="cuda")
    d_fc = torch.tensor(func_c, dtype=torch.int32, device="cuda")
    shape = hb.make_shape(2, int(off[-1]), 2, 64, 1, 70, 0.125)
    for bad in ([0, 3, 2], [1, 2, 5], [0, 2, 4]):  # decreasing, first not 0, last not C
        ws = hb.targets_workspace(shape, 5)
        o_c = torch.full((5, 2, 64), 7.0, dtype=torch.bfloat16, device="cuda")
        hb.fwd_targets(q_c, k, v, d_off, torch.tensor(bad, dtype=torch.int32, device="cuda"), d_fc, 70, 0.125,
                       ws=ws, out=o_c)
        assert hb.device_status(ws) == 5, bad  # HSTU_ERR_DEVICE_INPUT
        assert torch.all(o_c == 7.0)


def test_multi_candidate_backward_is_bitwise_repeatable():
    lens, counts = [700, 260], [12, 5]
    off, cand_off, k, v, q_c, do_c, func_c = _setup(lens, counts, 2, 128, 128, 3, seed=9)
    a = _run(off, cand_off, k, v, q_c, do_c, func_c, 700, 0.088)
    for _ in range(3):
        b = _run(off, cand_off, k, v, q_c, do_c, func_c, 700, 0.088)
        assert torch.equal(a[0], b[0])
        for x, y in zip(a[1], b[1]):
            assert torch.equal(x, y)
