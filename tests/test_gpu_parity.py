"""GPU parity: the CUDA path (through the C ABI) against the CPU fp64 oracle.

Small batches are compared element by element in full; the full-size
workloads are run whole on the GPU and compared on a seeded sample of
sequences (always holding the longest and the shortest one).
"""
import math

import numpy as np
import pytest
import torch

import oracle.hstu_oracle as orc
from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl
from hstu_testutil import GpuBatch, check_grad, check_o, compare, np64, sample_seqs

pytestmark = pytest.mark.gpu


def _gen(lens, H, D, seed):
    T = int(np.sum(lens))
    g = torch.Generator().manual_seed(seed)
    return [wl.randn_bf16((T, H, D), g) for _ in range(4)]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_full_parity(seed):
    gb = GpuBatch.from_config(wl.CONFIGS["tiny"], seed)
    compare(gb.run(), gb.oracle())


@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("mask", ["tiny", "sla", "causal", "onerank"])
def test_ragged_tails_all_masks(D, mask):
    """Lengths that end mid-tile, a one-row and an empty sequence, several
    tiles per sequence, every mask family, every head size."""
    lens = [1, 130, 0, 300, 127, 257] if mask != "onerank" else [40, 300, 129, 257]
    nfunc = 1 if mask == "causal" else 5
    cfg = wl.Config("t", len(lens), 0, 0, 2, D, mask, nfunc, k1=70, k2=20)
    func = wl.build_func(cfg, np.array(lens), nfunc)
    q, k, v, do = _gen(lens, 2, D, seed=D)
    gb = GpuBatch(lens, func, q, k, v, do, max_seqlen=320)
    compare(gb.run(), gb.oracle())


def test_item_hand_offs_with_every_tile_count():
    """Hundreds of short work items whose visited-tile counts run through
    1..6 (with runs that are multiples of three) and empty sequences among
    them: the forward's O read-out moves between epilogue groups from item
    to item and the backward's roles alternate in windows, so every
    hand-off order occurs; the whole batch is compared with the oracle."""
    rng = np.random.default_rng(7)
    pattern = [384, 384, 384, 0, 128, 1, 768, 640, 256, 0, 512, 130, 384, 384, 700, 3]
    lens = np.array([pattern[i % len(pattern)] if i % 5 else int(rng.integers(1, 769))
                     for i in range(96)])
    cfg = wl.Config("h", len(lens), 0, 0, 2, 64, "causal", 1)
    func = wl.build_func(cfg, lens, 1)
    q, k, v, do = _gen(lens, 2, 64, seed=5)
    gb = GpuBatch(lens, func, q, k, v, do, max_seqlen=768)
    compare(gb.run(), gb.oracle())


@pytest.mark.parametrize("nfunc", [1, 3, 5, 7, 9])
def test_random_intervals(nfunc):
    """Arbitrary (also negative, out-of-range, reversed) func values."""
    lens = np.array([200, 77, 384, 5])
    T = int(lens.sum())
    rng = np.random.default_rng(nfunc)
    func = rng.integers(-20, 420, size=(nfunc, T)).astype(np.int32)
    q, k, v, do = _gen(lens, 3, 64, seed=11)
    gb = GpuBatch(lens, func, q, k, v, do, max_seqlen=400)
    compare(gb.run(), gb.oracle())


def test_all_intervals_empty_gives_zeros():
    lens = np.array([150, 40])
    func = np.zeros((3, 190), dtype=np.int32)
    q, k, v, do = _gen(lens, 2, 128, seed=3)
    gb = GpuBatch(lens, func, q, k, v, do)
    out = gb.run()
    for n in ("o", "dq", "dk", "dv"):
        assert not out[n].any(), n
    assert not out["counts"].any()


@pytest.mark.parametrize("nfunc_padded", [5, 9])
def test_sla_padding_is_bitwise_inert(nfunc_padded):
    cfg = wl.CONFIGS["sla_b32_s1024"]
    gp = GpuBatch.from_config(cfg, 0, nfunc=nfunc_padded)
    g3 = GpuBatch(gp.lens, gp.func[:3], gp.q, gp.k, gp.v, gp.do)
    a, b = gp.run(), g3.run()
    for n in ("o", "dq", "dk", "dv", "counts"):
        assert torch.equal(a[n], b[n]), n


@pytest.mark.parametrize("name", ["sla_b32_s1024", "sla_b16_s2048", "onerank_b64"])
def test_config_parity_sampled(name):
    cfg = wl.CONFIGS[name]
    gb = GpuBatch.from_config(cfg, 0)
    out = gb.run()
    seqs = sample_seqs(gb.lens, 4)
    compare(out, gb.oracle(seqs))
    # visible counts of every row, bitwise
    ref_counts = orc.visible_counts(gb.offsets, gb.func, gb.nfunc)
    assert np.array_equal(out["counts"].cpu().numpy(), ref_counts)


def test_dlrm_full_length_sampled():
    cfg = wl.CONFIGS["dlrm_b1024"]
    gb = GpuBatch.from_config(cfg, 0, device="cuda")
    out = gb.run()
    seqs = sample_seqs(gb.lens, 3)
    compare(out, gb.oracle(seqs))
    # causal counts of every row: i + 1, closed form
    exp = np.concatenate([np.arange(L) + 1 for L in gb.lens])
    assert np.array_equal(out["counts"].cpu().numpy(), exp)


def _targets_inputs(gb, seed=5):
    B = len(gb.lens)
    H, D = gb.q.shape[1], gb.q.shape[2]
    g = torch.Generator(device="cuda").manual_seed(seed)
    q_c = wl.randn_bf16((B, H, D), g, "cuda")
    do_c = wl.randn_bf16((B, H, D), g, "cuda")
    func_c = wl.build_func_candidates(gb.lens, gb.nfunc)
    return q_c, do_c, func_c


def _run_targets(gb, q_c, do_c, func_c):
    d_fc = torch.tensor(func_c, dtype=torch.int32, device="cuda")
    shape = hb.make_shape(len(gb.lens), gb.total, gb.q.shape[1], gb.q.shape[2], gb.nfunc, gb.max_seqlen,
                          gb.alpha)
    ws = hb.alloc_workspace(shape, hb.WS_TARGETS)
    o_c = hb.fwd_targets_only(q_c, gb.k, gb.v, gb.d_off, d_fc, gb.max_seqlen, gb.alpha, ws=ws)
    dq_c, dk, dv = hb.bwd_targets_only(do_c, q_c, gb.k, gb.v, gb.d_off, d_fc, gb.max_seqlen, gb.alpha, ws=ws)
    assert hb.device_status(ws) == hb.HSTU_OK
    return o_c, dq_c, dk, dv


def test_targets_only_equals_full_candidate_row():
    """Targets-only output equals the full path's candidate row on the GPU,
    and both match the oracle."""
    lens = np.array([300, 1, 129, 513, 64])
    cfg = wl.Config("c", 5, 0, 0, 2, 128, "causal", 1)
    func = wl.build_func(cfg, lens, 1)
    q, k, v, do = _gen(lens, 2, 128, seed=9)
    gb = GpuBatch(lens, func, q, k, v, do)
    cand = torch.as_tensor(gb.offsets[1:] - 1, device="cuda")
    q_c = gb.q.index_select(0, cand).contiguous()
    do_c = gb.do.index_select(0, cand).contiguous()
    func_c = wl.build_func_candidates(lens, 1)
    o_c, dq_c, dk, dv = _run_targets(gb, q_c, do_c, func_c)
    full = gb.run(want_bwd=False)["o"].index_select(0, cand)
    check_o(np64(o_c), np64(full).astype(np.float64), "targets vs full row")
    ref = orc.fwd_targets_only(np64(q_c), np64(gb.k), np64(gb.v), gb.offsets, func_c, 1, gb.max_seqlen, gb.alpha)
    check_o(np64(o_c), ref)
    rdq, rdk, rdv = orc.bwd_targets_only(np64(do_c), np64(q_c), np64(gb.k), np64(gb.v), gb.offsets, func_c, 1,
                                         gb.max_seqlen, gb.alpha)
    check_grad(np64(dq_c), rdq, "dq_c")
    check_grad(np64(dk), rdk, "dk")
    check_grad(np64(dv), rdv, "dv")


@pytest.mark.parametrize("nfunc", [3, 5, 7, 9])
def test_targets_only_interval_masks(nfunc):
    lens = np.array([700, 33, 260])
    T = int(lens.sum())
    rng = np.random.default_rng(nfunc + 7)
    q, k, v, do = _gen(lens, 4, 64, seed=13)
    gb = GpuBatch(lens, np.zeros((nfunc, T), np.int32), q, k, v, do)
    func_c = rng.integers(-10, 720, size=(nfunc, 3)).astype(np.int32)
    g = torch.Generator().manual_seed(3)
    q_c = wl.randn_bf16((3, 4, 64), g).cuda()
    do_c = wl.randn_bf16((3, 4, 64), g).cuda()
    o_c, dq_c, dk, dv = _run_targets(gb, q_c, do_c, func_c)
    ref = orc.fwd_targets_only(np64(q_c), np64(gb.k), np64(gb.v), gb.offsets, func_c, nfunc, gb.max_seqlen,
                               gb.alpha)
    check_o(np64(o_c), ref)
    rdq, rdk, rdv = orc.bwd_targets_only(np64(do_c), np64(q_c), np64(gb.k), np64(gb.v), gb.offsets, func_c,
                                         nfunc, gb.max_seqlen, gb.alpha)
    check_grad(np64(dq_c), rdq, "dq_c")
    check_grad(np64(dk), rdk, "dk")
    check_grad(np64(dv), rdv, "dv")


def test_dlrm_targets_only_full_size():
    cfg = wl.CONFIGS["dlrm_b1024"]
    gb = GpuBatch.from_config(cfg, 0, device="cuda")
    q_c, do_c, func_c = _targets_inputs(gb)
    o_c, dq_c, dk, dv = _run_targets(gb, q_c, do_c, func_c)
    # forward and dq_c for every sequence: the oracle does one row each
    ref_o = orc.fwd_targets_only(np64(q_c), np64(gb.k), np64(gb.v), gb.offsets, func_c, 1, gb.max_seqlen,
                                 gb.alpha)
    check_o(np64(o_c), ref_o)
    # dk/dv on sampled sequences (full fp64 copies of dk/dv would be 2.8 GB each)
    seqs = sample_seqs(gb.lens, 4)
    rows, sub_off, _, (q, k, v, do) = gb.sub(seqs)
    fc = func_c[:, seqs]
    rdq, rdk, rdv = orc.bwd_targets_only(np64(do_c[seqs]), np64(q_c[seqs]), k, v, sub_off, fc, 1,
                                         gb.max_seqlen, gb.alpha)
    ridx = torch.as_tensor(rows, device="cuda")
    check_grad(np64(dq_c[seqs]), rdq, "dq_c")
    check_grad(np64(dk.index_select(0, ridx)), rdk, "dk")
    check_grad(np64(dv.index_select(0, ridx)), rdv, "dv")


@pytest.mark.parametrize("lens", [[5], [130], [5, 130, 64]])
def test_small_batches_never_reach_a_wait_limit(lens):
    """A CTA that uses only some of its ring slots must not wait on the
    others at exit: each launch on a tiny batch ends far inside the 2 s limit
    of the in-kernel waits."""
    lens = np.array(lens)
    q, k, v, do = _gen(lens, 1, 64, seed=5)
    gb = GpuBatch(lens, wl.build_func(wl.Config("c", len(lens), 0, 0, 1, 64, "causal", 1), lens, 1),
                  q, k, v, do)
    gb.run()  # warm-up: library load, first launches
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    e[0].record()
    out = gb.run()
    e[1].record()
    torch.cuda.synchronize()
    assert e[0].elapsed_time(e[1]) < 200.0  # milliseconds
    compare(out, gb.oracle())


def test_many_short_sequences_all_items_run():
    """Eight thousand sequences of mixed length (zero included): the plan's
    list builder takes several rounds per thread, and its warps hold
    sequences of several tile counts at once. Every row of every output is
    written (the outputs start as NaN), the visible counts are exactly
    i + 1 (causal), and sampled sequences match the oracle."""
    rng = np.random.default_rng(11)
    lens = rng.integers(1, 300, size=8000)
    lens[rng.choice(len(lens), 400, replace=False)] = 0
    H, D = 1, 32
    q, k, v, do = _gen(lens, H, D, seed=11)
    gb = GpuBatch(lens, wl.build_func(wl.Config("many", len(lens), 0, 0, H, D, "causal", 1), lens, 1),
                  q, k, v, do)
    T = gb.total
    shape = hb.make_shape(len(lens), T, H, D, 1, gb.max_seqlen, gb.alpha)
    ws = hb.alloc_workspace(shape)
    counts = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    o = torch.full_like(gb.q, float("nan"))
    grads = tuple(torch.full_like(gb.q, float("nan")) for _ in range(3))
    hb.fwd(gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws, row_counts=counts, out=o)
    hb.bwd(gb.do, gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws, reuse_plan=True,
           outs=grads)
    torch.cuda.synchronize()
    assert hb.device_status(ws) == hb.HSTU_OK
    for name, t in zip(("o", "dq", "dk", "dv"), (o,) + grads):
        assert not torch.isnan(t).any(), f"{name}: rows left unwritten"
    local = np.arange(T) - np.repeat(gb.offsets[:-1], lens)
    assert np.array_equal(counts.cpu().numpy(), local + 1)
    nz = np.nonzero(lens)[0]
    seqs = [int(nz[0]), int(np.argmax(lens)), int(nz[np.argmin(lens[nz])]), int(nz[-1]), int(nz[len(nz) // 2])]
    compare({"o": o, "dq": grads[0], "dk": grads[1], "dv": grads[2], "counts": counts}, gb.oracle(seqs))


def test_batch_of_empty_sequences():
    """No rows at all: every entry point accepts it, writes nothing, and the
    targets-only candidates (which see no key) get zeros."""
    lens = np.array([0, 0, 0])
    q, k, v, do = _gen(lens, 2, 64, seed=2)
    gb = GpuBatch(lens, np.zeros((3, 0), np.int32), q, k, v, do, max_seqlen=16)
    out = gb.run()
    for n in ("o", "dq", "dk", "dv"):
        assert out[n].numel() == 0, n
    g = torch.Generator().manual_seed(4)
    q_c = wl.randn_bf16((3, 2, 64), g).cuda()
    do_c = wl.randn_bf16((3, 2, 64), g).cuda()
    o_c, dq_c, dk, dv = _run_targets(gb, q_c, do_c, np.zeros((3, 3), np.int32))
    assert not o_c.any() and not dq_c.any()
    assert dk.numel() == 0 and dv.numel() == 0


def test_wait_timeout_reaches_the_host_and_the_context_stays_usable():
    """A bounded in-kernel wait that nothing ends gives up after its limit and
    reports HSTU_ERR_TIMEOUT through the workspace; the next plan clears it and
    the same workspace runs the op correctly."""
    lens = np.array([130, 7])
    q, k, v, do = _gen(lens, 2, 64, seed=8)
    func = wl.build_func(wl.Config("c", 2, 0, 0, 2, 64, "causal", 1), lens, 1)
    gb = GpuBatch(lens, func, q, k, v, do)
    shape = hb.make_shape(2, gb.total, 2, 64, 1, gb.max_seqlen, gb.alpha)
    ws = hb.alloc_workspace(shape)
    hb.plan(gb.d_off, gb.d_func, shape, ws)
    assert hb.device_status(ws) == hb.HSTU_OK
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    e[0].record()
    hb.selftest_wait_timeout(ws, 20)
    e[1].record()
    assert hb.device_status(ws) == 6  # HSTU_ERR_TIMEOUT
    assert 19.0 <= e[0].elapsed_time(e[1]) < 1000.0
    o = hb.fwd(gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws)
    assert hb.device_status(ws) == hb.HSTU_OK
    ref = gb.oracle(want_bwd=False)
    check_o(np64(o), ref["o"])


def test_backward_is_bitwise_repeatable():
    gb = GpuBatch.from_config(wl.CONFIGS["onerank_b64"], 1)
    a = gb.run()
    for _ in range(5):
        b = gb.run()
        for n in ("o", "dq", "dk", "dv"):
            assert torch.equal(a[n], b[n]), n


def test_maximum_sequence_length():
    """One sequence of the maximum length (32768 rows, 256 tiles), causal.
    dO is zero except on a few rows, so dK, dV and dQ over the whole sequence
    are the sum of those rows' contributions, which the oracle computes one
    row at a time (the targets-only routine is the full op's row); O is
    checked on sampled rows the same way, and the visible counts in full."""
    L, H, D = 32768, 1, 128
    lens = np.array([L])
    g = torch.Generator().manual_seed(21)
    q, k, v = (wl.randn_bf16((L, H, D), g) for _ in range(3))
    rows = [0, 127, 128, 20000, 32639, L - 1]
    do = torch.zeros((L, H, D), dtype=torch.bfloat16)
    do[rows] = wl.randn_bf16((len(rows), H, D), g)
    func = wl.build_func(wl.Config("c", 1, 0, 0, H, D, "causal", 1), lens, 1)
    gb = GpuBatch(lens, func, q, k, v, do)
    out = gb.run()
    assert np.array_equal(out["counts"].cpu().numpy(), np.arange(L) + 1)
    hq, hk, hv, hdo = (np64(t) for t in (q, k, v, do))
    off = np.array([0, L])
    ref_dk, ref_dv = np.zeros_like(hk), np.zeros_like(hv)
    ref_dq = np.zeros_like(hq)
    for r in rows + [1, 129, 4095, 31000]:
        fc = func[:, r:r + 1]
        o_r = orc.fwd_targets_only(hq[r:r + 1], hk, hv, off, fc, 1, L, gb.alpha)
        check_o(np64(out["o"][r:r + 1]), o_r)
        if r in rows:
            dq_r, dk_r, dv_r = orc.bwd_targets_only(hdo[r:r + 1], hq[r:r + 1], hk, hv, off, fc, 1, L, gb.alpha)
            ref_dq[r:r + 1] = dq_r
            ref_dk += dk_r
            ref_dv += dv_r
    check_grad(np64(out["dq"]), ref_dq, "dq")
    check_grad(np64(out["dk"]), ref_dk, "dk")
    check_grad(np64(out["dv"]), ref_dv, "dv")


def test_results_do_not_depend_on_the_rest_of_the_batch():
    """A sequence's outputs are bitwise the same alone or inside a batch (with
    the same N): every output element is computed by one CTA in a fixed order
    from that sequence's rows only."""
    lens = np.array([300, 129, 77])
    q, k, v, do = _gen(lens, 2, 128, seed=12)
    cfg = wl.Config("s", 3, 0, 0, 2, 128, "sla", 5, k1=100, k2=20)
    full = GpuBatch(lens, wl.build_func(cfg, lens, 5), q, k, v, do, max_seqlen=300)
    a = full.run()
    r0, r1 = 300, 429  # rows of the second sequence
    alone_lens = np.array([129])
    one = GpuBatch(alone_lens, wl.build_func(cfg, alone_lens, 5), q[r0:r1], k[r0:r1], v[r0:r1], do[r0:r1],
                   max_seqlen=300)
    b = one.run()
    for n in ("o", "dq", "dk", "dv", "counts"):
        assert torch.equal(a[n][r0:r1], b[n]), n


@pytest.mark.parametrize("bad_offsets", [[0, 120, 150],   # L_0 = 120 > max_seqlen 100
                                         [0, 100, 140],   # last offset is not total (150)
                                         [0, 100, 90],    # decreasing
                                         [10, 100, 150]])  # first offset is not 0
def test_device_side_offset_error_sets_status_and_writes_nothing(bad_offsets):
    lens = np.array([100, 50])
    q, k, v, do = _gen(lens, 2, 64, seed=1)
    func = wl.build_func(wl.Config("c", 2, 0, 0, 2, 64, "causal", 1), lens, 1)
    gb = GpuBatch(lens, func, q, k, v, do)
    bad = torch.tensor(bad_offsets, dtype=torch.int32, device="cuda")
    shape = hb.make_shape(2, 150, 2, 64, 1, 100, gb.alpha)
    ws = hb.alloc_workspace(shape)
    o = torch.full_like(gb.q, 7.0)
    hb.fwd(gb.q, gb.k, gb.v, bad, gb.d_func, 100, gb.alpha, ws=ws, out=o)
    assert hb.device_status(ws) == 5  # HSTU_ERR_DEVICE_INPUT
    assert torch.all(o == 7.0)
    grads = tuple(torch.full_like(gb.q, 7.0) for _ in range(3))
    hb.bwd(gb.do, gb.q, gb.k, gb.v, bad, gb.d_func, 100, gb.alpha, ws=ws, outs=grads)
    assert hb.device_status(ws) == 5
    assert all(torch.all(t == 7.0) for t in grads)
    # targets-only reports the same offsets, and leaves o_c and dq_c alone
    tshape = hb.make_shape(2, 150, 2, 64, 1, 100, gb.alpha)
    tws = hb.alloc_workspace(tshape, hb.WS_TARGETS)
    q_c = gb.q[:2].clone()
    fc = torch.tensor([[100, 50]], dtype=torch.int32, device="cuda")
    o_c = torch.full_like(q_c, 7.0)
    hb.fwd_targets_only(q_c, gb.k, gb.v, bad, fc, 100, gb.alpha, ws=tws, out=o_c)
    assert hb.device_status(tws) == 5
    assert torch.all(o_c == 7.0)
    # the same workspace recovers with valid offsets
    o2 = hb.fwd(gb.q, gb.k, gb.v, gb.d_off, gb.d_func, 100, gb.alpha, ws=ws)
    assert hb.device_status(ws) == hb.HSTU_OK
    assert torch.isfinite(o2.float()).all()


def _launch(gb, ws, shape, reuse):
    o = hb.fwd(gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws, reuse_plan=reuse)
    dq, dk, dv = hb.bwd(gb.do, gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws,
                        reuse_plan=True)
    torch.cuda.synchronize()
    assert hb.device_status(ws) == hb.HSTU_OK
    return {"o": o, "dq": dq, "dk": dk, "dv": dv}


def test_reused_plan_hands_out_all_work_every_launch():
    # A ragged batch takes its work from device counters; they must be back
    # at zero after every launch, or a later launch on the same plan would
    # find no work left.
    gb = GpuBatch.from_config(wl.CONFIGS["onerank_b64"], 3)
    shape = hb.make_shape(len(gb.lens), gb.total, gb.q.shape[1], gb.q.shape[2], gb.nfunc, gb.max_seqlen,
                          gb.alpha)
    ws = hb.alloc_workspace(shape, hb.WS_FULL)
    first = _launch(gb, ws, shape, reuse=False)
    for _ in range(3):
        again = _launch(gb, ws, shape, reuse=True)
        for n in ("o", "dq", "dk", "dv"):
            assert torch.equal(first[n], again[n]), n
    sub = sample_seqs(gb.lens, 3, seed=0)
    ref = gb.oracle(sub)
    rows = torch.as_tensor(ref["rows"], device="cuda", dtype=torch.long)
    check_o(np64(first["o"].index_select(0, rows)), ref["o"])
    check_grad(np64(first["dq"].index_select(0, rows)), ref["dq"], "dq")


def test_workspace_switches_between_equal_length_and_ragged_batches():
    # An equal-length batch is split by a fixed stride, a ragged one through
    # the counters; one workspace serves both in turn.
    uni = GpuBatch.from_config(wl.CONFIGS["sla_b32_s1024"], 0)
    rag = GpuBatch.from_config(wl.CONFIGS["tiny"], 5)
    big = hb.make_shape(len(uni.lens), uni.total, uni.q.shape[1], uni.q.shape[2], uni.nfunc, uni.max_seqlen,
                        uni.alpha)
    ws = hb.alloc_workspace(big, hb.WS_FULL)
    for gb in (rag, uni, rag):
        shape = hb.make_shape(len(gb.lens), gb.total, gb.q.shape[1], gb.q.shape[2], gb.nfunc, gb.max_seqlen,
                              gb.alpha)
        assert ws.numel() >= hb.workspace_size(shape, hb.WS_FULL)
        out = _launch(gb, ws, shape, reuse=False)
        out2 = _launch(gb, ws, shape, reuse=True)
        for n in ("o", "dq", "dk", "dv"):
            assert torch.equal(out[n], out2[n]), n
    ref = rag.oracle()
    check_o(np64(out["o"]), ref["o"])
    check_grad(np64(out["dk"]), ref["dk"], "dk")
