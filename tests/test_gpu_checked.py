"""The checked build (libhstu_attn_checked.so, compiled with HSTU_CHECKED).

On valid batches it must give the release build's results bit for bit and
report no error. With a bad entry planted in the plan's work list (a
sequence outside the batch, or a tile past the end of its sequence), its
kernels must refuse the entry before any load or store goes through it,
finish promptly and record HSTU_ERR_DEVICE_CHECK; the same workspace,
planned again, computes the oracle's results. The bad entries are only ever
given to the checked build."""
import numpy as np
import pytest
import torch

from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl
from hstu_testutil import GpuBatch, compare

pytestmark = pytest.mark.gpu

HSTU_ERR_DEVICE_CHECK = 7
ROLE_DKDV = 1 << 30


@pytest.fixture
def checked():
    prev = hb.select_library(hb.CHECKED_LIB_PATH)
    try:
        yield
    finally:
        hb.select_library(prev)


@pytest.fixture(scope="module")
def batch():
    # ragged lengths with partial tails, nfunc 3 (a causal mask plus a band)
    cfg = wl.Config("checked", 40, 200, 700, 2, 128, "sla", 3)
    return GpuBatch.from_config(cfg, 5)


def _shape(gb):
    return hb.make_shape(len(gb.lens), gb.total, gb.q.shape[1], gb.q.shape[2], gb.nfunc, gb.max_seqlen, gb.alpha)


def _list_offsets(gb):
    """Byte offsets of the forward and backward work lists in the workspace:
    a 256-byte header, then (batch x tiles-per-sequence) int32 entries for
    each list, every region rounded up to 256 bytes."""
    nt = (gb.max_seqlen + 127) // 128
    items = len(gb.lens) * nt
    fwd = 256
    bwd = fwd + (items * 4 + 255) // 256 * 256
    return fwd, bwd


def _plant(ws, byte_offset, code):
    ws[byte_offset:byte_offset + 4].view(torch.int32).fill_(code)


def _timed(fn):
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    e[0].record()
    fn()
    e[1].record()
    torch.cuda.synchronize()
    return e[0].elapsed_time(e[1])


def test_checked_build_equals_release_bitwise(batch):
    release = batch.run()
    prev = hb.select_library(hb.CHECKED_LIB_PATH)
    try:
        got = batch.run()  # asserts HSTU_OK inside
    finally:
        hb.select_library(prev)
    for name in ("o", "dq", "dk", "dv", "counts"):
        assert torch.equal(got[name], release[name]), name


def _bad_codes(gb):
    short = int(np.argmin(gb.lens))  # fewest tiles
    past_end = (int(gb.lens[short]) + 127) // 128 + 1
    return {
        "sequence_outside_batch": (len(gb.lens) + 3) << 8,
        "tile_past_sequence_end": (short << 8) | past_end,
    }


@pytest.mark.parametrize("which", ["fwd", "bwd_dkdv", "bwd_dq"])
@pytest.mark.parametrize("bad", ["sequence_outside_batch", "tile_past_sequence_end"])
def test_bad_list_entry_is_refused(batch, checked, which, bad):
    gb = batch
    shape = _shape(gb)
    ws = hb.alloc_workspace(shape)
    fwd_off, bwd_off = _list_offsets(gb)
    code = _bad_codes(gb)[bad]
    o = torch.empty_like(gb.q)
    grads = tuple(torch.empty_like(gb.q) for _ in range(3))

    hb.plan(gb.d_off, gb.d_func, shape, ws)
    assert hb.device_status(ws) == hb.HSTU_OK
    if which == "fwd":
        _plant(ws, fwd_off, code)
        ms = _timed(lambda: hb.fwd(gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws,
                                   reuse_plan=True, out=o))
    else:
        _plant(ws, bwd_off, code | (ROLE_DKDV if which == "bwd_dkdv" else 0))
        ms = _timed(lambda: hb.bwd(gb.do, gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws,
                                   reuse_plan=True, outs=grads))
    assert hb.device_status(ws) == HSTU_ERR_DEVICE_CHECK
    assert ms < 1000.0

    # planned again (by the forward), the same workspace computes the
    # oracle's results
    counts = torch.full((gb.total,), -1, dtype=torch.int32, device="cuda")
    o = hb.fwd(gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws, row_counts=counts, out=o)
    dq, dk, dv = hb.bwd(gb.do, gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws,
                        reuse_plan=True, outs=grads)
    torch.cuda.synchronize()
    assert hb.device_status(ws) == hb.HSTU_OK
    seqs = [0, int(np.argmax(gb.lens)), len(gb.lens) - 1]
    compare({"o": o, "dq": dq, "dk": dk, "dv": dv, "counts": counts}, gb.oracle(seqs))
