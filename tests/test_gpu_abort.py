"""The abort path inside the real attention kernels, exercised without a
fault: the accumulator hand-off wait of the MMA-issuing thread is made to
give up at once (hstu_attn_test_set_handoff_limit with 1 ns) while the next
work item's TMA copies and MMAs are in flight. Every role must drain what it
issued and free TMEM; the host then reads HSTU_ERR_TIMEOUT from the
workspace, and the same workspace computes correct results afterwards."""
import numpy as np
import pytest
import torch

from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl
from hstu_testutil import GpuBatch, check_grad, check_o, np64

pytestmark = pytest.mark.gpu

HSTU_ERR_TIMEOUT = 6


@pytest.fixture
def batch():
    # ragged, several kv tiles per sequence and far more work items than
    # CTAs, so every CTA takes a second item while its first is in flight
    cfg = wl.Config("abort", 48, 300, 900, 2, 128, "causal", 1)
    return GpuBatch.from_config(cfg, 3)


def _timed(fn):
    e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    e[0].record()
    fn()
    e[1].record()
    torch.cuda.synchronize()
    return e[0].elapsed_time(e[1])


@pytest.mark.parametrize("which", ["fwd", "bwd"])
def test_handoff_wait_runs_out_and_the_workspace_recovers(batch, which):
    gb = batch
    shape = hb.make_shape(len(gb.lens), gb.total, gb.q.shape[1], gb.q.shape[2], gb.nfunc, gb.max_seqlen, gb.alpha)
    ws = hb.alloc_workspace(shape)
    hb.plan(gb.d_off, gb.d_func, shape, ws)
    assert hb.device_status(ws) == hb.HSTU_OK
    o = torch.empty_like(gb.q)
    grads = tuple(torch.empty_like(gb.q) for _ in range(3))

    def launch():
        if which == "fwd":
            hb.fwd(gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws, reuse_plan=True, out=o)
        else:
            hb.bwd(gb.do, gb.q, gb.k, gb.v, gb.d_off, gb.d_func, gb.max_seqlen, gb.alpha, ws=ws, reuse_plan=True,
                   outs=grads)

    hb.set_handoff_limit_for_tests(1)  # nanoseconds: give up at once
    try:
        ms = _timed(launch)
    finally:
        hb.set_handoff_limit_for_tests(0)
    assert hb.device_status(ws) == HSTU_ERR_TIMEOUT
    assert ms < 1000.0  # aborted and drained, far inside the 2 s drain limits
    # the next plan clears the error word; the same workspace computes right
    out = gb.run()  # its own workspace
    hb.plan(gb.d_off, gb.d_func, shape, ws)
    launch()
    torch.cuda.synchronize()
    assert hb.device_status(ws) == hb.HSTU_OK
    if which == "fwd":
        assert torch.equal(o, out["o"])
    else:
        for got, ref in zip(grads, (out["dq"], out["dk"], out["dv"])):
            assert torch.equal(got, ref)
    ref = gb.oracle(seqs=[0, 7, 47])
    rows = torch.as_tensor(ref["rows"], device="cuda")
    check_o(np64(out["o"].index_select(0, rows)), ref["o"])
    check_grad(np64(out["dk"].index_select(0, rows)), ref["dk"], "dk")

