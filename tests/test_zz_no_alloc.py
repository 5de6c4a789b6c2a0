"""GPU test of hstu_attn_fwd_noalloc, the forward entry point for callers
that cannot allocate device memory (a runtime that reserves all device
memory up front, or one for which cudaMalloc would synchronise or fail): its
plan scratch is a fixed array inside the library instead of a caller
workspace.

It is called through the C ABI and checked against hstu_attn_fwd on two
calls in a row with different batches, so that contents the shared scratch
keeps from the first call cannot leak into the second. This file is collected
last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl
from hstu_testutil import GpuBatch, check_o, np64

pytestmark = pytest.mark.gpu


def _noalloc(lib, gb, out, counts):
    shape = hb.make_shape(len(gb.lens), gb.total, gb.q.shape[1], gb.q.shape[2], gb.nfunc, gb.max_seqlen,
                          gb.alpha)
    vp = ctypes.c_void_p
    st = lib.hstu_attn_fwd_noalloc(vp(gb.q.data_ptr()), vp(gb.k.data_ptr()), vp(gb.v.data_ptr()),
                                   vp(out.data_ptr()), vp(gb.d_off.data_ptr()), vp(gb.d_func.data_ptr()),
                                   ctypes.byref(shape), vp(counts.data_ptr()),
                                   vp(torch.cuda.current_stream().cuda_stream))
    return st


def _batch(name, seed, lens=None):
    if lens is None:
        return GpuBatch.from_config(wl.CONFIGS[name], seed)
    cfg = wl.CONFIGS[name]
    lens = np.asarray(lens)
    func = wl.build_func(cfg, lens)
    T = int(lens.sum())
    g = torch.Generator().manual_seed(seed)
    q, k, v, do = (wl.randn_bf16((T, cfg.heads, cfg.dim), g) for _ in range(4))
    return GpuBatch(lens, func, q, k, v, do)


def test_noalloc_forward_matches_workspace_forward_twice():
    lib = hb.load()
    batches = [_batch("sla_b32_s1024", 0), _batch("onerank_b64", 1, lens=[700, 41, 1300, 513, 96])]
    for gb in batches:  # two calls in a row, different shapes and data
        out = torch.full_like(gb.q, float("nan"))
        counts = torch.full((gb.total,), -1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, gb, out, counts) == hb.HSTU_OK
        torch.cuda.synchronize()
        ref = gb.run(want_bwd=False)
        check_o(np64(out), np64(ref["o"]), "noalloc vs workspace forward")
        assert torch.equal(counts, ref["counts"])


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = hb.load()
    gb = _batch("tiny", 0)
    big = hb.make_shape(4096, gb.total, 2, 32, 5, 32768, 0.1)
    assert hb.workspace_size(big, hb.WS_FULL) > hb.NOALLOC_SCRATCH_BYTES
    vp = ctypes.c_void_p
    out = torch.empty_like(gb.q)
    st = lib.hstu_attn_fwd_noalloc(vp(gb.q.data_ptr()), vp(gb.k.data_ptr()), vp(gb.v.data_ptr()),
                                   vp(out.data_ptr()), vp(gb.d_off.data_ptr()), vp(gb.d_func.data_ptr()),
                                   ctypes.byref(big), None, None)
    assert st == 3  # HSTU_ERR_WORKSPACE, nothing enqueued
