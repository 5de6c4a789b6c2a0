"""Shape and type variants against the oracle: D_qk != D_v (the attention dim
and the linear dim of an HSTU layer), every pair of 32 / 64 / 128, and fp16
inputs as well as bf16, on ragged batches with partial tiles and several mask
families; the targets-only path on the same variants."""
import numpy as np
import pytest
import torch

import oracle.hstu_oracle as orc
from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl
from hstu_testutil import GpuBatch, check_grad, check_o, compare, np64

pytestmark = pytest.mark.gpu

DTYPES = {"bf16": torch.bfloat16, "f16": torch.float16}


def _batch(lens, H, dq, dv, dtype, mask, nfunc, seed, max_seqlen=None):
    T = int(np.sum(lens))
    g = torch.Generator().manual_seed(seed)
    q = wl.randn((T, H, dq), g, dtype=dtype)
    k = wl.randn((T, H, dq), g, dtype=dtype)
    v = wl.randn((T, H, dv), g, dtype=dtype)
    do = wl.randn((T, H, dv), g, dtype=dtype)
    cfg = wl.Config("v", len(lens), 0, 0, H, dq, mask, nfunc, k1=70, k2=20)
    func = wl.build_func(cfg, np.asarray(lens), nfunc)
    return GpuBatch(lens, func, q, k, v, do, max_seqlen=max_seqlen)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("dq,dv", [(128, 64), (64, 128), (32, 128), (128, 32), (32, 64), (64, 64)])
def test_mixed_head_dims(dtype, dq, dv):
    lens = [1, 130, 0, 300, 127, 257]
    gb = _batch(lens, 2, dq, dv, DTYPES[dtype], "sla", 5, seed=dq + dv, max_seqlen=320)
    out = gb.run()
    assert out["o"].shape[2] == dv and out["dq"].shape[2] == dq and out["dk"].shape[2] == dq
    assert out["dv"].shape[2] == dv and out["o"].dtype == DTYPES[dtype]
    compare(out, gb.oracle())


@pytest.mark.parametrize("mask,nfunc", [("tiny", 5), ("causal", 1), ("onerank", 7)])
def test_fp16_masks_at_d128(mask, nfunc):
    lens = [40, 300, 129, 513] if mask == "onerank" else [1, 130, 0, 300, 127, 257]
    gb = _batch(lens, 3, 128, 128, torch.float16, mask, nfunc, seed=5)
    compare(gb.run(), gb.oracle())


def test_fp16_sla_config_sampled():
    cfg = wl.CONFIGS["sla_b32_s1024"]
    lens = wl.lengths(cfg, 0)
    gb = _batch(list(lens), cfg.heads, 128, 128, torch.float16, "sla", 5, seed=0)
    out = gb.run()
    compare(out, gb.oracle([0, 17, 31]))


def test_fp16_and_bf16_on_the_same_values():
    """bf16 values are exact in fp16 here (|x| < 6.5e4, 8-bit mantissa), so
    both paths see the same inputs: both must match the oracle on them."""
    lens = [300, 64, 200]
    a = _batch(lens, 2, 128, 64, torch.bfloat16, "sla", 5, seed=9)
    b = GpuBatch(a.lens, a.func, *(t.to(torch.float16) for t in (a.q, a.k, a.v, a.do)))
    ra, rb = a.run(), b.run()
    assert torch.equal(ra["counts"], rb["counts"])
    ref = a.oracle()
    compare(ra, ref)
    compare(rb, ref)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("dq,dv", [(128, 64), (64, 128), (32, 32), (128, 128)])
def test_targets_only_variants(dtype, dq, dv):
    lens = np.array([700, 33, 260, 1])
    gb = _batch(list(lens), 2, dq, dv, DTYPES[dtype], "causal", 3, seed=7)
    B = len(lens)
    g = torch.Generator().manual_seed(11)
    q_c = wl.randn((B, 2, dq), g, dtype=DTYPES[dtype]).cuda()
    do_c = wl.randn((B, 2, dv), g, dtype=DTYPES[dtype]).cuda()
    rng = np.random.default_rng(dq * dv)
    func_c = rng.integers(-10, 720, size=(3, B)).astype(np.int32)
    d_fc = torch.tensor(func_c, device="cuda")
    shape = hb.make_shape(B, gb.total, 2, dq, 3, gb.max_seqlen, gb.alpha, dim_v=dv, dtype=hb.DTYPES[q_c.dtype])
    ws = hb.alloc_workspace(shape, hb.WS_TARGETS)
    o_c = hb.fwd_targets_only(q_c, gb.k, gb.v, gb.d_off, d_fc, gb.max_seqlen, gb.alpha, ws=ws)
    dq_c, dk, dvv = hb.bwd_targets_only(do_c, q_c, gb.k, gb.v, gb.d_off, d_fc, gb.max_seqlen, gb.alpha, ws=ws)
    assert hb.device_status(ws) == hb.HSTU_OK
    assert o_c.shape == (B, 2, dv) and dq_c.shape == (B, 2, dq)
    hk, hv = np64(gb.k), np64(gb.v)
    ref = orc.fwd_targets_only(np64(q_c), hk, hv, gb.offsets, func_c, 3, gb.max_seqlen, gb.alpha)
    check_o(np64(o_c), ref)
    rdq, rdk, rdv = orc.bwd_targets_only(np64(do_c), np64(q_c), hk, hv, gb.offsets, func_c, 3, gb.max_seqlen,
                                         gb.alpha)
    check_grad(np64(dq_c), rdq, "dq_c")
    check_grad(np64(dk), rdk, "dk")
    check_grad(np64(dvv), rdv, "dv")


def test_mixed_dims_backward_is_bitwise_repeatable():
    gb = _batch([300, 700, 129], 2, 128, 64, torch.float16, "onerank", 5, seed=3)
    a = gb.run()
    for _ in range(3):
        b = gb.run()
        for n in ("o", "dq", "dk", "dv"):
            assert torch.equal(a[n], b[n]), n
