"""Device-side func builders (hstu_attn_build_func / _candidates): the func
they write equals the host builders' in workloads.py bit for bit, and
attention through a device-built func matches the oracle."""
import numpy as np
import pytest
import torch

from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl
from hstu_testutil import GpuBatch, compare

pytestmark = pytest.mark.gpu

LENS = [1, 130, 0, 300, 127, 257, 33, 32, 31, 2048]


def _device_func(cfg, lens, nfunc, **kw):
    off = torch.tensor(wl.offsets_from_lengths(np.array(lens)), dtype=torch.int32, device="cuda")
    T = int(np.sum(lens))
    return hb.build_func(cfg.mask, off, T, max(1, max(lens)), nfunc, **kw)


@pytest.mark.parametrize("nfunc", [1, 3, 5, 9])
def test_causal_func_is_bitwise_the_host_builders(nfunc):
    cfg = wl.Config("c", len(LENS), 0, 0, 1, 64, "causal", nfunc)
    got = _device_func(cfg, LENS, nfunc).cpu().numpy()
    assert np.array_equal(got, wl.build_func(cfg, np.array(LENS), nfunc))


@pytest.mark.parametrize("nfunc", [3, 5, 7, 9])
@pytest.mark.parametrize("k1,k2", [(256, 32), (70, 20), (0, 5), (5, 0), (4096, 1)])
def test_sla_func_is_bitwise_the_host_builders(nfunc, k1, k2):
    cfg = wl.Config("s", len(LENS), 0, 0, 1, 64, "sla", nfunc, k1=k1, k2=k2)
    got = _device_func(cfg, LENS, nfunc, k1=k1, k2=k2).cpu().numpy()
    assert np.array_equal(got, wl.build_func(cfg, np.array(LENS), nfunc))


@pytest.mark.parametrize("nfunc", [5, 7, 9])
def test_onerank_func_is_bitwise_the_host_builders(nfunc):
    # lengths at, below and above the 32 rows the groups take (8 x (1 + 3))
    cfg = wl.Config("o", len(LENS), 0, 0, 1, 64, "onerank", nfunc)
    got = _device_func(cfg, LENS, nfunc, groups=8, task_tokens=3).cpu().numpy()
    assert np.array_equal(got, wl.build_func(cfg, np.array(LENS), nfunc))


def test_full_size_configs_build_on_the_device():
    for name in ("sla_b32_s1024", "onerank_b64", "dlrm_b1024"):
        cfg = wl.CONFIGS[name]
        lens = wl.lengths(cfg, 0)
        kw = dict(k1=cfg.k1, k2=cfg.k2) if cfg.mask == "sla" else {}
        got = _device_func(cfg, list(lens), cfg.nfunc, **kw).cpu().numpy()
        assert np.array_equal(got, wl.build_func(cfg, lens)), name


def test_candidates_func_is_bitwise_the_host_builders():
    off = torch.tensor(wl.offsets_from_lengths(np.array(LENS)), dtype=torch.int32, device="cuda")
    for nfunc in (1, 3, 5):
        got = hb.build_func_candidates(off, nfunc).cpu().numpy()
        assert np.array_equal(got, wl.build_func_candidates(np.array(LENS), nfunc))


@pytest.mark.parametrize("mask", ["sla", "onerank"])
def test_attention_through_a_device_built_func_matches_the_oracle(mask):
    lens = np.array([300, 77, 513, 40])
    cfg = wl.Config("d", len(lens), 0, 0, 2, 128, mask, 5, k1=100, k2=24)
    T = int(lens.sum())
    g = torch.Generator().manual_seed(31)
    q, k, v, do = (wl.randn_bf16((T, 2, 128), g) for _ in range(4))
    host_func = wl.build_func(cfg, lens)
    gb = GpuBatch(lens, host_func, q, k, v, do)
    kw = dict(k1=100, k2=24) if mask == "sla" else dict(groups=8, task_tokens=3)
    gb.d_func = hb.build_func(mask, gb.d_off, T, gb.max_seqlen, 5, **kw)  # the kernels read this one
    compare(gb.run(), gb.oracle())
