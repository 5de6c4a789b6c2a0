"""Host-side logic of bench.py that needs no GPU: clock-sample parsing, the
peak table and its fallback, the kernel-source hash that guards recorded
ncu traffic, and the split of a job's batch over ranks."""
import json
import os
import shutil

import numpy as np
import pytest

import bench
import oracle.hstu_oracle as orc
from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import build_ext
from jagged_hstu_attention_gb300 import workloads as wl


def test_clock_samples_median_max_and_reasons():
    lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    r = bench.parse_clock_samples(lines)
    assert r == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    hot = ["0, 1500, 2070, 1400, 0x60, Active, Active, Not Active, Not Active"]
    assert bench.parse_clock_samples(hot)["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.parse_clock_samples([]) is None


def test_peaks_measured_then_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.load_peaks()
    assert fb["source"] == "fallback" and fb["bf16_tflops"] == 1900.0 and fb["hbm_gbs"] == 6800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1904.1, "hbm_gbs": 6783.5}))
    m = bench.load_peaks()
    assert m["source"] == "measured" and m["bf16_tflops"] == 1904.1 and m["hbm_gbs"] == 6783.5
    assert m["bf16_tflops_sustained"] == 1904.1  # absent: the burst figure


def _copy_sources(dst):
    src = os.path.join(bench.ROOT, "jagged_hstu_attention_gb300", "csrc")
    out = dst / "jagged_hstu_attention_gb300" / "csrc"
    out.mkdir(parents=True)
    for name in ("attn_bwd.cuh", "attn_bwd_bf16.cu", "common.cuh", "sm103_primitives.cuh"):
        shutil.copy(os.path.join(src, name), out / name)
    return out


def test_kernel_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    out = _copy_sources(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_sources_sha()
    p = out / "attn_bwd.cuh"
    text = p.read_text()
    p.write_text("// a new comment line\n" + text.replace("\n", "\n\n", 3) + "\n/* block\n comment */\n")
    assert bench.kernel_sources_sha() == base
    assert "kDpSlots = 1" in text
    p.write_text(text.replace("kDpSlots = 1", "kDpSlots = 2", 1))
    assert bench.kernel_sources_sha() != base


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return hb.load()


def _oracle_costs(cfg, lens):
    """Visible pairs of every sequence, from the oracle's row counts (the
    causal mask's counts are i + 1, pinned in the oracle tests, so a causal
    sequence brings L (L + 1) / 2)."""
    if cfg.mask == "causal":
        return lens * (lens + 1) // 2
    out = []
    for L in lens:
        f = wl.func_rows(cfg, int(L))
        out.append(int(orc.visible_counts(np.array([0, int(L)]), f, cfg.nfunc).sum()))
    return np.array(out, dtype=np.int64)


@pytest.mark.parametrize("name", ["sla_b32_s1024", "dlrm_b1024", "onerank_b64"])
@pytest.mark.parametrize("world", [1, 2, 4])
def test_rank_shares_partition_the_job_batch(lib, name, world):
    cfg = wl.CONFIGS[name]
    job = bench.job_lengths(cfg, 0, world)
    cost = _oracle_costs(cfg, job)
    shares = [bench.rank_sequences(cfg, 0, world, r, cost) for r in range(world)]
    idx = np.concatenate([s[0] for s in shares])
    assert sorted(idx.tolist()) == list(range(cfg.batch * world))
    n_max = {s[2] for s in shares}
    assert len(n_max) == 1  # every rank uses the batch-wide N
    assert np.array_equal(job, wl.lengths(wl.Config(cfg.name, cfg.batch * world, cfg.len_lo, cfg.len_hi,
                                                    cfg.heads, cfg.dim, cfg.mask, cfg.nfunc), 0))
    assert n_max.pop() == int(job.max())
    for ids, lens, _ in shares:
        assert np.array_equal(job[ids], lens)
    # weak scaling: per-rank work (visible pairs) stays near one rank's batch
    loads = [int(cost[ids].sum()) for ids, _, _ in shares]
    assert max(loads) <= sum(loads) / world + int(cost.max())
    if world == 1:
        assert np.array_equal(shares[0][1], wl.lengths(cfg, 0))


def test_split_over_ranks_needs_costs(lib):
    with pytest.raises(ValueError):
        bench.rank_sequences(wl.CONFIGS["tiny"], 0, 2, 0)
