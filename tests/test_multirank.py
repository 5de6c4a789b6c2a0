"""The data-parallel path on CPU: two gloo ranks, no GPU.

The op shards by whole sequences with no exchange between ranks. These tests
check the split itself (a partition, deterministic, within Graham's bound of
the optimal makespan, checked against brute force on small batches), that
the ranks' results put back together are the unsplit batch's results
exactly (oracle on each rank's share, with the batch-wide N), and the
max-time / sum-work reduction the benchmark reports.
"""
import itertools
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle.hstu_oracle as orc
from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import build_ext
from jagged_hstu_attention_gb300 import workloads as wl

WORLD = 2
CFG = wl.Config("shard_test", 5, 8, 90, 2, 16, "tiny", 5)
SEED = 3


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_ext.build()
    return hb.load()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _optimal_makespan(cost, world):
    best = None
    for assign in itertools.product(range(world), repeat=len(cost)):
        load = [0] * world
        for c, r in zip(cost, assign):
            load[r] += c
        m = max(load)
        best = m if best is None else min(best, m)
    return best


def test_shard_is_a_partition_with_the_reported_loads():
    rng = np.random.default_rng(0)
    cost = rng.integers(0, 1000, size=37)
    owner, load = hb.shard_sequences(cost, 4)
    owner = owner.numpy()
    assert owner.min() >= 0 and owner.max() < 4
    for r in range(4):
        assert int(load[r]) == int(cost[owner == r].sum())
    again, _ = hb.shard_sequences(cost, 4)
    assert np.array_equal(again.numpy(), owner)


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("seed", range(6))
def test_shard_within_graham_bound_of_brute_force_optimum(world, seed):
    rng = np.random.default_rng(100 + seed)
    cost = [int(c) for c in rng.integers(1, 50, size=8)]
    _, load = hb.shard_sequences(cost, world)
    opt = _optimal_makespan(cost, world)
    assert int(load.max()) * 3 * world <= (4 * world - 1) * opt


def test_shard_follows_longest_first_greedy_on_a_worked_case():
    # 7, 6, 5 go to ranks 0, 1, 2; then 4 joins the lightest (rank 2, 5),
    # 3 joins rank 1 (6), 2 joins rank 0 (7): loads 9, 9, 9.
    owner, load = hb.shard_sequences([2, 7, 3, 6, 4, 5], 3)
    assert owner.tolist() == [0, 0, 1, 1, 2, 2]
    assert load.tolist() == [9, 9, 9]


def test_shard_edge_cases_and_errors():
    owner, load = hb.shard_sequences([], 3)
    assert owner.numel() == 0 and load.tolist() == [0, 0, 0]
    owner, load = hb.shard_sequences([5, 5], 4)
    assert owner.tolist() == [0, 1] and load.tolist() == [5, 5, 0, 0]
    owner, _ = hb.shard_sequences([0, 0, 0], 2)  # loads stay equal: the lower rank takes each
    assert owner.tolist() == [0, 0, 0]
    for cost, world in (([1, -1], 2), ([1], 0), ([2 ** 62, 2 ** 62], 2)):
        with pytest.raises(hb.HstuError):
            hb.shard_sequences(cost, world)


def _rank_main(rank, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        hb.load()
        job = bench.job_lengths(CFG, SEED, WORLD)
        jcfg = wl.Config(CFG.name, 1, 0, 0, CFG.heads, CFG.dim, CFG.mask, CFG.nfunc)
        cost = [int(orc.visible_counts(np.array([0, int(L)]), wl.func_rows(jcfg, int(L)), CFG.nfunc).sum())
                for L in job]
        idx, lens, n_max = bench.rank_sequences(CFG, SEED, WORLD, rank, cost)
        # The job's batch, built the same way on every rank; this rank keeps
        # only its own sequences.
        gcfg = wl.Config(CFG.name, CFG.batch * WORLD, CFG.len_lo, CFG.len_hi, CFG.heads, CFG.dim,
                         CFG.mask, CFG.nfunc)
        full = wl.make_batch(gcfg, SEED)
        g_off = full.offsets
        rows = np.concatenate([np.arange(g_off[b], g_off[b + 1]) for b in idx])
        off = wl.offsets_from_lengths(lens)
        f64 = lambda t: t.float().numpy().astype(np.float64)[rows]
        q, k, v, do = (f64(t) for t in (full.q, full.k, full.v, full.do))
        func = full.func[:, rows]
        alpha = 1.0 / np.sqrt(CFG.dim)
        o = orc.fwd_dense(q, k, v, off, func, CFG.nfunc, n_max, alpha)
        dq, dk, dv = orc.bwd_dense(do, q, k, v, off, func, CFG.nfunc, n_max, alpha)
        shares = [None] * WORLD
        dist.all_gather_object(shares, (idx, lens, n_max, rows, o, dq, dk, dv))
        ms, work = bench.reduce_over_ranks(1.5 + rank, 10.0 * (rank + 1), torch.device("cpu"), WORLD)
        if rank == 0:
            np.save(os.path.join(out_dir, "reduce.npy"), np.array([ms, work]))
            T = int(g_off[-1])
            shape = (T, CFG.heads, CFG.dim)
            got = {n: np.full(shape, np.nan) for n in ("o", "dq", "dk", "dv")}
            seen = []
            for s_idx, s_lens, s_n, s_rows, *outs in shares:
                assert s_n == int(full.lens.max())
                assert np.array_equal(full.lens[s_idx], s_lens)
                seen.extend(int(b) for b in s_idx)
                for n, a in zip(("o", "dq", "dk", "dv"), outs):
                    got[n][s_rows] = a
            assert sorted(seen) == list(range(gcfg.batch))
            ref = {"o": orc.fwd_dense(f64_all(full.q), f64_all(full.k), f64_all(full.v), g_off, full.func,
                                      CFG.nfunc, int(full.lens.max()), alpha)}
            ref["dq"], ref["dk"], ref["dv"] = orc.bwd_dense(
                f64_all(full.do), f64_all(full.q), f64_all(full.k), f64_all(full.v), g_off, full.func,
                CFG.nfunc, int(full.lens.max()), alpha)
            for n in got:
                np.testing.assert_array_equal(got[n], ref[n], err_msg=n)
            with open(os.path.join(out_dir, "ok"), "w") as f:
                f.write("ok")
    finally:
        dist.destroy_process_group()


def f64_all(t):
    return t.float().numpy().astype(np.float64)


def test_two_ranks_reassemble_the_unsplit_batch_exactly(tmp_path):
    mp.spawn(_rank_main, args=(_free_port(), str(tmp_path)), nprocs=WORLD, join=True)
    assert (tmp_path / "ok").exists()
    ms, work = np.load(tmp_path / "reduce.npy")
    assert ms == 2.5 and work == 30.0
