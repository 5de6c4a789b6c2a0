#!/usr/bin/env python3
"""Benchmark: jagged HSTU masked attention fwd+bwd on one GB300 per rank.

A step is one pass of the whole hot path over one synthetic batch: the plan
(offset validation, tile classification, longest-first work lists), the
forward kernel and the backward kernel, all through the C ABI. The headline
workload is the DLRMv4 last-layer shape of MLCommons training PR #903
(layer-timing table): B=1024 sequences of 2663 +-50% ragged length (about
2.77 M tokens), H=4, D=128, causal with one candidate per sequence. Two
sub-measurements ride on the same JSON line:

  padding       the SLA mask of TorchEasyRec PR #670 at B=32, S=1024, H=4,
                D=128, NFUNC=5 (third interval padded empty) against NFUNC=3
                on the same batch, legs interleaved: the cost of the padding;
  targets_only  the same DLRM batch in targets-only mode (one candidate row
                per sequence against full-length K/V), HBM-bound.

Metric: useful TFLOP/s = visible (row, column) pairs x heads x (4 D forward +
10 D backward) / step time. Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --config onerank_b64|sla_b16_s2048|sla_b32_s1024 ...
  python bench.py --mode targets ...      (targets-only line on its own)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "HSTU masked attn fwd+bwd ms and useful TFLOP/s (% bf16 TC peak), 1xGB300"
UNIT = "TFLOP/s"
DEFAULT_CONFIG = "dlrm_b1024"
PADDING_CONFIG = "sla_b32_s1024"
L2_FLUSH_BYTES = 512 << 20

# DRAM bytes (read + write) of the backward kernel per token, by mask family,
# from one ncu capture of a smaller case of the same family (named in
# "captured_on"), with the hash of the kernel sources it was taken on. The
# backward reads q, k, v, dO and writes dq, dk, dv once, so its traffic grows
# in proportion to the tokens of a launch; it is reported only while the
# sources are unchanged.
NCU_TRAFFIC = {
    "causal": {"bytes_per_token": (811448576 + 500409344) / 172107,
               "captured_on": "hstu_bwd_kernel on dlrm_b1024@b64 (172,107 tokens, same length mix and mask), "
                              "dram__bytes_read.sum + dram__bytes_write.sum, scaled by tokens",
               "sources_sha": "db05f2b57fdff167"},
}


def kernel_sources_sha() -> str:
    """Hash of the code the backward kernel is compiled from (comments and
    blank space left out); the recorded ncu traffic of that kernel is only
    reported while it matches."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "jagged_hstu_attention_gb300", "csrc")
    for name in ("attn_bwd.cuh", "attn_bwd_bf16.cu", "common.cuh", "sm103_primitives.cuh"):
        with open(os.path.join(csrc, name)) as f:
            code = f.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(name.encode())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"bf16_tflops": float(p["bf16_tflops"]), "hbm_gbs": float(p["hbm_gbs"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"hstu_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            res = parse_clock_samples(f)
        os.unlink(self.path)
        return res


def parse_clock_samples(lines):
    """Median and maximum SM clock and the throttle reasons seen, from
    `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits`
    lines; None if no sample parses."""
    sm, mx, reasons = [], [], set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for n, val in zip(names, parts[5:9]):
            if val.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
            "reasons": sorted(reasons)}


# ---------------------------------------------------------------- GPU legs
class Leg:
    """One jagged batch resident on the GPU with preallocated outputs."""

    def __init__(self, cfg, seed, nfunc, device, shared=None, lens=None, max_seqlen=None):
        import torch
        from jagged_hstu_attention_gb300 import binding as hb
        from jagged_hstu_attention_gb300 import workloads as wl
        self.hb = hb
        if shared is None:
            gen_dev = "cuda" if cfg.name.startswith("dlrm") else "cpu"
            b = wl.make_batch(cfg, seed, device=gen_dev, nfunc=nfunc, lens=lens)
            self.lens, self.offsets, self.func = b.lens, b.offsets, b.func
            self.q, self.k, self.v, self.do = (t.to(device) for t in (b.q, b.k, b.v, b.do))
        else:  # same activations, another func width
            self.lens, self.offsets = shared.lens, shared.offsets
            self.func = wl.build_func(cfg, self.lens, nfunc)
            self.q, self.k, self.v, self.do = shared.q, shared.k, shared.v, shared.do
        self.cfg, self.nfunc = cfg, nfunc
        self.T = int(self.offsets[-1])
        self.N = int(self.lens.max()) if max_seqlen is None else int(max_seqlen)
        self.alpha = 1.0 / math.sqrt(cfg.dim)
        self.d_off = torch.tensor(self.offsets, dtype=torch.int32, device=device)
        self.d_func = torch.tensor(self.func, dtype=torch.int32, device=device)
        self.shape = hb.make_shape(len(self.lens), self.T, cfg.heads, cfg.dim, nfunc, self.N, self.alpha)
        self.ws = hb.alloc_workspace(self.shape, hb.WS_FULL, device)
        self.counts = torch.empty(self.T, dtype=torch.int32, device=device)
        self.o = torch.empty_like(self.q)
        self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        hb.plan(self.d_off, self.d_func, self.shape, self.ws, row_counts=self.counts)
        torch.cuda.synchronize()
        if hb.device_status(self.ws) != hb.HSTU_OK:
            raise RuntimeError("plan reported a device-side error")
        self.pairs = int(self.counts.sum().item())  # visible pairs per head

    def flops(self):
        H, D = self.cfg.heads, self.cfg.dim
        return self.pairs * H * 4 * D, self.pairs * H * 10 * D

    def step(self, ev):
        hb = self.hb
        ev[0].record()
        hb.plan(self.d_off, self.d_func, self.shape, self.ws)
        ev[1].record()
        hb.fwd(self.q, self.k, self.v, self.d_off, self.d_func, self.N, self.alpha, ws=self.ws,
               reuse_plan=True, out=self.o)
        ev[2].record()
        hb.bwd(self.do, self.q, self.k, self.v, self.d_off, self.d_func, self.N, self.alpha, ws=self.ws,
               reuse_plan=True, outs=(self.dq, self.dk, self.dv))
        ev[3].record()


LAUNCHES_PER_STEP = 3  # plan (classify + work lists) + forward + backward


def time_legs(legs, steps, warmup, flush):
    import torch
    for _ in range(warmup):
        for leg in legs:
            leg.step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
    torch.cuda.synchronize()
    rec = [[] for _ in legs]
    for i in range(steps):
        # Alternate the order of the legs so that neither always runs first.
        order = range(len(legs)) if i % 2 == 0 else reversed(range(len(legs)))
        for li in order:
            leg = legs[li]
            flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            leg.step(ev)
            rec[li].append(ev)
    torch.cuda.synchronize()
    out = []
    for evs in rec:
        plan = [e[0].elapsed_time(e[1]) for e in evs]
        fwd = [e[1].elapsed_time(e[2]) for e in evs]
        bwd = [e[2].elapsed_time(e[3]) for e in evs]
        stp = [e[0].elapsed_time(e[3]) for e in evs]
        out.append({"plan": plan, "fwd": fwd, "bwd": bwd, "step": stp})
    return out


def e2e_leg(leg, steps, warmup):
    """Same step through the C ABI from pinned HOST buffers: every step copies
    its inputs in and its outputs out, inside the timed region. The steps are
    pipelined over three streams (inputs of step i + 1 go in while step i
    computes and the outputs of step i - 1 come out), with two device buffer
    sets, the way a training loop feeds a device from host memory."""
    import torch
    hb = leg.hb
    pin = lambda t: t.cpu().pin_memory()
    h_in = [pin(t) for t in (leg.q, leg.k, leg.v, leg.do, leg.d_off, leg.d_func)]
    h_out = [[torch.empty(leg.q.shape, dtype=leg.q.dtype).pin_memory() for _ in range(4)] for _ in range(2)]
    d_in = [[torch.empty_like(t, device="cuda") for t in h_in] for _ in range(2)]
    d_out = [[torch.empty_like(leg.q) for _ in range(4)] for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def one(i):
        b = i % 2
        s_in.wait_event(ev_comp[b])  # step i - 2 has finished reading buffer set b
        with torch.cuda.stream(s_in):
            for d, h in zip(d_in[b], h_in):
                d.copy_(h, non_blocking=True)
        ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        s_comp.wait_event(ev_out[b])  # outputs of step i - 2 have left buffer set b
        q, k, v, do, off, func = d_in[b]
        hb.plan(off, func, leg.shape, leg.ws, stream=s_comp)
        hb.fwd(q, k, v, off, func, leg.N, leg.alpha, ws=leg.ws, reuse_plan=True, out=d_out[b][0],
               stream=s_comp)
        hb.bwd(do, q, k, v, off, func, leg.N, leg.alpha, ws=leg.ws, reuse_plan=True,
               outs=tuple(d_out[b][1:]), stream=s_comp)
        ev_comp[b].record(s_comp)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            for h, d in zip(h_out[b], d_out[b]):
                h.copy_(d, non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize()
    main = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    s_in.wait_event(e0)
    for i in range(warmup, warmup + steps):
        one(i)
    main.wait_stream(s_out)
    e1.record(main)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return ms, h2d, d2h


# ---------------------------------------------------------------- CPU oracle
def oracle_sample(cfg, seed, budget_s, min_seqs=1, max_seqs=None, order="longest"):
    """Times the fp64 oracle (as it stands) on whole sequences of the workload
    until the time budget is spent. Sequences are taken longest first
    (order="longest") or in a seeded random order ("random"). Returns
    (useful flops, seconds, sequences done, sequences in the batch, visible
    pairs per head done)."""
    import torch
    import oracle.hstu_oracle as orc
    from jagged_hstu_attention_gb300 import workloads as wl
    lens = wl.lengths(cfg, seed)
    N = int(lens.max())
    alpha = 1.0 / math.sqrt(cfg.dim)
    if order == "longest":
        seq_order = np.argsort(-lens, kind="stable")
    else:
        seq_order = np.random.default_rng(seed + 77).permutation(len(lens))
    g = torch.Generator().manual_seed(seed)
    flops = 0.0
    secs = 0.0
    done = 0
    pairs_done = 0
    limit = max_seqs if max_seqs is not None else len(lens)
    for b in seq_order[:limit]:
        L = int(lens[b])
        f = wl.func_rows(cfg, L)
        shape = (L, cfg.heads, cfg.dim)
        q, k, v, do = (wl.randn_bf16(shape, g).float().numpy().astype(np.float64) for _ in range(4))
        off = np.array([0, L])
        t0 = time.perf_counter()
        orc.fwd_dense(q, k, v, off, f, cfg.nfunc, N, alpha)
        orc.bwd_dense(do, q, k, v, off, f, cfg.nfunc, N, alpha)
        secs += time.perf_counter() - t0
        pairs = int(orc.visible_counts(off, f, cfg.nfunc).sum())
        pairs_done += pairs
        flops += pairs * cfg.heads * 14 * cfg.dim
        done += 1
        if done >= min_seqs and secs >= budget_s:
            break
    return flops, secs, done, len(lens), pairs_done


def cpu_model() -> str:
    """The host CPU's model name (x86) or part description (Arm), best effort."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model name"):
            for line in info.splitlines():
                if line.startswith(key):
                    return line.split(":", 1)[1].strip()
        parts = sorted({line.split(":", 1)[1].strip() for line in info.splitlines()
                        if line.startswith("CPU part")})
        if parts:
            return f"{platform.machine()} (CPU part {', '.join(parts)})"
    except OSError:
        pass
    return platform.machine()


def cpu_cores():
    """(threads the oracle's BLAS pool runs, cores the OS reports, cores this
    process may run on)."""
    blas = 0
    try:
        from threadpoolctl import threadpool_info
        blas = max((int(i.get("num_threads", 0)) for i in threadpool_info()), default=0)
    except Exception:
        pass
    try:
        affinity = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        affinity = os.cpu_count()
    return (blas or affinity), os.cpu_count(), affinity


def cpu_baseline_record(value, secs, seqs, n_batch, sample, extra=None):
    used, total, affinity = cpu_cores()
    rec = {"value": value, "unit": UNIT, "cores": used, "os_cpu_count": total, "affinity_cores": affinity,
           "cpu": cpu_model(), "kind": "oracle", "sample": sample}
    if extra:
        rec.update(extra)
    return rec


# ---------------------------------------------------------------- ranks
def job_lengths(cfg, seed, world):
    """Lengths of the job's batch: cfg.batch * world sequences from `seed`."""
    import dataclasses
    from jagged_hstu_attention_gb300 import workloads as wl
    return wl.lengths(dataclasses.replace(cfg, batch=cfg.batch * world), seed)


def job_costs(cfg, seed, world, device):
    """Visible (row, column) pairs of every sequence of the job's batch, from
    the plan's per-row counts (hstu_attn_plan on this GPU): the work each
    sequence brings, whatever its mask."""
    import torch
    from jagged_hstu_attention_gb300 import binding as hb
    from jagged_hstu_attention_gb300 import workloads as wl
    lens = job_lengths(cfg, seed, world)
    off = wl.offsets_from_lengths(lens)
    T = int(off[-1])
    func = wl.build_func(cfg, lens)
    d_off = torch.tensor(off, dtype=torch.int32, device=device)
    d_func = torch.tensor(func, dtype=torch.int32, device=device)
    shape = hb.make_shape(len(lens), T, cfg.heads, cfg.dim, cfg.nfunc, int(lens.max()))
    ws = hb.alloc_workspace(shape, hb.WS_FULL, device)
    counts = torch.empty(max(T, 1), dtype=torch.int32, device=device)
    hb.plan(d_off, d_func, shape, ws, row_counts=counts)
    if hb.device_status(ws) != hb.HSTU_OK:
        raise RuntimeError("plan reported a device-side error")
    c = torch.cumsum(counts[:T].to(torch.int64), 0).cpu().numpy()
    c = np.concatenate([[0], c])
    return c[off[1:]] - c[off[:-1]]


def rank_sequences(cfg, seed, world, rank, cost=None):
    """This rank's share of the job's batch: (indices into the job's batch,
    their lengths, the batch-wide max_seqlen).

    The job's batch is ``cfg.batch * world`` sequences drawn from ``seed``;
    hstu_attn_shard_sequences splits it by whole sequences with the given
    per-sequence cost (the bench passes each sequence's visible pairs, see
    job_costs), so the work per rank stays fixed as the number of ranks grows
    (weak scaling). N is the batch-wide maximum on every rank: the op's 1/N
    scale must not depend on the split."""
    from jagged_hstu_attention_gb300 import binding as hb
    lens = job_lengths(cfg, seed, world)
    if world == 1:
        return np.arange(len(lens)), lens, int(lens.max())
    if cost is None:
        raise ValueError("a split over ranks needs each sequence's cost")
    owner, _ = hb.shard_sequences(np.asarray(cost, dtype=np.int64), world)
    idx = np.nonzero(owner.numpy() == rank)[0]
    return idx, lens[idx], int(lens.max())


def reduce_over_ranks(ms, work, device, world):
    """(max over ranks of the step time, sum over ranks of the work)."""
    if world == 1:
        return ms, work
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    w = torch.tensor([work], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(w, op=dist.ReduceOp.SUM)
    return float(t.item()), float(w.item())


# ---------------------------------------------------------------- main
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measure_targets(k, v, lens, N, steps, warmup, flush, seed):
    """Targets-only fwd + bwd over a resident batch: one candidate row per
    sequence (its last row, causal: it sees the whole sequence) against
    full-length K/V. Returns the timings and the algorithmic bytes."""
    import torch
    from jagged_hstu_attention_gb300 import binding as hb
    from jagged_hstu_attention_gb300 import workloads as wl
    device = k.device
    off = wl.offsets_from_lengths(lens)
    T, B, H, D = int(off[-1]), len(lens), k.shape[1], k.shape[2]
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 1000)
    q_c = wl.randn_bf16((B, H, D), gen, device)
    do_c = wl.randn_bf16((B, H, D), gen, device)
    d_off = torch.tensor(off, dtype=torch.int32, device=device)
    fc = torch.tensor(wl.build_func_candidates(lens, 1), dtype=torch.int32, device=device)
    alpha = 1.0 / math.sqrt(D)
    shape = hb.make_shape(B, T, H, D, 1, N, alpha)
    ws = hb.alloc_workspace(shape, hb.WS_TARGETS, device)
    o_c, dq_c = torch.empty_like(q_c), torch.empty_like(q_c)
    dk, dv = torch.empty_like(k), torch.empty_like(v)

    def step(ev):
        ev[0].record()
        hb.fwd_targets_only(q_c, k, v, d_off, fc, N, alpha, ws=ws, out=o_c)
        ev[1].record()
        hb.bwd_targets_only(do_c, q_c, k, v, d_off, fc, N, alpha, ws=ws, outs=(dq_c, dk, dv))
        ev[2].record()

    for _ in range(warmup):
        step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    torch.cuda.synchronize()
    if hb.device_status(ws) != hb.HSTU_OK:
        raise RuntimeError("targets-only reported a device-side error")
    recs = []
    for _ in range(steps):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        step(ev)
        recs.append(ev)
    torch.cuda.synchronize()
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in recs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in recs)
    row = H * D * 2
    bytes_fwd = 2 * T * row + 2 * B * row   # read K, V, q_c; write o_c
    bytes_bwd = 4 * T * row + 3 * B * row   # read K, V, q_c, dO_c; write dK, dV, dq_c
    del dk, dv
    return {"fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "ms": fwd_ms + bwd_ms, "bytes": bytes_fwd + bytes_bwd,
            "T": T, "B": B, "H": H, "D": D, "launches": 4 * steps}


def measure_layer(leg, steps, warmup, flush, seed, d_model=512):
    """The last HSTU layer's input projection plus attention, full length
    against targets-only, fwd + bwd (MLCommons training PR #903, layer-timing
    table: 512-dim layer, 4 heads, qk and linear dim 128).

      full     project all T rows to U, V, Q, K (silu(x W_uvqk^T + b), 4 H D
               outputs), attention over every row (plan, forward, backward),
               the projection's backward;
      targets  project all rows to K, V, only the candidate rows to U, Q,
               targets-only attention, both projections' backward.

    The attention runs on the leg's resident q, k, v, dO (the projections'
    outputs have their shapes); the rest of the layer (normalisation, output
    projection) is the same in both arms and left out."""
    import torch
    from jagged_hstu_attention_gb300 import binding as hb
    from jagged_hstu_attention_gb300 import workloads as wl
    device = leg.q.device
    T, H, D = leg.T, leg.cfg.heads, leg.cfg.dim
    B = len(leg.lens)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 2000)
    x = wl.randn_bf16((T, d_model), gen, device)
    w_all = (wl.randn_bf16((4 * H * D, d_model), gen, device).float() / math.sqrt(d_model)).to(torch.bfloat16)
    b_all = torch.zeros(4 * H * D, dtype=torch.bfloat16, device=device)
    w_kv, w_uq = w_all[: 2 * H * D].contiguous(), w_all[2 * H * D:].contiguous()
    b_kv, b_uq = b_all[: 2 * H * D].contiguous(), b_all[2 * H * D:].contiguous()
    cand = torch.tensor(leg.offsets[1:] - 1, dtype=torch.int32, device=device)
    ws_f = hb.project_workspace(0, d_model, 4 * H * D, False, device)
    ws_fb = hb.project_workspace(T, d_model, 4 * H * D, True, device)
    dy_all = wl.randn_bf16((T, 4 * H * D), gen, device)
    ws_kv = hb.project_workspace(0, d_model, 2 * H * D, False, device)
    ws_kvb = hb.project_workspace(T, d_model, 2 * H * D, True, device)
    ws_uq = hb.project_workspace(B, d_model, 2 * H * D, False, device)
    ws_uqb = hb.project_workspace(B, d_model, 2 * H * D, True, device)
    dy_kv = dy_all[:, : 2 * H * D].contiguous()
    dy_uq = wl.randn_bf16((B, 2 * H * D), gen, device)
    q_c = leg.q.index_select(0, cand.long()).contiguous()
    do_c = leg.do.index_select(0, cand.long()).contiguous()
    fc = hb.build_func_candidates(leg.d_off, 1)
    tws = hb.alloc_workspace(hb.make_shape(B, T, H, D, 1, leg.N, leg.alpha), hb.WS_TARGETS, device)
    o_c, dq_c = torch.empty_like(q_c), torch.empty_like(q_c)

    def full(ev):
        ev[0].record()
        y, z = hb.project_rows(x, w_all, bias=b_all, ws=ws_f)
        leg.step([torch.cuda.Event(enable_timing=True) for _ in range(4)])
        hb.project_rows_bwd(dy_all, z, x, w_all, ws=ws_fb)
        ev[1].record()

    def targets(ev):
        ev[0].record()
        _, z_kv = hb.project_rows(x, w_kv, bias=b_kv, ws=ws_kv)
        _, z_uq = hb.project_rows(x, w_uq, rows=cand, bias=b_uq, ws=ws_uq)
        hb.fwd_targets_only(q_c, leg.k, leg.v, leg.d_off, fc, leg.N, leg.alpha, ws=tws, out=o_c)
        hb.bwd_targets_only(do_c, q_c, leg.k, leg.v, leg.d_off, fc, leg.N, leg.alpha, ws=tws,
                            outs=(dq_c, leg.dk, leg.dv))
        hb.project_rows_bwd(dy_kv, z_kv, x, w_kv, ws=ws_kvb)
        hb.project_rows_bwd(dy_uq, z_uq, x, w_uq, rows=cand, ws=ws_uqb)
        ev[1].record()

    res = {}
    for name, fn in (("full", full), ("targets_only", targets)):
        for _ in range(warmup):
            fn([torch.cuda.Event(enable_timing=True) for _ in range(2)])
        torch.cuda.synchronize()
        recs = []
        for _ in range(steps):
            flush.zero_()
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            fn(ev)
            recs.append(ev)
        torch.cuda.synchronize()
        res[name] = statistics.mean(e[0].elapsed_time(e[1]) for e in recs)
    if hb.device_status(tws) != hb.HSTU_OK:
        raise RuntimeError("targets-only reported a device-side error")
    gemm_flops = 2.0 * T * d_model * 4 * H * D
    return {"d_model": d_model, "full_ms": res["full"], "targets_only_ms": res["targets_only"],
            "speedup": res["full"] / res["targets_only"],
            "projection_gflop_fwd_full": gemm_flops / 1e9,
            "parts": "input projection (fwd+bwd, tcgen05 GEMMs) + attention (fwd+bwd)",
            "source": "MLCommons training PR #903 layer-timing table shape: 512-dim layer, 4 heads, dims 128"}


def run_targets(args, cfg, device, world, rank):
    """Targets-only mode as a line of its own: HBM-bound, reported as
    achieved bytes/s against the measured copy bandwidth."""
    import torch
    import torch.distributed as dist
    from jagged_hstu_attention_gb300 import workloads as wl
    seed = args.seed + rank
    cost = job_costs(cfg, args.seed, world, device) if world > 1 else None
    _, lens, N = rank_sequences(cfg, args.seed, world, rank, cost)
    T = int(np.sum(lens))
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    k = wl.randn_bf16((T, cfg.heads, cfg.dim), gen, device)
    v = wl.randn_bf16((T, cfg.heads, cfg.dim), gen, device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    sampler = ClockSampler(torch.cuda.current_device())
    if world > 1:
        dist.barrier()
    sampler.start()
    m = measure_targets(k, v, lens, N, args.steps, args.warmup, flush, seed)
    clocks = sampler.stop()
    ms, job_bytes = reduce_over_ranks(m["ms"], float(m["bytes"]), device, world)
    if rank != 0:
        return
    H, D = cfg.heads, cfg.dim
    useful = float(T) * H * 14 * D          # every key is visible to its candidate
    peaks = load_peaks()
    gbs = m["bytes"] / (m["ms"] * 1e-3) / 1e9
    line = {
        "metric": "HSTU targets-only fwd+bwd ms and achieved HBM GB/s (% of measured copy bandwidth)",
        "mode": "targets_only", "value": job_bytes / (ms * 1e-3) / 1e9, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": cfg.name + ":targets_only", "batch": len(lens), "global_batch": cfg.batch * world,
                   "total_tokens": T, "heads": H, "head_dim": D, "candidates_per_seq": 1,
                   "parallelism": f"dp{world}" if world > 1 else "single", "l2": "flushed between steps"},
        "breakdown_ms": {"fwd": m["fwd_ms"], "bwd": m["bwd_ms"]},
        "useful_tflops": useful / (m["ms"] * 1e-3) / 1e12,
        "gpu_launches": m["launches"],
        "roofline": {"kernel": "tgt_partial_kernel (fwd + bwd)", "bound": "hbm", "achieved": gbs,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                     "traffic": None, "peak_source": peaks["source"] + " copy bandwidth"},
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_reference(args, cfg):
    """The oracle as it stands on the host cores. Each step is a bounded
    sample of the workload: one whole sequence, taken in a seeded random
    order over the batch, all heads, fwd + bwd."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from jagged_hstu_attention_gb300 import workloads as wl
    lens = wl.lengths(cfg, args.seed)
    seq_order = np.random.default_rng(args.seed + 77).permutation(len(lens))
    times, flops_all = [], []
    for i in range(args.warmup + args.steps):
        one = wl.Config(cfg.name, 1, 0, 0, cfg.heads, cfg.dim, cfg.mask, cfg.nfunc, cfg.k1, cfg.k2)
        f, s, _, _, _ = oracle_sample_lengths(one, [int(lens[seq_order[i % len(lens)]])], int(lens.max()),
                                              args.seed + i)
        if i >= args.warmup:
            times.append(s)
            flops_all.append(f)
    value = sum(flops_all) / sum(times) / 1e12
    sample = (f"1 of {cfg.batch} sequences per step (seeded random order over the batch), all heads, "
              "fwd+bwd, dense fp64 numpy")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(cfg, lens, int(np.sum(lens)), 1),
            "cpu_baseline": cpu_baseline_record(value, sum(times), args.steps, cfg.batch, sample),
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def oracle_sample_lengths(cfg, lens, N, seed):
    """Times the oracle on sequences of the given lengths (max_seqlen N)."""
    import torch
    import oracle.hstu_oracle as orc
    from jagged_hstu_attention_gb300 import workloads as wl
    alpha = 1.0 / math.sqrt(cfg.dim)
    g = torch.Generator().manual_seed(seed)
    flops, secs, pairs_done = 0.0, 0.0, 0
    for L in lens:
        f = wl.func_rows(cfg, L)
        shape = (L, cfg.heads, cfg.dim)
        q, k, v, do = (wl.randn_bf16(shape, g).float().numpy().astype(np.float64) for _ in range(4))
        off = np.array([0, L])
        t0 = time.perf_counter()
        orc.fwd_dense(q, k, v, off, f, cfg.nfunc, N, alpha)
        orc.bwd_dense(do, q, k, v, off, f, cfg.nfunc, N, alpha)
        secs += time.perf_counter() - t0
        pairs = int(orc.visible_counts(off, f, cfg.nfunc).sum())
        pairs_done += pairs
        flops += pairs * cfg.heads * 14 * cfg.dim
    return flops, secs, len(lens), len(lens), pairs_done


def workload_config(cfg, lens, T, world):
    return {"workload": cfg.name, "batch": len(lens), "global_batch": cfg.batch * world,
            "seq_len": cfg.len_hi if cfg.len_lo == cfg.len_hi else f"U[{cfg.len_lo},{cfg.len_hi}]",
            "heads": cfg.heads, "head_dim": cfg.dim, "nfunc": cfg.nfunc, "mask": cfg.mask, "total_tokens": T,
            "parallelism": f"dp{world}" if world > 1 else "single", "l2": "flushed between steps"}


def bwd_traffic(cfg, T):
    """DRAM bytes per backward launch for this workload, scaled from the
    recorded capture by tokens (the backward's traffic is linear in tokens:
    q, k, v, dO read and dq, dk, dv written once), while the kernel sources
    are those the capture was taken on; else None."""
    rec = NCU_TRAFFIC.get(cfg.mask)
    if rec is None or rec["sources_sha"] != kernel_sources_sha():
        return None, None
    return rec["bytes_per_token"] * T, rec["captured_on"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (small profiling cases only)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="time the main workload only (no padding / targets-only / e2e sub-measurements)")
    ap.add_argument("--mode", default="full", choices=["full", "targets"],
                    help="full: plan + fwd + bwd over every row; targets: targets-only fwd + bwd")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    import dataclasses
    from jagged_hstu_attention_gb300 import workloads as wl
    cfg = wl.CONFIGS[args.config]
    if args.batch is not None:
        cfg = dataclasses.replace(cfg, batch=args.batch, name=f"{cfg.name}@b{args.batch}")
    if args.impl == "reference":
        run_reference(args, cfg)
        return

    import torch
    import torch.distributed as dist
    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from jagged_hstu_attention_gb300 import build_ext
    # One rank per node compiles (the ranks share the object files and the
    # library's path); the others wait for it.
    if local == 0:
        build_ext.build()
    if world > 1:
        dist.barrier(device_ids=[local])
    from jagged_hstu_attention_gb300 import binding as hb
    hb.load()
    if args.mode == "targets":
        run_targets(args, cfg, device, world, rank)
        if world > 1:
            dist.destroy_process_group()
        return

    # Each rank runs its share of a batch of cfg.batch * world sequences (whole
    # sequences, split by visible pairs); no data-path collective; weak
    # scaling. Activations are drawn from seed + rank.
    seed = args.seed + rank
    cost = job_costs(cfg, args.seed, world, device) if world > 1 else None
    _, lens, n_max = rank_sequences(cfg, args.seed, world, rank, cost)
    leg_main = Leg(cfg, seed, cfg.nfunc, device, lens=lens, max_seqlen=n_max)
    legs = [leg_main]
    padding_inline = cfg.mask == "sla" and cfg.nfunc == 5
    if padding_inline:
        legs.append(Leg(cfg, seed, 3, device, shared=leg_main))
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)

    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    res = time_legs(legs, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()

    r = res[0]
    ms_step = statistics.mean(r["step"])
    f_fwd, f_bwd = leg_main.flops()
    useful = f_fwd + f_bwd
    ms_max, job_useful = reduce_over_ranks(ms_step, useful, device, world)
    value = job_useful / (ms_max * 1e-3) / 1e12

    extras = {}
    if not args.no_extras:
        e2e_ms, h2d, d2h = e2e_leg(leg_main, max(3, args.steps // 2), 2)
        e2e_max, _ = reduce_over_ranks(e2e_ms, useful, device, world)
        extras["e2e"] = {"value": job_useful / (e2e_max * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
                         "d2h_bytes_per_step": d2h, "ms_per_step": e2e_max}
        torch.cuda.empty_cache()
        if rank == 0 and cfg.mask == "causal":
            extras["targets"] = measure_targets(leg_main.k, leg_main.v, leg_main.lens, leg_main.N, args.steps,
                                                args.warmup, flush, seed)
            extras["layer"] = measure_layer(leg_main, max(3, args.steps // 4), 2, flush, seed)
            torch.cuda.empty_cache()
        if rank == 0 and not padding_inline:
            pcfg = wl.CONFIGS[PADDING_CONFIG]
            p5 = Leg(pcfg, args.seed, 5, device)
            p3 = Leg(pcfg, args.seed, 3, device, shared=p5)
            extras["padding"] = (time_legs([p5, p3], max(args.steps, 20), args.warmup, flush), p5)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    peaks = load_peaks()
    ms_bwd = statistics.mean(r["bwd"])
    ms_fwd = statistics.mean(r["fwd"])
    achieved = f_bwd / (ms_bwd * 1e-3) / 1e12
    traffic, traffic_src = bwd_traffic(cfg, leg_main.T)
    launches = LAUNCHES_PER_STEP * args.steps * len(legs)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(cfg, lens, leg_main.T, world),
        "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
        "breakdown_ms": {k: statistics.mean(r[k]) for k in ("plan", "fwd", "bwd")},
        "step_ms_stats": {"mean": ms_step, "median": statistics.median(r["step"]), "min": min(r["step"]),
                          "max": max(r["step"])},
        "useful_gflop_per_step": useful / 1e9,
        "gpu_launches": launches,
        "roofline": {"kernel": "hstu_bwd_kernel", "bound": "tensor", "achieved": achieved,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                     "traffic_basis": traffic_src,
                     "algorithmic_bytes": 7 * leg_main.T * cfg.heads * cfg.dim * 2 + 4 * cfg.nfunc * leg_main.T,
                     "peak_source": peaks["source"] + " burst bf16",
                     "frac_of_sustained": achieved / peaks["bf16_tflops_sustained"],
                     "fwd": {"kernel": "hstu_fwd_kernel", "achieved": f_fwd / (ms_fwd * 1e-3) / 1e12,
                             "frac": f_fwd / (ms_fwd * 1e-3) / 1e12 / peaks["bf16_tflops"]}},
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if "e2e" in extras:
        line["e2e"] = extras["e2e"]
    if len(legs) > 1:
        line["padding"] = padding_record(res, legs[1], PADDING_CONFIG if args.config == PADDING_CONFIG else cfg.name)
    elif "padding" in extras:
        pres, p5 = extras["padding"]
        line["padding"] = padding_record(pres, p5, PADDING_CONFIG)
    if "targets" in extras:
        m = extras["targets"]
        gbs = m["bytes"] / (m["ms"] * 1e-3) / 1e9
        line["targets_only"] = {
            "workload": cfg.name + ":targets_only", "ms_per_step": m["ms"],
            "breakdown_ms": {"fwd": m["fwd_ms"], "bwd": m["bwd_ms"]}, "achieved_gbs": gbs,
            "hbm_frac": gbs / peaks["hbm_gbs"], "peak_gbs": peaks["hbm_gbs"],
            "speedup_vs_full_step": ms_step / m["ms"], "candidates_per_seq": 1,
            "algorithmic_bytes": m["bytes"], "gpu_launches": m["launches"]}
    if "layer" in extras:
        line["layer"] = extras["layer"]
    if not args.no_cpu_baseline:
        f, s, n, nb, pairs = oracle_sample(cfg, seed, args.cpu_budget,
                                           order="random" if cfg.batch > 64 else "longest")
        full_s = s * leg_main.pairs / max(pairs, 1)
        sample = (f"{n} of {nb} sequences ({'seeded random order' if cfg.batch > 64 else 'longest first'}), "
                  f"all heads, fwd+bwd, dense fp64 numpy, {s:.1f} s")
        extra = None
        if n < nb:
            extra = {"extrapolated_full_step_s": full_s,
                     "extrapolation": "sample time x (visible pairs of the batch / visible pairs of the sample)"}
        line["cpu_baseline"] = cpu_baseline_record(f / s / 1e12, s, n, nb, sample, extra)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def padding_record(res, leg, workload):
    r5, r3 = res[0], res[1]
    med5, med3 = statistics.median(r5["step"]), statistics.median(r3["step"])
    return {"workload": workload, "ms_per_step": {"nfunc5": statistics.mean(r5["step"]),
                                                  "nfunc3": statistics.mean(r3["step"])},
            "breakdown_ms": {"nfunc5": {k: statistics.mean(r5[k]) for k in ("plan", "fwd", "bwd")},
                             "nfunc3": {k: statistics.mean(r3[k]) for k in ("plan", "fwd", "bwd")}},
            "median_ms_per_step": {"nfunc5": med5, "nfunc3": med3},
            "padding_overhead_pct": 100.0 * (med5 - med3) / med3,
            "useful_tflops_nfunc5": sum(leg.flops()) / (med5 * 1e-3) / 1e12,
            "padding_overhead_basis": "medians over the timed steps; legs alternate order"}


if __name__ == "__main__":
    main()
