"""Helpers shared by the GPU parity tests: run the CUDA path through the
binding, slice sequences out of a jagged batch, compare against the oracle."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle.hstu_oracle as orc
from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl

# Tolerances of the parity contract: O max-abs and relative L2, gradients
# relative L2 (bf16 inputs, fp32 accumulation, bf16 P and dS operands).
O_MAX_ABS = 2e-2
O_REL_L2 = 5e-3
GRAD_REL_L2 = 1e-2


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / den) if den > 0 else float(np.linalg.norm(got))


# Achieved errors of every comparison in the session, so that the headroom
# against the tolerances can be read after a run (tests/conftest.py writes
# them to the file named by HSTU_PARITY_LOG, if set).
MARGINS = []
CURRENT_TEST = {"name": ""}


def _record(what, max_abs, rl, tol_abs, tol_rel):
    MARGINS.append({"test": CURRENT_TEST["name"], "what": what, "max_abs": max_abs, "rel_l2": rl,
                    "tol_max_abs": tol_abs, "tol_rel_l2": tol_rel})


def check_o(got, ref, what="O"):
    err = float(np.max(np.abs(np.asarray(got, np.float64) - ref))) if ref.size else 0.0
    rl = rel_l2(got, ref)
    _record(what, err, rl, O_MAX_ABS, O_REL_L2)
    assert err <= O_MAX_ABS and rl <= O_REL_L2, f"{what}: max-abs {err:.3e}, rel-L2 {rl:.3e}"
    return err, rl


def check_grad(got, ref, what):
    rl = rel_l2(got, ref)
    err = float(np.max(np.abs(np.asarray(got, np.float64) - ref))) if np.asarray(ref).size else 0.0
    _record(what, err, rl, None, GRAD_REL_L2)
    assert rl <= GRAD_REL_L2, f"{what}: rel-L2 {rl:.3e}"
    return rl


class GpuBatch:
    """A jagged batch resident on the GPU plus the host copies the oracle needs."""

    def __init__(self, lens, func, q, k, v, do, max_seqlen=None, alpha=None):
        self.lens = np.asarray(lens, dtype=np.int64)
        self.offsets = wl.offsets_from_lengths(self.lens)
        self.func = np.ascontiguousarray(func, dtype=np.int32)
        self.nfunc = self.func.shape[0]
        self.q, self.k, self.v, self.do = (t.cuda() for t in (q, k, v, do))
        self.max_seqlen = int(max_seqlen if max_seqlen is not None else max(1, int(self.lens.max())))
        self.alpha = float(alpha if alpha is not None else 1.0 / math.sqrt(q.shape[2]))
        self.d_off = torch.tensor(self.offsets, dtype=torch.int32, device="cuda")
        self.d_func = torch.tensor(self.func, dtype=torch.int32, device="cuda")

    @classmethod
    def from_config(cls, cfg, seed=0, nfunc=None, device="cpu"):
        b = wl.make_batch(cfg, seed, device=device, nfunc=nfunc)
        return cls(b.lens, b.func, b.q, b.k, b.v, b.do)

    @property
    def total(self):
        return int(self.offsets[-1])

    def run(self, want_bwd=True):
        T = self.total
        counts = torch.full((max(T, 1),), -1, dtype=torch.int32, device="cuda")
        shape = hb.make_shape(len(self.lens), T, self.q.shape[1], self.q.shape[2], self.nfunc,
                              self.max_seqlen, self.alpha, dim_v=self.v.shape[2], dtype=hb.DTYPES[self.q.dtype])
        ws = hb.alloc_workspace(shape, hb.WS_FULL)
        o = hb.fwd(self.q, self.k, self.v, self.d_off, self.d_func, self.max_seqlen, self.alpha, ws=ws,
                   row_counts=counts)
        out = {"o": o, "counts": counts[:T]}
        if want_bwd:
            dq, dk, dv = hb.bwd(self.do, self.q, self.k, self.v, self.d_off, self.d_func, self.max_seqlen,
                                self.alpha, ws=ws, reuse_plan=True)
            out.update(dq=dq, dk=dk, dv=dv)
        torch.cuda.synchronize()
        assert hb.device_status(ws) == hb.HSTU_OK
        return out

    def sub(self, seqs):
        """Host fp64 inputs and func of the given sequences (as their own batch)."""
        seqs = list(seqs)
        rows = np.concatenate([np.arange(self.offsets[b], self.offsets[b + 1]) for b in seqs]) \
            if seqs else np.zeros(0, dtype=np.int64)
        idx = torch.as_tensor(rows, device="cuda", dtype=torch.long)
        sub_off = wl.offsets_from_lengths(self.lens[seqs])
        host = [np64(t.index_select(0, idx)) for t in (self.q, self.k, self.v, self.do)]
        return rows, sub_off, self.func[:, rows], host

    def oracle(self, seqs=None, want_bwd=True):
        seqs = range(len(self.lens)) if seqs is None else seqs
        rows, sub_off, sub_func, (q, k, v, do) = self.sub(seqs)
        ref = {"rows": rows,
               "o": orc.fwd_dense(q, k, v, sub_off, sub_func, self.nfunc, self.max_seqlen, self.alpha),
               "counts": orc.visible_counts(sub_off, sub_func, self.nfunc)}
        if want_bwd:
            ref["dq"], ref["dk"], ref["dv"] = orc.bwd_dense(do, q, k, v, sub_off, sub_func, self.nfunc,
                                                            self.max_seqlen, self.alpha)
        return ref


def compare(gpu, ref, want_bwd=True):
    rows = torch.as_tensor(ref["rows"], device="cuda", dtype=torch.long)
    take = lambda t: np64(t.index_select(0, rows))
    counts = gpu["counts"].index_select(0, rows).cpu().numpy()
    assert np.array_equal(counts, ref["counts"]), "visible counts differ"
    res = {"o": check_o(take(gpu["o"]), ref["o"])}
    if want_bwd:
        for n in ("dq", "dk", "dv"):
            res[n] = check_grad(take(gpu[n]), ref[n], n)
    return res


def sample_seqs(lens, n, seed=0):
    """Seeded sample of sequence indices, always holding the longest and the
    shortest sequence."""
    lens = np.asarray(lens)
    pick = {int(np.argmax(lens)), int(np.argmin(lens))}
    rng = np.random.default_rng(seed + 1234)
    while len(pick) < min(n, len(lens)):
        pick.add(int(rng.integers(0, len(lens))))
    return sorted(pick)
