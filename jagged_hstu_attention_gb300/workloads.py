"""Seeded synthetic workloads for jagged HSTU masked attention.

This module only draws inputs: sequence lengths, the jagged offsets, the
``func`` interval tensor of each mask family and N(0, 1) bf16 activations. It
holds none of the attention arithmetic, so both the CUDA path and the CPU
oracle can be fed from it without sharing any computation.

Mask families (func layout: ``(nfunc, total)`` int32, local column indices,
interval 0 = ``[0, func[0])``, interval t >= 1 = ``[func[2t-1], func[2t])``;
an interval whose end <= start is empty):

* ``tiny`` -- prefix ``[0, 8)`` plus the causal window ``[i-7, i+1)`` plus one
  padded empty interval (NFUNC=5). The prefix lets rows i < 7 see a few future
  columns, which exercises non-causal visibility.
* ``sla`` -- TorchEasyRec PR #670 (SLA mask): global prefix of K1 columns
  (clipped causally) plus a causal local window of K2 columns; with NFUNC=5
  the third interval is padded empty by repeating the window end, as that
  page describes for ``build_sla_func_tensor``.
* ``onerank`` -- TorchEasyRec PR #670 (OneRank, three intervals: prefix +
  candidate + task token). The page does not fix K (task tokens) or C
  (candidates); these workloads take C=8 groups of K+1=4 tokens at the end
  of each sequence and give history rows a candidate and a task token too, so
  that every row carries three non-empty intervals.
* ``causal`` -- MLCommons training PR #903 (DLRMv4 last layer): plain causal
  ``[0, i+1)`` with NFUNC=1; one candidate per sequence, its last row.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

BLOCK = 128


@dataclasses.dataclass(frozen=True)
class Config:
    name: str
    batch: int
    len_lo: int
    len_hi: int
    heads: int
    dim: int
    mask: str
    nfunc: int
    k1: int = 256
    k2: int = 32


CONFIGS = {
    "tiny": Config("tiny", 4, 16, 64, 2, 32, "tiny", 5),
    "sla_b32_s1024": Config("sla_b32_s1024", 32, 1024, 1024, 4, 128, "sla", 5),
    "sla_b16_s2048": Config("sla_b16_s2048", 16, 2048, 2048, 8, 128, "sla", 5),
    "onerank_b64": Config("onerank_b64", 64, 512, 2048, 4, 128, "onerank", 5),
    "dlrm_b1024": Config("dlrm_b1024", 1024, 1332, 3994, 4, 128, "causal", 1),
}


def lengths(cfg: Config, seed: int = 0) -> np.ndarray:
    """Sequence lengths, uniform integers in [len_lo, len_hi]."""
    if cfg.len_lo == cfg.len_hi:
        return np.full(cfg.batch, cfg.len_lo, dtype=np.int64)
    rng = np.random.default_rng(seed)
    return rng.integers(cfg.len_lo, cfg.len_hi + 1, size=cfg.batch).astype(np.int64)


def offsets_from_lengths(lens: np.ndarray) -> np.ndarray:
    off = np.zeros(len(lens) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lens)
    return off


def _rows_tiny(L: int, nfunc: int) -> np.ndarray:
    i = np.arange(L, dtype=np.int64)
    f = np.empty((nfunc, L), dtype=np.int64)
    f[0] = min(8, L)
    f[1] = np.maximum(0, i - 7)
    f[2] = i + 1
    for t in range(3, nfunc):
        f[t] = i + 1  # padded empty intervals: [i+1, i+1)
    return f


def _rows_sla(L: int, nfunc: int, k1: int, k2: int) -> np.ndarray:
    i = np.arange(L, dtype=np.int64)
    f = np.empty((nfunc, L), dtype=np.int64)
    f[0] = np.minimum(k1, i + 1)
    f[1] = np.maximum(0, i - (k2 - 1))
    f[2] = i + 1
    for t in range(3, nfunc):
        f[t] = i + 1  # pad by repeating the window end: max <= min, skipped
    return f


def _rows_onerank(L: int, nfunc: int, groups: int = 8, task_tokens: int = 3) -> np.ndarray:
    assert nfunc >= 5
    gsize = task_tokens + 1
    lp = L - groups * gsize
    if lp <= 0:  # too short for the group layout: causal rows
        return _rows_causal(L, nfunc)
    f = np.empty((nfunc, L), dtype=np.int64)
    for r in range(L):
        if r < lp:
            g = r % groups
            e = lp + g * gsize
            t = e + 1 + (r % task_tokens)
            row = [r + 1, e, e + 1, t, t + 1]
        else:
            g = (r - lp) // gsize
            e = lp + g * gsize
            if r == e:
                row = [lp, e, e + 1, e, e + 1]
            else:
                row = [lp, e, e + 1, r, r + 1]
        f[:5, r] = row
    for t in range(5, nfunc):
        f[t] = f[4]
    return f


def _rows_causal(L: int, nfunc: int) -> np.ndarray:
    i = np.arange(L, dtype=np.int64)
    f = np.empty((nfunc, L), dtype=np.int64)
    for t in range(nfunc):
        f[t] = i + 1
    return f


def func_rows(cfg: Config, L: int, nfunc: Optional[int] = None) -> np.ndarray:
    nfunc = cfg.nfunc if nfunc is None else nfunc
    if cfg.mask == "tiny":
        return _rows_tiny(L, nfunc)
    if cfg.mask == "sla":
        return _rows_sla(L, nfunc, cfg.k1, cfg.k2)
    if cfg.mask == "onerank":
        return _rows_onerank(L, nfunc)
    if cfg.mask == "causal":
        return _rows_causal(L, nfunc)
    raise ValueError(cfg.mask)


def build_func(cfg: Config, lens: np.ndarray, nfunc: Optional[int] = None) -> np.ndarray:
    """(nfunc, total) int32 func tensor for the whole jagged batch."""
    nfunc = cfg.nfunc if nfunc is None else nfunc
    parts = [func_rows(cfg, int(L), nfunc) for L in lens]
    return np.concatenate(parts, axis=1).astype(np.int32)


def build_func_candidates(lens: np.ndarray, nfunc: int = 1) -> np.ndarray:
    """(nfunc, B) int32 func of each sequence's candidate row (its last row,
    causal: it sees [0, L_b))."""
    f = np.empty((nfunc, len(lens)), dtype=np.int64)
    for t in range(nfunc):
        f[t] = lens
    return f.astype(np.int32)


def randn_bf16(shape, gen: torch.Generator, device="cpu") -> torch.Tensor:
    """N(0, 1) drawn in fp32, rounded to bf16."""
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(torch.bfloat16)


def randn(shape, gen: torch.Generator, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """N(0, 1) drawn in fp32, rounded to ``dtype`` (bf16 or fp16)."""
    return torch.randn(shape, generator=gen, dtype=torch.float32, device=device).to(dtype)


@dataclasses.dataclass
class Batch:
    cfg: Config
    lens: np.ndarray
    offsets: np.ndarray  # (B+1,) int64
    func: np.ndarray  # (nfunc, T) int32
    q: torch.Tensor  # (T, H, D) bf16
    k: torch.Tensor
    v: torch.Tensor
    do: torch.Tensor

    @property
    def total(self) -> int:
        return int(self.offsets[-1])

    @property
    def max_seqlen(self) -> int:
        return int(self.lens.max())


def make_batch(cfg: Config, seed: int = 0, device="cpu", nfunc: Optional[int] = None,
               with_grad_out: bool = True, lens: Optional[np.ndarray] = None) -> Batch:
    """A jagged batch of the workload; ``lens`` (optional) replaces the drawn
    lengths, e.g. with one rank's share of a larger batch."""
    lens = lengths(cfg, seed) if lens is None else np.asarray(lens, dtype=np.int64)
    off = offsets_from_lengths(lens)
    func = build_func(cfg, lens, nfunc)
    T = int(off[-1])
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (T, cfg.heads, cfg.dim)
    q = randn_bf16(shape, gen, device)
    k = randn_bf16(shape, gen, device)
    v = randn_bf16(shape, gen, device)
    do = randn_bf16(shape, gen, device) if with_grad_out else None
    return Batch(cfg, lens, off, func, q, k, v, do)
