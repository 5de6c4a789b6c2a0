"""Thin Python binding of the C ABI in ``include/hstu_attn.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library. Tensors are torch CUDA tensors (torch supplies device memory and the
current stream); the library is loaded with ctypes from this directory and the
binding raises if it is missing -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhstu_attn.so")
# The same entry points compiled with device-side index checks (see
# hstu_attn.h); select_library() switches the wrappers below to it.
CHECKED_LIB_PATH = os.path.join(_HERE, "libhstu_attn_checked.so")

HSTU_OK = 0
STATUS_NAMES = {
    0: "HSTU_OK", 1: "HSTU_ERR_INVALID_ARG", 2: "HSTU_ERR_UNSUPPORTED", 3: "HSTU_ERR_WORKSPACE",
    4: "HSTU_ERR_CUDA", 5: "HSTU_ERR_DEVICE_INPUT", 6: "HSTU_ERR_TIMEOUT", 7: "HSTU_ERR_DEVICE_CHECK",
}
WS_FULL = 0
WS_TARGETS = 1
FLAG_REUSE_PLAN = 1

EXPORTED = (
    "hstu_attn_nfunc_supported", "hstu_attn_workspace_size", "hstu_attn_plan", "hstu_attn_fwd",
    "hstu_attn_bwd", "hstu_attn_fwd_targets_only", "hstu_attn_bwd_targets_only",
    "hstu_attn_get_device_status", "hstu_status_string", "hstu_attn_fwd_noalloc",
    "hstu_attn_shard_sequences", "hstu_attn_test_wait_timeout", "hstu_attn_build_func",
    "hstu_attn_build_func_candidates", "hstu_attn_targets_workspace_size", "hstu_attn_fwd_targets",
    "hstu_attn_bwd_targets", "hstu_attn_project_workspace_size", "hstu_attn_project_rows",
    "hstu_attn_project_rows_bwd", "hstu_attn_test_set_handoff_limit",
)
FUNC_CAUSAL, FUNC_SLA, FUNC_ONERANK = 0, 1, 2
NOALLOC_SCRATCH_BYTES = 8 << 20


class HstuError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class FuncSpec(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32),
        ("k1", ctypes.c_int32),
        ("k2", ctypes.c_int32),
        ("groups", ctypes.c_int32),
        ("task_tokens", ctypes.c_int32),
    ]


class Shape(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("total", ctypes.c_int64),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("nfunc", ctypes.c_int32),
        ("max_seqlen", ctypes.c_int32),
        ("alpha", ctypes.c_float),
        ("head_dim_v", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
    ]


_libs = {}
_active = LIB_PATH


def select_library(path: str) -> str:
    """Makes the wrappers of this module call the library at ``path`` (the
    release or the checked build); returns the previously selected path."""
    global _active
    prev, _active = _active, path
    return prev


def load(path: str = None) -> ctypes.CDLL:
    """Loads the selected library (once per path). Raises if it has not been
    built."""
    path = _active if path is None else path
    if path in _libs:
        return _libs[path]
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library {path} is missing: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    vp, i32, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
    sp = ctypes.POINTER(Shape)
    sig = {
        "hstu_attn_nfunc_supported": (ctypes.c_int, [i32]),
        "hstu_attn_workspace_size": (sz, [sp, i32]),
        "hstu_attn_plan": (ctypes.c_int, [vp, vp, sp, vp, vp, sz, vp]),
        "hstu_attn_fwd": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, sp, vp, vp, sz, u32, vp]),
        "hstu_attn_bwd": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp, sp, vp, sz, u32, vp]),
        "hstu_attn_fwd_targets_only": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, sp, vp, sz, vp]),
        "hstu_attn_bwd_targets_only": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp, sp, vp, sz, vp]),
        "hstu_attn_get_device_status": (ctypes.c_int, [vp, vp]),
        "hstu_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "hstu_attn_fwd_noalloc": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, sp, vp, vp]),
        "hstu_attn_shard_sequences": (ctypes.c_int, [vp, i32, i32, vp, vp]),
        "hstu_attn_test_wait_timeout": (ctypes.c_int, [vp, i32, vp]),
        "hstu_attn_test_set_handoff_limit": (ctypes.c_int, [ctypes.c_uint64]),
        "hstu_attn_build_func": (ctypes.c_int, [ctypes.POINTER(FuncSpec), vp, i32, ctypes.c_int64, i32, i32, vp,
                                                vp]),
        "hstu_attn_build_func_candidates": (ctypes.c_int, [vp, i32, i32, vp, vp]),
        "hstu_attn_targets_workspace_size": (sz, [sp, ctypes.c_int64]),
        "hstu_attn_project_workspace_size": (sz, [ctypes.c_int64, i32, i32, i32]),
        "hstu_attn_project_rows": (ctypes.c_int, [vp, ctypes.c_int64, vp, ctypes.c_int64, vp, vp, i32, i32, i32, vp,
                                                  vp, vp, sz, vp]),
        "hstu_attn_project_rows_bwd": (ctypes.c_int, [vp, vp, vp, ctypes.c_int64, vp, ctypes.c_int64, vp, i32, i32,
                                                      i32, vp, vp, vp, vp, sz, vp]),
        "hstu_attn_fwd_targets": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, sp, vp, sz, vp]),
        "hstu_attn_bwd_targets": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int64, vp, sp, vp,
                                                 sz, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _libs[path] = lib
    return lib


def status_string(status: int) -> str:
    try:
        return load().hstu_status_string(status).decode()
    except Exception:  # library missing: still format the error
        return STATUS_NAMES.get(status, "unknown")


def _check(status: int, what: str):
    if status != HSTU_OK:
        raise HstuError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if isinstance(dtype, tuple):
        if t.dtype not in dtype:
            raise ValueError(f"{name} must be one of {dtype}, got {t.dtype}")
    elif t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


DTYPES = {torch.bfloat16: 0, torch.float16: 1}
_FLOATS = tuple(DTYPES)


def _same_dtype(*ts):
    d = ts[0].dtype
    for t in ts[1:]:
        if t.dtype != d:
            raise ValueError(f"all tensors must share one dtype, got {d} and {t.dtype}")
    return DTYPES[d]


def make_shape(batch: int, total: int, heads: int, dim: int, nfunc: int, max_seqlen: int,
               alpha: Optional[float] = None, dim_v: int = 0, dtype: int = 0) -> Shape:
    """The C shape struct. ``dim`` is D_qk, ``dim_v`` D_v (0: equal to D_qk),
    ``dtype`` 0 for bf16 and 1 for fp16."""
    if alpha is None:
        alpha = 1.0 / math.sqrt(dim)
    return Shape(batch, total, heads, dim, nfunc, max_seqlen, alpha, dim_v, dtype)


def nfunc_supported(nfunc: int) -> bool:
    return bool(load().hstu_attn_nfunc_supported(nfunc))


def workspace_size(shape: Shape, mode: int = WS_FULL) -> int:
    return int(load().hstu_attn_workspace_size(ctypes.byref(shape), mode))


def alloc_workspace(shape: Shape, mode: int = WS_FULL, device="cuda") -> torch.Tensor:
    n = workspace_size(shape, mode)
    if n == 0:
        raise HstuError(2, "workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _shape_full(q, v, seq_offsets, func, max_seqlen, alpha):
    T, H, D = q.shape
    return make_shape(seq_offsets.numel() - 1, T, H, D, func.shape[0], max_seqlen, alpha, dim_v=v.shape[2],
                      dtype=DTYPES[q.dtype])


def plan(seq_offsets, func, shape: Shape, ws: torch.Tensor, row_counts=None, stream=None):
    _need(seq_offsets, torch.int32, "seq_offsets")
    _need(func, torch.int32, "func")
    _check(load().hstu_attn_plan(_ptr(seq_offsets), _ptr(func), ctypes.byref(shape), _ptr(row_counts),
                                 _ptr(ws), ws.numel(), _stream(stream)), "hstu_attn_plan")


def fwd(q, k, v, seq_offsets, func, max_seqlen: int, alpha: Optional[float] = None,
        ws: Optional[torch.Tensor] = None, row_counts: Optional[torch.Tensor] = None,
        reuse_plan: bool = False, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """o = HSTU attention over the jagged batch (see include/hstu_attn.h).
    q, k are (T, H, D_qk) and v (T, H, D_v), all bf16 or all fp16; o is
    (T, H, D_v)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, _FLOATS, n)
    _same_dtype(q, k, v)
    _need(seq_offsets, torch.int32, "seq_offsets")
    _need(func, torch.int32, "func")
    shape = _shape_full(q, v, seq_offsets, func, max_seqlen, alpha)
    if ws is None:
        ws = alloc_workspace(shape, WS_FULL, q.device)
    o = q.new_empty((q.shape[0], q.shape[1], v.shape[2])) if out is None else out
    flags = FLAG_REUSE_PLAN if reuse_plan else 0
    _check(load().hstu_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(seq_offsets), _ptr(func),
                                ctypes.byref(shape), _ptr(row_counts), _ptr(ws), ws.numel(), flags,
                                _stream(stream)), "hstu_attn_fwd")
    return o


def bwd(do, q, k, v, seq_offsets, func, max_seqlen: int, alpha: Optional[float] = None,
        ws: Optional[torch.Tensor] = None, reuse_plan: bool = False, outs=None,
        stream=None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(dq, dk, dv) of sum(o * do)."""
    for t, n in ((do, "dout"), (q, "q"), (k, "k"), (v, "v")):
        _need(t, _FLOATS, n)
    _same_dtype(do, q, k, v)
    _need(seq_offsets, torch.int32, "seq_offsets")
    _need(func, torch.int32, "func")
    shape = _shape_full(q, v, seq_offsets, func, max_seqlen, alpha)
    if ws is None:
        ws = alloc_workspace(shape, WS_FULL, q.device)
    dq, dk, dv = outs if outs is not None else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    flags = FLAG_REUSE_PLAN if reuse_plan else 0
    _check(load().hstu_attn_bwd(_ptr(do), _ptr(q), _ptr(k), _ptr(v), _ptr(dq), _ptr(dk), _ptr(dv),
                                _ptr(seq_offsets), _ptr(func), ctypes.byref(shape), _ptr(ws), ws.numel(),
                                flags, _stream(stream)), "hstu_attn_bwd")
    return dq, dk, dv


def _shape_targets(q_c, k, v, seq_offsets, func_c, max_seqlen, alpha):
    B, H, D = q_c.shape
    return make_shape(B, k.shape[0], H, D, func_c.shape[0], max_seqlen, alpha, dim_v=v.shape[2],
                      dtype=DTYPES[q_c.dtype])


def fwd_targets_only(q_c, k, v, seq_offsets, func_c, max_seqlen: int, alpha: Optional[float] = None,
                     ws: Optional[torch.Tensor] = None, out=None, stream=None) -> torch.Tensor:
    for t, n in ((q_c, "q_c"), (k, "k"), (v, "v")):
        _need(t, _FLOATS, n)
    _same_dtype(q_c, k, v)
    _need(seq_offsets, torch.int32, "seq_offsets")
    _need(func_c, torch.int32, "func_c")
    shape = _shape_targets(q_c, k, v, seq_offsets, func_c, max_seqlen, alpha)
    if ws is None:
        ws = alloc_workspace(shape, WS_TARGETS, q_c.device)
    o_c = q_c.new_empty((q_c.shape[0], q_c.shape[1], v.shape[2])) if out is None else out
    _check(load().hstu_attn_fwd_targets_only(_ptr(q_c), _ptr(k), _ptr(v), _ptr(o_c), _ptr(seq_offsets),
                                             _ptr(func_c), ctypes.byref(shape), _ptr(ws), ws.numel(),
                                             _stream(stream)), "hstu_attn_fwd_targets_only")
    return o_c


def bwd_targets_only(do_c, q_c, k, v, seq_offsets, func_c, max_seqlen: int,
                     alpha: Optional[float] = None, ws: Optional[torch.Tensor] = None, outs=None,
                     stream=None):
    for t, n in ((do_c, "dout_c"), (q_c, "q_c"), (k, "k"), (v, "v")):
        _need(t, _FLOATS, n)
    _same_dtype(do_c, q_c, k, v)
    _need(seq_offsets, torch.int32, "seq_offsets")
    _need(func_c, torch.int32, "func_c")
    shape = _shape_targets(q_c, k, v, seq_offsets, func_c, max_seqlen, alpha)
    if ws is None:
        ws = alloc_workspace(shape, WS_TARGETS, q_c.device)
    dq_c, dk, dv = outs if outs is not None else (torch.empty_like(q_c), torch.empty_like(k),
                                                  torch.empty_like(v))
    _check(load().hstu_attn_bwd_targets_only(_ptr(do_c), _ptr(q_c), _ptr(k), _ptr(v), _ptr(dq_c), _ptr(dk),
                                             _ptr(dv), _ptr(seq_offsets), _ptr(func_c), ctypes.byref(shape),
                                             _ptr(ws), ws.numel(), _stream(stream)),
           "hstu_attn_bwd_targets_only")
    return dq_c, dk, dv


def device_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the workspace status code."""
    return int(load().hstu_attn_get_device_status(_ptr(ws), _stream(stream)))


def fwd_noalloc(q, k, v, seq_offsets, func, max_seqlen: int, alpha: Optional[float] = None,
                row_counts: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                stream=None) -> torch.Tensor:
    """Forward pass for callers that cannot allocate device memory: the plan's
    scratch is a fixed array inside the library (hstu_attn_fwd_noalloc).
    ``out`` lets the caller supply the output buffer too."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, _FLOATS, n)
    _same_dtype(q, k, v)
    _need(seq_offsets, torch.int32, "seq_offsets")
    _need(func, torch.int32, "func")
    shape = _shape_full(q, v, seq_offsets, func, max_seqlen, alpha)
    o = q.new_empty((q.shape[0], q.shape[1], v.shape[2])) if out is None else out
    _check(load().hstu_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(seq_offsets), _ptr(func),
                                        ctypes.byref(shape), _ptr(row_counts), _stream(stream)),
           "hstu_attn_fwd_noalloc")
    return o


def shard_sequences(cost, world: int) -> Tuple[torch.Tensor, torch.Tensor]:
    """Splits a batch over ``world`` data-parallel ranks by whole sequences
    (hstu_attn_shard_sequences, host-only). ``cost`` is one non-negative work
    estimate per sequence. Returns (owner, rank_load): the rank of each
    sequence (int32) and each rank's total cost (int64), as CPU tensors."""
    c = torch.as_tensor(cost, dtype=torch.int64).contiguous()
    if c.dim() != 1 or c.is_cuda:
        raise ValueError("cost must be a 1-D host array")
    owner = torch.empty(c.numel(), dtype=torch.int32)
    load_ = torch.empty(max(world, 0), dtype=torch.int64)
    _check(load().hstu_attn_shard_sequences(_ptr(c), c.numel(), world, _ptr(owner), _ptr(load_)),
           "hstu_attn_shard_sequences")
    return owner, load_


def selftest_wait_timeout(ws: torch.Tensor, limit_ms: int, stream=None) -> None:
    """Enqueues the failure-path test of the in-kernel waits
    (hstu_attn_test_wait_timeout): a wait that nothing ends gives up after
    ``limit_ms`` and records HSTU_ERR_TIMEOUT in ``ws``."""
    _check(load().hstu_attn_test_wait_timeout(_ptr(ws), int(limit_ms), _stream(stream)),
           "hstu_attn_test_wait_timeout")


_KINDS = {"causal": FUNC_CAUSAL, "sla": FUNC_SLA, "onerank": FUNC_ONERANK}


def build_func(mask: str, seq_offsets: torch.Tensor, total: int, max_seqlen: int, nfunc: int, k1: int = 0,
               k2: int = 0, groups: int = 8, task_tokens: int = 3, out: Optional[torch.Tensor] = None,
               stream=None) -> torch.Tensor:
    """func (nfunc, total) int32 of a mask family, built on the device
    (hstu_attn_build_func). ``mask`` is "causal", "sla" or "onerank"."""
    _need(seq_offsets, torch.int32, "seq_offsets")
    if mask not in _KINDS:
        raise ValueError(f"mask must be one of {sorted(_KINDS)}")
    spec = FuncSpec(_KINDS[mask], k1, k2, groups, task_tokens)
    func = torch.empty((nfunc, total), dtype=torch.int32, device=seq_offsets.device) if out is None else out
    _check(load().hstu_attn_build_func(ctypes.byref(spec), _ptr(seq_offsets), seq_offsets.numel() - 1, total,
                                       max_seqlen, nfunc, _ptr(func), _stream(stream)), "hstu_attn_build_func")
    return func


def build_func_candidates(seq_offsets: torch.Tensor, nfunc: int = 1, out: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """func_c (nfunc, batch) int32 of the targets-only entry points (each
    sequence's last row sees the whole sequence), built on the device."""
    _need(seq_offsets, torch.int32, "seq_offsets")
    B = seq_offsets.numel() - 1
    func_c = torch.empty((nfunc, B), dtype=torch.int32, device=seq_offsets.device) if out is None else out
    _check(load().hstu_attn_build_func_candidates(_ptr(seq_offsets), B, nfunc, _ptr(func_c), _stream(stream)),
           "hstu_attn_build_func_candidates")
    return func_c


def targets_workspace(shape: Shape, num_candidates: int, device="cuda") -> torch.Tensor:
    n = int(load().hstu_attn_targets_workspace_size(ctypes.byref(shape), num_candidates))
    if n == 0:
        raise HstuError(2, "hstu_attn_targets_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _shape_multi(q_c, k, v, seq_offsets, func_c, max_seqlen, alpha):
    C, H, D = q_c.shape
    return make_shape(seq_offsets.numel() - 1, k.shape[0], H, D, func_c.shape[0], max_seqlen, alpha,
                      dim_v=v.shape[2], dtype=DTYPES[q_c.dtype])


def fwd_targets(q_c, k, v, seq_offsets, cand_offsets, func_c, max_seqlen: int, alpha: Optional[float] = None,
                ws: Optional[torch.Tensor] = None, out=None, stream=None) -> torch.Tensor:
    """Targets-only forward with any number of candidates per sequence
    (hstu_attn_fwd_targets): rows cand_offsets[b] .. cand_offsets[b+1] of
    q_c belong to sequence b."""
    for t, n in ((q_c, "q_c"), (k, "k"), (v, "v")):
        _need(t, _FLOATS, n)
    _same_dtype(q_c, k, v)
    for t, n in ((seq_offsets, "seq_offsets"), (cand_offsets, "cand_offsets"), (func_c, "func_c")):
        _need(t, torch.int32, n)
    shape = _shape_multi(q_c, k, v, seq_offsets, func_c, max_seqlen, alpha)
    C = q_c.shape[0]
    if ws is None:
        ws = targets_workspace(shape, C, q_c.device)
    o_c = q_c.new_empty((C, q_c.shape[1], v.shape[2])) if out is None else out
    _check(load().hstu_attn_fwd_targets(_ptr(q_c), _ptr(k), _ptr(v), _ptr(o_c), _ptr(seq_offsets),
                                        _ptr(cand_offsets), C, _ptr(func_c), ctypes.byref(shape), _ptr(ws),
                                        ws.numel(), _stream(stream)), "hstu_attn_fwd_targets")
    return o_c


def bwd_targets(do_c, q_c, k, v, seq_offsets, cand_offsets, func_c, max_seqlen: int,
                alpha: Optional[float] = None, ws: Optional[torch.Tensor] = None, outs=None, stream=None):
    """(dq_c, dk, dv) of the multi-candidate targets-only forward."""
    for t, n in ((do_c, "dout_c"), (q_c, "q_c"), (k, "k"), (v, "v")):
        _need(t, _FLOATS, n)
    _same_dtype(do_c, q_c, k, v)
    for t, n in ((seq_offsets, "seq_offsets"), (cand_offsets, "cand_offsets"), (func_c, "func_c")):
        _need(t, torch.int32, n)
    shape = _shape_multi(q_c, k, v, seq_offsets, func_c, max_seqlen, alpha)
    C = q_c.shape[0]
    if ws is None:
        ws = targets_workspace(shape, C, q_c.device)
    dq_c, dk, dv = outs if outs is not None else (torch.empty_like(q_c), torch.empty_like(k), torch.empty_like(v))
    _check(load().hstu_attn_bwd_targets(_ptr(do_c), _ptr(q_c), _ptr(k), _ptr(v), _ptr(dq_c), _ptr(dk), _ptr(dv),
                                        _ptr(seq_offsets), _ptr(cand_offsets), C, _ptr(func_c),
                                        ctypes.byref(shape), _ptr(ws), ws.numel(), _stream(stream)),
           "hstu_attn_bwd_targets")
    return dq_c, dk, dv


def project_workspace(num_rows: int, d_in: int, d_out: int, backward: bool, device="cuda") -> torch.Tensor:
    n = int(load().hstu_attn_project_workspace_size(num_rows, d_in, d_out, 1 if backward else 0))
    if n == 0:
        raise HstuError(2, "hstu_attn_project_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def project_rows(x, w, rows=None, bias=None, want_z=True, ws=None, stream=None):
    """(y, z) = (silu(x[rows] w^T + bias), x[rows] w^T + bias) on the
    listed rows of x (all rows if ``rows`` is None), hstu_attn_project_rows.
    x (T, d_in), w (d_out, d_in), one dtype (bf16 or fp16)."""
    _need(x, _FLOATS, "x")
    _need(w, _FLOATS, "w")
    ts = [x, w] + ([bias] if bias is not None else [])
    dtype = _same_dtype(*ts)
    if rows is not None:
        _need(rows, torch.int32, "rows")
    n = x.shape[0] if rows is None else rows.numel()
    d_out, d_in = w.shape
    if ws is None:
        ws = project_workspace(n if rows is not None else 0, d_in, d_out, False, x.device)
    y = x.new_empty((n, d_out))
    z = x.new_empty((n, d_out)) if want_z else None
    _check(load().hstu_attn_project_rows(_ptr(x), x.shape[0], _ptr(rows), n, _ptr(w), _ptr(bias), d_in, d_out,
                                         dtype, _ptr(y), _ptr(z), _ptr(ws), ws.numel(), _stream(stream)),
           "hstu_attn_project_rows")
    return y, z


def project_rows_bwd(dy, z, x, w, rows=None, want_dbias=True, ws=None, stream=None):
    """(dx_rows, dw, dbias) of sum(y * dy) for project_rows."""
    for t, name in ((dy, "dy"), (z, "z"), (x, "x"), (w, "w")):
        _need(t, _FLOATS, name)
    dtype = _same_dtype(dy, z, x, w)
    if rows is not None:
        _need(rows, torch.int32, "rows")
    n = x.shape[0] if rows is None else rows.numel()
    d_out, d_in = w.shape
    if ws is None:
        ws = project_workspace(n, d_in, d_out, True, x.device)
    dx = x.new_empty((n, d_in))
    dw = torch.empty_like(w)
    db = w.new_empty((d_out,)) if want_dbias else None
    _check(load().hstu_attn_project_rows_bwd(_ptr(dy), _ptr(z), _ptr(x), x.shape[0], _ptr(rows), n, _ptr(w), d_in,
                                             d_out, dtype, _ptr(dx), _ptr(dw), _ptr(db), _ptr(ws), ws.numel(),
                                             _stream(stream)), "hstu_attn_project_rows_bwd")
    return dx, dw, db


def set_handoff_limit_for_tests(limit_ns: int) -> None:
    """Test hook (hstu_attn_test_set_handoff_limit): shortens the attention
    kernels' accumulator hand-off wait; 0 restores the normal limit."""
    _check(load().hstu_attn_test_set_handoff_limit(int(limit_ns)), "hstu_attn_test_set_handoff_limit")
