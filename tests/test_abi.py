"""C ABI checks that need no GPU: the library loads, exports every function
the header declares, and rejects bad arguments on the host with the right
status before anything is enqueued."""
import ctypes
import os
import re

import pytest

from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hstu_attn.h")


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    return hb.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hstu_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("hstu_attn_fwd", "hstu_attn_bwd", "hstu_attn_fwd_targets_only",
              "hstu_attn_bwd_targets_only", "hstu_attn_plan", "hstu_attn_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) <= set(hb.EXPORTED) | set(_declared())


def test_checked_build_exports_the_same_symbols(lib):
    checked = hb.load(hb.CHECKED_LIB_PATH)
    for name in _declared():
        assert hasattr(checked, name), name
    assert checked.hstu_status_string(7).decode() == lib.hstu_status_string(7).decode()
    assert "checked build" in lib.hstu_status_string(7).decode()


def _shape(**kw):
    s = dict(batch=4, total=1000, heads=2, dim=128, nfunc=5, max_seqlen=300, alpha=0.1, dim_v=0, dtype=0)
    s.update(kw)
    return hb.make_shape(s["batch"], s["total"], s["heads"], s["dim"], s["nfunc"], s["max_seqlen"],
                         s["alpha"], dim_v=s["dim_v"], dtype=s["dtype"])


def test_shape_variants_accepted_and_rejected(lib):
    for dim in (32, 64, 128):
        for dim_v in (0, 32, 64, 128):
            for dtype in (0, 1):
                assert hb.workspace_size(_shape(dim=dim, dim_v=dim_v, dtype=dtype), hb.WS_FULL) > 0
    # targets-only partials hold rows of the wider of D_qk and D_v
    assert hb.workspace_size(_shape(dim=32, dim_v=128), hb.WS_TARGETS) == \
        hb.workspace_size(_shape(dim=128, dim_v=32), hb.WS_TARGETS) == hb.workspace_size(_shape(), hb.WS_TARGETS)
    for bad in (dict(dim_v=48), dict(dim_v=256), dict(dim=256), dict(dtype=2), dict(dtype=-1)):
        assert hb.workspace_size(_shape(**bad), hb.WS_FULL) == 0, bad


def test_nfunc_supported(lib):
    assert [hb.nfunc_supported(n) for n in range(12)] == [False, True, False, True, False, True, False,
                                                          True, False, True, False, False]
    assert not hb.nfunc_supported(-1)


def test_workspace_size(lib):
    full = hb.workspace_size(_shape(), hb.WS_FULL)
    tgt = hb.workspace_size(_shape(), hb.WS_TARGETS)
    assert full > 0 and full % 256 == 0 and tgt > 0
    assert hb.workspace_size(_shape(max_seqlen=3000), hb.WS_FULL) > full
    for bad in (dict(nfunc=2), dict(dim=96), dict(batch=0), dict(max_seqlen=0),
                dict(max_seqlen=40000), dict(heads=0), dict(total=-1)):
        assert hb.workspace_size(_shape(**bad), hb.WS_FULL) == 0, bad
    assert hb.workspace_size(_shape(), 7) == 0


def test_work_index_bound(lib):
    """Backward list entries x heads must stay below 2^30 (the kernels' int32
    work index, plus a grid of overrun): 2 min(B NT, T/128 + B) entries."""
    # 2 * min(1000 * 256, 2**20 // 128 + 1000) = 18384 entries
    ok = _shape(batch=1000, total=1 << 20, max_seqlen=32768, heads=(1 << 30) // 18384)
    assert hb.workspace_size(ok, hb.WS_FULL) > 0
    bad = _shape(batch=1000, total=1 << 20, max_seqlen=32768, heads=(1 << 30) // 18384 + 1)
    assert hb.workspace_size(bad, hb.WS_FULL) == 0
    # here T / 128 + B decides: 2 * min(4 * 3, 1000 // 128 + 4) = 22 entries
    assert hb.workspace_size(_shape(max_seqlen=300, heads=(1 << 30) // 22), hb.WS_FULL) > 0
    assert hb.workspace_size(_shape(max_seqlen=300, heads=(1 << 30) // 22 + 1), hb.WS_FULL) == 0
    # and B NT for a small maximum: 2 * min(4 * 1, 7 + 4) = 8 entries
    assert hb.workspace_size(_shape(max_seqlen=100, heads=(1 << 30) // 8 - 1), hb.WS_FULL) > 0
    assert hb.workspace_size(_shape(max_seqlen=100, heads=(1 << 30) // 8), hb.WS_FULL) == 0


def _fwd(lib, shape, q=1 << 20, k=1 << 20, v=1 << 20, o=1 << 20, off=1 << 20, func=1 << 20,
         ws=1 << 20, ws_bytes=1 << 30):
    vp = ctypes.c_void_p
    return lib.hstu_attn_fwd(vp(q), vp(k), vp(v), vp(o), vp(off), vp(func), ctypes.byref(shape), None,
                             vp(ws), ws_bytes, 0, None)


def test_host_validation_statuses(lib):
    s = _shape()
    assert _fwd(lib, s, q=0) == 1                       # null tensor
    assert _fwd(lib, s, o=(1 << 20) + 8) == 1           # misaligned tensor
    assert _fwd(lib, s, off=0) == 1                     # null offsets
    assert _fwd(lib, _shape(nfunc=4)) == 2              # unsupported nfunc
    assert _fwd(lib, _shape(dim=80)) == 2               # unsupported head_dim
    assert _fwd(lib, s, ws=0) == 3                      # null workspace
    assert _fwd(lib, s, ws=(1 << 20) + 64) == 3         # misaligned workspace
    assert _fwd(lib, s, ws_bytes=16) == 3               # workspace too small
    assert _fwd(lib, _shape(alpha=float("nan"))) == 1   # NaN alpha
    vp = ctypes.c_void_p
    assert lib.hstu_attn_bwd(vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), vp(0), vp(1 << 20), vp(1 << 20),
                             ctypes.byref(s), vp(1 << 20), 1 << 30, 0, None) == 1
    assert lib.hstu_attn_fwd_targets_only(vp(0), vp(1 << 20), vp(1 << 20), vp(1 << 20), vp(1 << 20),
                                          vp(1 << 20), ctypes.byref(s), vp(1 << 20), 1 << 30, None) == 1
    assert lib.hstu_attn_plan(vp(1 << 20), vp(1 << 20), ctypes.byref(_shape(nfunc=0)), None, vp(1 << 20),
                              1 << 30, None) == 2
    assert lib.hstu_attn_get_device_status(vp(0), None) == 3


def test_status_strings(lib):
    for st in range(7):
        assert len(hb.status_string(st)) > 0
    assert "unknown" in hb.status_string(42)


def test_wait_timeout_hook_checks_its_arguments(lib):
    vp = ctypes.c_void_p
    assert lib.hstu_attn_test_wait_timeout(None, 20, None) == 3          # null workspace
    assert lib.hstu_attn_test_wait_timeout(vp((1 << 20) + 64), 20, None) == 3  # misaligned
    assert lib.hstu_attn_test_wait_timeout(vp(1 << 20), 0, None) == 1    # limit too small
    assert lib.hstu_attn_test_wait_timeout(vp(1 << 20), 2001, None) == 1  # limit too large


def test_binding_fails_loudly_without_the_library():
    with pytest.raises(RuntimeError, match="missing"):
        hb.load(os.path.join(ROOT, "no_such_dir", "libhstu_attn.so"))
    prev = hb.select_library(os.path.join(ROOT, "no_such_dir", "libhstu_attn.so"))
    try:
        with pytest.raises(RuntimeError, match="missing"):
            hb.load()
    finally:
        hb.select_library(prev)


def test_binding_has_no_cpu_path():
    import torch
    q = torch.zeros((4, 1, 32), dtype=torch.bfloat16)
    off = torch.tensor([0, 4], dtype=torch.int32)
    func = torch.full((1, 4), 4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        hb.fwd(q, q, q, off, func, 4)
    with pytest.raises(ValueError, match="CUDA"):
        hb.bwd(q, q, q, q, off, func, 4)


def _spec(kind=0, k1=0, k2=0, groups=8, task_tokens=3):
    return hb.FuncSpec(kind, k1, k2, groups, task_tokens)


def test_build_func_rejects_bad_arguments_on_the_host(lib):
    vp = ctypes.c_void_p
    fake = vp(256)  # never dereferenced: every case fails its host check first
    cases = [
        (None, fake, 2, 100, 64, 5, fake, 1),                      # no spec
        (_spec(), None, 2, 100, 64, 5, fake, 1),                   # no offsets
        (_spec(), fake, 0, 100, 64, 5, fake, 1),                   # batch < 1
        (_spec(), fake, 2, -1, 64, 5, fake, 1),                    # total < 0
        (_spec(), fake, 2, 100, 0, 5, fake, 1),                    # max_seqlen < 1
        (_spec(), fake, 2, 100, 64, 4, fake, 2),                   # even nfunc
        (_spec(), fake, 2, 100, 64, 5, None, 1),                   # no func
        (_spec(), vp(258), 2, 100, 64, 5, fake, 1),                # misaligned offsets
        (_spec(kind=7), fake, 2, 100, 64, 5, fake, 1),             # unknown family
        (_spec(kind=1, k1=-1), fake, 2, 100, 64, 5, fake, 1),      # negative prefix
        (_spec(kind=1, k1=4, k2=2), fake, 2, 100, 64, 1, fake, 2),  # SLA needs two intervals
        (_spec(kind=2, groups=0), fake, 2, 100, 64, 5, fake, 1),   # no groups
        (_spec(kind=2), fake, 2, 100, 64, 3, fake, 2),             # OneRank needs three intervals
    ]
    for spec, off, batch, total, n, nfunc, func, want in cases:
        st = lib.hstu_attn_build_func(ctypes.byref(spec) if spec is not None else None, off, batch, total, n,
                                      nfunc, func, None)
        assert st == want, (spec and spec.kind, batch, total, n, nfunc, st)
    assert lib.hstu_attn_build_func_candidates(None, 2, 1, fake, None) == 1
    assert lib.hstu_attn_build_func_candidates(fake, 2, 2, fake, None) == 2
    assert lib.hstu_attn_build_func_candidates(fake, 0, 1, fake, None) == 1


def test_handoff_limit_hook_rejects_out_of_range(lib):
    with pytest.raises(hb.HstuError):
        hb.set_handoff_limit_for_tests(3_000_000_000)
    hb.set_handoff_limit_for_tests(5)
    hb.set_handoff_limit_for_tests(0)  # back to the kernels' normal limit
