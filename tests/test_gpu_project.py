"""The candidate-row projection of the targets-only layer (tcgen05 GEMMs with
a fused bias + SiLU epilogue) against the oracle: forward y and z,
backward dx of the listed rows, dw and the bias gradient; M, N and K tails;
all rows and a row list; bf16 and fp16; more output tiles than SMs, and
rows wider than one block of the SiLU-gradient kernel (d_out > 2048).

Tolerances follow from the arithmetic: inputs in the 16-bit type, fp32
accumulation, outputs rounded once to the 16-bit type (relative 2^-9 for
bf16), and G = dy * silu'(z) rounded to the 16-bit type before the two
backward GEMMs; relative L2 5e-3 on y and z, 1e-2 on the gradients."""
import numpy as np
import pytest
import torch

import oracle.hstu_oracle as orc
from jagged_hstu_attention_gb300 import binding as hb
from jagged_hstu_attention_gb300 import workloads as wl
from hstu_testutil import check_grad, np64, rel_l2

pytestmark = pytest.mark.gpu

Y_REL = 5e-3


def _inputs(T, d_in, d_out, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    x = wl.randn((T, d_in), g, dtype=dtype).cuda()
    w = (wl.randn((d_out, d_in), g).float() / np.sqrt(d_in)).to(dtype).cuda()
    b = (0.1 * wl.randn((d_out,), g).float()).to(dtype).cuda()
    dy = wl.randn((T, d_out), g, dtype=dtype).cuda()
    return x, w, b, dy


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("T,d_in,d_out,n_rows", [(300, 128, 192, 77), (1000, 512, 1024, 260), (50, 64, 64, 1),
                                                  (700, 256, 320, None), (5000, 128, 2112, None)])
def test_projection_matches_the_oracle(dtype, T, d_in, d_out, n_rows):
    x, w, b, dy_all = _inputs(T, d_in, d_out, dtype, seed=d_in + d_out)
    if n_rows is None:
        rows, hrows = None, np.arange(T)
    else:
        hrows = np.random.default_rng(n_rows).choice(T, size=n_rows, replace=False)
        rows = torch.tensor(hrows, dtype=torch.int32, device="cuda")
    y, z = hb.project_rows(x, w, rows=rows, bias=b)
    ry, rz = orc.project_rows(np64(x), hrows, np64(w), np64(b))
    assert rel_l2(np64(z), rz) <= Y_REL and rel_l2(np64(y), ry) <= Y_REL, (rel_l2(np64(z), rz), rel_l2(np64(y), ry))
    dy = dy_all[: len(hrows)].contiguous()
    dx, dw, db = hb.project_rows_bwd(dy, z, x, w, rows=rows)
    torch.cuda.synchronize()
    # the oracle differentiates through its own z; the kernels through the
    # rounded z they were given, which is within the z tolerance above
    rdx, rdw, rdb = orc.project_rows_backward(np64(dy), np64(x), hrows, np64(w), np64(b))
    check_grad(np64(dx), rdx[hrows], "dx_rows")
    check_grad(np64(dw), rdw, "dw")
    check_grad(np64(db), rdb, "dbias")


def test_projection_without_bias_and_z():
    x, w, _, _ = _inputs(129, 128, 256, torch.bfloat16, seed=1)
    rows = torch.tensor([128, 0, 64, 5], dtype=torch.int32, device="cuda")
    y, z = hb.project_rows(x, w, rows=rows, want_z=False)
    assert z is None
    ry, _ = orc.project_rows(np64(x), rows.cpu().numpy(), np64(w), None)
    assert rel_l2(np64(y), ry) <= Y_REL


def test_projection_rows_out_of_range_are_reported():
    x, w, b, _ = _inputs(64, 64, 64, torch.bfloat16, seed=2)
    rows = torch.tensor([3, 64, -1], dtype=torch.int32, device="cuda")
    ws = hb.project_workspace(3, 64, 64, False)
    y, _ = hb.project_rows(x, w, rows=rows, bias=b, ws=ws)
    assert hb.device_status(ws) == 5  # HSTU_ERR_DEVICE_INPUT
    ry, _ = orc.project_rows(np64(x), [3], np64(w), np64(b))
    assert rel_l2(np64(y[:1]), ry) <= Y_REL  # the valid row is still right


def test_projection_is_bitwise_repeatable():
    x, w, b, dy = _inputs(500, 256, 512, torch.bfloat16, seed=3)
    rows = torch.arange(0, 500, 3, dtype=torch.int32, device="cuda")
    a = hb.project_rows(x, w, rows=rows, bias=b)
    ga = hb.project_rows_bwd(dy[: rows.numel()].contiguous(), a[1], x, w, rows=rows)
    for _ in range(2):
        c = hb.project_rows(x, w, rows=rows, bias=b)
        gc = hb.project_rows_bwd(dy[: rows.numel()].contiguous(), c[1], x, w, rows=rows)
        assert torch.equal(a[0], c[0]) and torch.equal(a[1], c[1])
        for u, v in zip(ga, gc):
            assert torch.equal(u, v)
