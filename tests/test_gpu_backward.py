"""GPU parity of the backward of the two exchanges (moe_combine_backward,
moe_dispatch_backward) against the oracle.

Tolerances: d_yp = g*dy rounded once: relative
2^-8 (bf16) or 2^-22 (fp32) per element; d_gate is an fp32 dot product of d
terms: |err| <= 1e-5 * sum_c |dy_c * yp_c|; dx is a sum of <= k rows rounded
once: per row 2^-7 (bf16) / 1e-6 (fp32) of max|ref row|."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_rows_close

pytestmark = pytest.mark.gpu


def _case(T, d, E, k, cap, dtype, seed):
    idx = W.random_topk(T, E, k, seed=seed, skew=1.3)
    disp = oracle.dispatch(idx, E, 2, cap)
    g = W._gen(seed, "cpu")
    yp = W._grid_normal((max(disp["rows"], 1), d), 0.5, 2.0 ** -9, 4.0, g, "cpu").to(dtype)
    dy = W._grid_normal((T, d), 0.5, 2.0 ** -9, 4.0, g, "cpu").to(dtype)
    gate = torch.rand((T, k), generator=g)
    cfg = moe.make_config(T, d, E, k, 2, 64, 0, "bf16" if dtype == torch.bfloat16 else "f32",
                          "softmax", True, 0.0, cap, "gelu")
    return cfg, disp, yp, dy, gate


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,d,E,k,cap", [(1, 64, 4, 2, 0), (777, 512, 16, 2, 80),
                                         (4100, 4096, 8, 2, 0), (2048, 7168, 256, 8, 50)])
def test_combine_backward(dtype, T, d, E, k, cap):
    cfg, disp, yp, dy, gate = _case(T, d, E, k, cap, dtype, seed=T + d)
    rows = yp.shape[0]
    d_yp = torch.full((rows, d), 3.0, dtype=dtype, device=DEV)
    d_gate = torch.full((T, k), float("nan"), device=DEV)
    moe.moe_combine_backward(cfg, dy.to(DEV), yp.to(DEV), disp["slot_row"].to(DEV), gate.to(DEV),
                             d_yp, d_gate)
    torch.cuda.synchronize()
    ref_yp, ref_g = oracle.combine_backward(dy, yp, disp["slot_row"], gate)
    used = disp["slot_row"][disp["slot_row"] >= 0].long()
    got = d_yp.cpu().double()
    rel = 2.0 ** -8 if dtype == torch.bfloat16 else 2.0 ** -22
    err = (got[used] - ref_yp[used]).abs()
    assert torch.all(err <= rel * ref_yp[used].abs() + 1e-30)
    unused = torch.ones(rows, dtype=torch.bool)
    unused[used] = False
    assert torch.all(got[unused] == 3.0)
    # gate gradients
    sr = disp["slot_row"].long()
    mag = torch.zeros((T, k), dtype=torch.float64)
    for j in range(k):
        kept = sr[:, j] >= 0
        mag[kept, j] = (dy.double()[kept] * yp.double()[sr[kept, j]]).abs().sum(1)
    gerr = (d_gate.cpu().double() - ref_g).abs()
    assert torch.all(gerr <= 1e-5 * mag + 1e-30)
    assert torch.all(d_gate.cpu()[sr < 0] == 0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("T,d,E,k,cap", [(333, 256, 8, 2, 60), (4096, 7168, 256, 8, 100)])
def test_dispatch_backward(dtype, T, d, E, k, cap):
    cfg, disp, yp, dy, gate = _case(T, d, E, k, cap, dtype, seed=T * 3 + d)
    dx = torch.empty((T, d), dtype=dtype, device=DEV)
    moe.moe_dispatch_backward(cfg, yp.to(DEV), disp["slot_row"].to(DEV), dx)
    torch.cuda.synchronize()
    ref = oracle.dispatch_backward(yp, disp["slot_row"], T)
    assert_rows_close(dx, ref, 2.0 ** -7 if dtype == torch.bfloat16 else 1e-6)
