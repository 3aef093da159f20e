"""GPU parity of Step 4 (Combine) against the oracle."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import Guarded, DEV, assert_rows_close

pytestmark = pytest.mark.gpu


def _setup(T, d, E, k, R, cap, dtype, seed):
    idx = W.random_topk(T, E, k, seed=seed, skew=1.2)
    C = oracle.capacity(T, k, E, 0.0, cap)
    disp = oracle.dispatch(idx, E, R, C)
    g = W._gen(seed, "cpu")
    rows = max(disp["rows"], 1)
    yp = W._grid_int((rows, d), -8, 8, 8.0, g, "cpu").to(dtype)
    gate = torch.rand((T, k), generator=g)
    x = W._grid_int((T, d), -8, 8, 8.0, g, "cpu").to(dtype)
    shared = W._grid_int((T, d), -8, 8, 16.0, g, "cpu").to(dtype)
    return disp, yp, gate, x, shared


@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, 2e-2), (torch.float32, 1e-4)])
@pytest.mark.parametrize("T,d,E,k,cap,resid,shared", [
    (1, 64, 4, 2, 0, False, False),
    (3000, 1024, 64, 1, 40, True, False),   # top-1 (its own eight-in-flight variant), drops
    (2049, 576, 16, 1, 0, False, True),     # top-1, 72 vectors per bf16 row (not a multiple of 32)
    (333, 128, 8, 2, 60, False, False),
    (333, 128, 8, 2, 60, True, False),
    (1024, 512, 64, 8, 90, True, True),
    (4100, 7168, 256, 8, 0, False, True),
    # small batches of wide k = 8 rows, ragged T, drops, with and without a residual
    (3001, 4096, 128, 8, 50, False, False),
    (3001, 4096, 128, 8, 50, True, False),
])
def test_combine_matches_oracle(dtype, tol, T, d, E, k, cap, resid, shared):
    disp, yp, gate, x, sh = _setup(T, d, E, k, 4, cap, dtype, seed=T + d)
    cfg = moe.make_config(T, d, E, k, 4, 64, 1 if shared else 0,
                          "bf16" if dtype == torch.bfloat16 else "f32", "softmax", True, 0.0, cap,
                          "gelu", resid)
    yg = Guarded((T, d), dtype, 0)
    y = yg.t
    moe.moe_combine(cfg, yp.to(DEV), disp["slot_row"].to(DEV), gate.to(DEV),
                    sh.to(DEV) if shared else None, x.to(DEV) if resid else None, y)
    torch.cuda.synchronize()
    yg.check("y")
    toks = torch.arange(T)
    ref = oracle.combine(toks, yp, torch.arange(yp.shape[0], dtype=torch.int32), disp["slot_row"],
                         gate, sh.double() if shared else None, x if resid else None)
    assert_rows_close(y, ref, tol)
    dropped = (disp["slot_row"] < 0).all(1)
    if dropped.any():
        yd = y.cpu()[dropped].double()
        if not shared:
            expect = x[dropped].double() if resid else torch.zeros_like(yd)
            assert torch.equal(yd, expect)
