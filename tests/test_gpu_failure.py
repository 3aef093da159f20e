"""Failure detection without a GPU fault: a scan block that never publishes
makes its successor's bounded look-back wait run out.  The kernel records
MOE_DEV_LOOKBACK_TIMEOUT in the status word and returns; the host reads the
status, and the next normal dispatch on the same context is correct."""
import time

import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, run_dispatch

pytestmark = pytest.mark.gpu


def test_lookback_wait_times_out_and_context_survives():
    T, d, E, k, R = 256, 64, 8, 2, 4          # 8 scan blocks of 32 tokens
    cfg = moe.make_config(T, d, E, k, R, 0, 0, "bf16", "softmax", True, 0.0, 0, "identity")
    idx = W.random_topk(T, E, k, seed=2).to(DEV)
    x = W._grid_int((T, d), -8, 8, 8.0, W._gen(2, DEV), DEV).to(torch.bfloat16)
    rows = moe.moe_max_rows(cfg)
    i32 = dict(dtype=torch.int32, device=DEV)
    bufs = [torch.zeros((rows, d), dtype=torch.bfloat16, device=DEV), torch.zeros(rows, **i32),
            torch.zeros((T, k), **i32), torch.zeros(E, **i32), torch.zeros(E + 1, **i32),
            torch.zeros(R, **i32), torch.zeros((R, R), **i32), torch.zeros(1, **i32)]
    ws = moe.alloc_workspace(cfg)
    t0 = time.time()
    moe.moe_test_dispatch_stall(cfg, x, idx, *bufs, stall_block=1, wait_limit_us=20000, ws=ws)
    torch.cuda.synchronize()
    waited = time.time() - t0
    status = moe.moe_read_device_status(ws)
    assert status & moe.MOE_DEV_LOOKBACK_TIMEOUT
    assert waited < 3.0                        # bounded by the 20 ms limit, not the default 4 s
    # the same context and workspace still dispatch correctly
    out = run_dispatch(cfg, x, idx.cpu(), ws=ws)
    assert out["status"] == 0
    ref = oracle.dispatch(idx.cpu(), E, R, -1)
    assert torch.equal(out["slot_row"].cpu(), ref["slot_row"])
    assert torch.equal(out["expert_offsets"].cpu(), ref["expert_offsets"])


def test_stall_hook_rejects_bad_arguments():
    cfg = moe.make_config(64, 64, 8, 2, 4, 0, 0, "bf16", "softmax", True, 0.0, 0, "identity")
    with pytest.raises(moe.MoeError):
        moe.moe_test_dispatch_stall(cfg, 0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 0x6000, 0x7000,
                                    0x8000, None, 0x9000, stall_block=-1, wait_limit_us=10,
                                    ws=0xa000)
