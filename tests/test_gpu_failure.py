"""Failure detection without a GPU fault: a pipeline stage of the expert
GEMM that is never loaded makes the MMA issuer's bounded wait run out.  The
kernel records MOE_DEV_GEMM_TIMEOUT in the status word, raises its abort flag,
drains its MMAs, frees tensor memory and returns; the host reads the status,
and the next normal FFN call on the same context and workspace is correct."""
import time

import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_rows_close

pytestmark = pytest.mark.gpu


def _case(counts, d, f, act, seed):
    E = len(counts)
    offs = torch.zeros(E + 1, dtype=torch.int32)
    offs[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32), 0)
    N = int(offs[-1])
    rows_up = 2 * f if act == "swiglu" else f
    g = W._gen(seed, "cpu")
    w_up = W._grid_normal((E, rows_up, d), 0.08, 2.0 ** -9, 0.125, g, "cpu").to(torch.bfloat16)
    w_dn = W._grid_normal((E, d, f), 0.08, 2.0 ** -9, 0.125, g, "cpu").to(torch.bfloat16)
    xp = W._grid_int((N, d), -8, 8, 8.0, g, "cpu").to(torch.bfloat16)
    cfg = moe.make_config(N, d, E, 1, 1, f, 0, "bf16", "softmax", True, 0.0, 0, act)
    return cfg, offs, w_up, w_dn, xp


@pytest.mark.parametrize("act", ["swiglu", "gelu"])
def test_gemm_wait_times_out_and_context_survives(act):
    counts, d, f = [300, 0, 200, 77], 256, 256
    cfg, offs, w_up, w_dn, xp, = _case(counts, d, f, act, seed=5)
    N = xp.shape[0]
    xp_d, offs_d, wu_d, wd_d = xp.to(DEV), offs.to(DEV), w_up.to(DEV), w_dn.to(DEV)
    h = torch.zeros((N, f), dtype=torch.bfloat16, device=DEV)
    ws = moe.alloc_workspace(cfg)
    t0 = time.time()
    moe.moe_test_expert_ffn_stall(cfg, xp_d, offs_d, wu_d, h, stall_kb=1, wait_limit_us=20000,
                                  ws=ws)
    torch.cuda.synchronize()
    waited = time.time() - t0
    status = moe.moe_read_device_status(ws)
    assert status & moe.MOE_DEV_GEMM_TIMEOUT
    assert waited < 3.0                        # bounded by the 20 ms limit, not the default 4 s
    assert moe.moe_read_device_status(ws) == 0  # reading clears it
    # the same context and workspace still run the FFN correctly
    yp = torch.full((N, d), 7.0, dtype=torch.bfloat16, device=DEV)
    moe.moe_expert_ffn(cfg, xp_d, offs_d, wu_d, wd_d, h, yp, ws=ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    for e in range(len(counts)):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            ref = oracle.expert_ffn(xp[lo:hi], w_up[e], w_dn[e], act, f)
            assert_rows_close(yp[lo:hi], ref, 2e-2)


def test_stall_hook_rejects_bad_arguments():
    cfg, offs, w_up, w_dn, xp = _case([64, 64], 128, 128, "gelu", seed=1)
    ws = moe.alloc_workspace(cfg)
    h = torch.zeros((128, 128), dtype=torch.bfloat16, device=DEV)
    args = (xp.to(DEV), offs.to(DEV), w_up.to(DEV), h)
    for kb, us in ((-1, 1000), (2, 1000), (0, 0), (0, 5000000)):   # d/64 = 2 K blocks
        with pytest.raises(moe.MoeError):
            moe.moe_test_expert_ffn_stall(cfg, *args, stall_kb=kb, wait_limit_us=us, ws=ws)
    cfg32 = moe.make_config(128, 128, 2, 1, 1, 128, 0, "f32", "softmax", True, 0.0, 0, "gelu")
    with pytest.raises(moe.MoeError):
        moe.moe_test_expert_ffn_stall(cfg32, *args, stall_kb=0, wait_limit_us=1000, ws=ws)


@pytest.mark.parametrize("name,T", [("mixtral", 96), ("deepseek", 200), ("toy", 96),
                                    ("switch", 150)])
def test_nonfinite_router_input_is_reported(name, T):
    """A NaN and an infinity planted in x on the host (plain data: nothing
    faults) make those tokens' logits non-finite: the router sets
    MOE_DEV_NONFINITE in the status word, and every other token is routed
    exactly as the oracle routes it.  Clean inputs leave the bit clear."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, ffn=False, T=T)
    cfg = moe.config_from_workload(w, T=T)
    dev = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}

    def route(x):
        idx = torch.zeros((T, w.k), dtype=torch.int32, device=DEV)
        gate = torch.zeros((T, w.k), dtype=torch.float32, device=DEV)
        ws = moe.alloc_workspace(cfg)
        moe.moe_route(cfg, x, dev["w_router"], dev.get("logit_bias"), dev.get("sel_bias"), idx,
                      gate, ws)
        return idx.cpu(), moe.moe_read_device_status(ws)

    _, clean = route(dev["x"])
    assert clean == 0
    x = inp["x"].clone()
    x[5, 3] = float("nan")
    x[T - 7, 0] = float("inf")
    idx, status = route(x.to(DEV))
    assert status == moe.MOE_DEV_NONFINITE
    ridx, _ = oracle.route(inp["x"], inp["w_router"], w.k, w.score, w.renorm, inp["logit_bias"],
                           inp["sel_bias"])
    ok = torch.ones(T, dtype=torch.bool)
    ok[5] = ok[T - 7] = False
    assert torch.equal(idx[ok], ridx[ok])
