"""The backward pieces composed on a real forward's layout: after a GPU layer
forward, moe_combine_backward -> moe_expert_ffn_backward -> moe_dispatch_backward
on its slot rows, offsets, gates and expert rows, against the same chain
through the oracle (fed the GPU forward's own yp, gates and layout, so each
step is compared on identical inputs).

Tolerances: d_gate as the combine-backward test (fp32 dot products:
1e-5 * sum |dy * yp|); dx (the routed experts' part of dL/dx) per row
relative to the row's max |ref|: 3e-2 bf16 (the FFN backward's 2e-2 plus the
bf16 rounding of d_yp and of the summed rows), 1e-4 fp32; expert weight
gradients against each matrix's max |ref|, same tolerances."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_rows_close

pytestmark = pytest.mark.gpu

CASES = {
    # reduced-width versions of the page-shaped layers (the oracle stays fast)
    "mixtral": dict(T=512, d=512, d_ff=1024),
    "switch": dict(T=1024, d=256, d_ff=512, E=16),
    "deepseek": dict(T=256, d=512, d_ff=256, E=32),
    "toy": dict(T=512, d=256, d_ff=512),
}


@pytest.mark.parametrize("name", list(CASES))
def test_backward_chain_matches_oracle(name):
    w = W.get(name).replace(**CASES[name])
    inp = W.make_inputs(w, device=DEV)
    cfg = moe.config_from_workload(w)
    layer = moe.MoeLayer(cfg, inp["w_router"], inp["w_up"], inp["w_down"], inp.get("shared_up"),
                         inp.get("shared_down"), inp.get("logit_bias"), inp.get("sel_bias"),
                         device=DEV)
    layer(inp["x"])
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    b = layer.buf
    T, d = w.T, w.d
    dt = w.torch_dtype
    dy = W._grid_normal((T, d), 0.5, 2.0 ** -9, 4.0, W._gen(w.seed + 50, "cpu"), "cpu").to(dt)
    rows = max(moe.moe_max_rows(cfg), 1)
    d_yp = torch.zeros((rows, d), dtype=dt, device=DEV)
    d_gate = torch.full((T, w.k), float("nan"), device=DEV)
    moe.moe_combine_backward(cfg, dy.to(DEV), b.yp, b.slot_row, b.topk_gate, d_yp, d_gate)
    d_xp = torch.zeros((rows, d), dtype=dt, device=DEV)
    d_wu = torch.empty_like(inp["w_up"])
    d_wd = torch.empty_like(inp["w_down"])
    scratch = torch.empty(moe.moe_expert_ffn_backward_scratch_size(cfg, True), dtype=torch.uint8,
                          device=DEV)
    moe.moe_expert_ffn_backward(cfg, b.xp, b.expert_offsets, inp["w_up"], inp["w_down"], d_yp,
                                d_xp, d_wu, d_wd, scratch, b.ws)
    dx = torch.empty((T, d), dtype=dt, device=DEV)
    moe.moe_dispatch_backward(cfg, d_xp, b.slot_row, dx)
    torch.cuda.synchronize()
    assert layer.device_status() == 0

    # the same chain through the oracle, from the GPU forward's state
    sr = b.slot_row.cpu()
    gate = b.topk_gate.cpu()
    yp = b.yp.cpu()
    xp = b.xp.cpu()
    off = b.expert_offsets.cpu()
    n = int(off[-1])
    ref_dyp, ref_dgate = oracle.combine_backward(dy, yp, sr, gate)
    kept = sr.long() >= 0
    mag = torch.zeros((T, w.k), dtype=torch.float64)
    for j in range(w.k):
        kj = kept[:, j]
        mag[kj, j] = (dy.double()[kj] * yp.double()[sr[kj, j].long()]).abs().sum(1)
    gerr = (d_gate.cpu().double() - ref_dgate).abs()
    assert torch.all(gerr <= 1e-5 * mag + 1e-30)
    assert torch.all(d_gate.cpu()[~kept] == 0)

    tol = 3e-2 if dt == torch.bfloat16 else 1e-4
    ref_dxp = torch.zeros((max(n, 1), d), dtype=torch.float64)
    wu, wd = inp["w_up"].cpu(), inp["w_down"].cpu()
    # the oracle's expert FFN backward takes rows of one dtype: round d_yp as the GPU stores it
    ref_dyp_dt = ref_dyp.to(dt)
    for e in range(w.E):
        lo, hi = int(off[e]), int(off[e + 1])
        r_in, r_wu, r_wd = oracle.expert_ffn_backward(xp[lo:hi], wu[e], wd[e], ref_dyp_dt[lo:hi],
                                                      w.act, w.d_ff)
        ref_dxp[lo:hi] = r_in
        for got, ref in ((d_wu[e], r_wu), (d_wd[e], r_wd)):
            scale = float(ref.abs().max()) if ref.numel() else 0.0
            err = (got.double().cpu() - ref).abs()
            assert float(err.max()) <= tol * scale if scale else torch.all(err == 0)
    ref_dx = oracle.dispatch_backward(ref_dxp.float(), sr, T)  # fp32 storage: far below tol
    assert_rows_close(dx, ref_dx, tol)
    # a token with every slot dropped gets exactly zero
    dropped = ~kept.any(1)
    assert torch.all(dx.cpu()[dropped] == 0)
