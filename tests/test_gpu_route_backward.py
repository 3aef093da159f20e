"""GPU parity of the router backward (moe_route_backward) against the
oracle: the logit gradients through each gate form, the input, weight and
logit-bias gradients, on the forward's own expert choices.

Tolerances: d_logits per token within 2e-5 * sum_j |dg_j| (fp32 gates, exp
and sums of at most E terms; the off-choice entries of the sparse forms are
exactly 0); dx per row within tol * max|ref row| and d_w_router within
tol * max|ref| (tol 1e-4 fp32, 1e-2 bf16: one rounding of an fp32 sum);
d_logit_bias within 1e-4 * sum_t |dL[t,e]|."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_rows_close, run_route

pytestmark = pytest.mark.gpu


def _case(name, T, **over):
    w = W.WORKLOADS[name].replace(**over) if over else W.WORKLOADS[name]
    inp = W.make_inputs(w, ffn=False, T=T)
    return w, inp


@pytest.mark.parametrize("name,T,over", [
    ("toy", 333, {}),                                          # fp32, softmax renorm, k=2
    ("mixtral", 200, {"d": 1024}),                             # bf16 softmax renorm
    ("switch", 300, {}),                                       # full softmax gate, logit bias
    ("deepseek", 257, {"d": 512}),                             # sigmoid renorm + selection bias
    ("deepseek", 130, {"d": 512, "renorm": False}),            # plain sigmoid gates
    ("deepseek", 96, {"d": 512, "max_ranks": 4}),              # rank-limited choices
    ("deepseek", 64, {}),                                      # full width, 256 experts
    ("toy", 77, {"score": "sigmoid", "renorm": False, "E": 16, "R": 4, "k": 3}),  # fp32 sigmoid
    # long batches: the weight gradient's token range split over a cluster of 8 / 2 CTAs
    ("mixtral", 16384, {"d": 1024}),
    ("toy", 5000, {"E": 6, "R": 2}),                           # fp32, an expert block of 6
])
def test_route_backward_matches_oracle(name, T, over):
    w, inp = _case(name, T, **over)
    cfg = moe.config_from_workload(w, T=T)
    dev = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
    idx, _ = run_route(cfg, dev)
    g = torch.Generator().manual_seed(T + w.E)
    dg = torch.randn((T, w.k), generator=g)
    dt = w.torch_dtype
    dL = torch.full((T, w.E), float("nan"), device=DEV)
    dx = torch.empty((T, w.d), dtype=dt, device=DEV)
    dw = torch.empty((w.E, w.d), dtype=dt, device=DEV)
    dlb = torch.empty(w.E, device=DEV)
    moe.moe_route_backward(cfg, dev["x"], dev["w_router"], dev.get("logit_bias"), idx.to(DEV),
                           dg.to(DEV), dL, dx, dw, dlb)
    torch.cuda.synchronize()
    rL, rx, rw, rb = oracle.route_backward(inp["x"], inp["w_router"], idx, dg, w.score, w.renorm,
                                           inp["logit_bias"])
    gL = dL.cpu().double()
    scale = dg.double().abs().sum(1, keepdim=True)
    assert torch.all((gL - rL).abs() <= 2e-5 * scale), float(((gL - rL).abs() / scale).max())
    if w.score != "softmax" or w.renorm:
        assert torch.all(gL[rL == 0] == 0)
    tol = 1e-4 if w.dtype == "f32" else 1e-2
    assert_rows_close(dx.cpu(), rx, tol)
    err_w = float((dw.cpu().double() - rw).abs().max())
    assert err_w <= tol * float(rw.abs().max()), err_w
    lim = 1e-4 * rL.abs().sum(0) + 1e-12
    assert torch.all((dlb.cpu().double() - rb).abs() <= lim)


def test_route_backward_optional_outputs_and_empty_batch():
    """dx, d_w_router and d_logit_bias may be NULL; with no tokens the weight
    and bias gradients are zero."""
    w, inp = _case("switch", 50)
    cfg = moe.config_from_workload(w, T=50)
    dev = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
    idx, _ = run_route(cfg, dev)
    dg = torch.randn((50, w.k), generator=torch.Generator().manual_seed(3)).to(DEV)
    dL = torch.empty((50, w.E), device=DEV)
    moe.moe_route_backward(cfg, dev["x"], dev["w_router"], dev["logit_bias"], idx.to(DEV), dg, dL)
    torch.cuda.synchronize()
    rL, _, _, _ = oracle.route_backward(inp["x"], inp["w_router"], idx, dg.cpu(), w.score,
                                        w.renorm, inp["logit_bias"])
    assert torch.all((dL.cpu().double() - rL).abs() <= 2e-5 * dg.cpu().double().abs().sum(1, keepdim=True))
    cfg0 = moe.config_from_workload(w, T=0)
    dw = torch.full((w.E, w.d), 3.0, dtype=w.torch_dtype, device=DEV)
    dlb = torch.full((w.E,), 3.0, device=DEV)
    moe.moe_route_backward(cfg0, dev["x"], dev["w_router"], None, idx.to(DEV), dg, dL, None, dw,
                           dlb)
    torch.cuda.synchronize()
    assert torch.all(dw == 0) and torch.all(dlb == 0)


def test_route_backward_weight_gradient_is_deterministic():
    """The weight and bias gradients add their partial sums in a fixed order
    (also across the CTAs of a cluster): two calls agree bit for bit."""
    w, inp = _case("mixtral", 8192, d=1024)
    cfg = moe.config_from_workload(w, T=8192)
    dev = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
    idx, _ = run_route(cfg, dev)
    dg = torch.randn((8192, w.k), generator=torch.Generator().manual_seed(5)).to(DEV)
    outs = []
    for _ in range(2):
        dL = torch.empty((8192, w.E), device=DEV)
        dw = torch.empty((w.E, w.d), dtype=w.torch_dtype, device=DEV)
        dlb = torch.empty(w.E, device=DEV)
        moe.moe_route_backward(cfg, dev["x"], dev["w_router"], None, idx.to(DEV), dg, dL, None,
                               dw, dlb)
        torch.cuda.synchronize()
        outs.append((dw.view(torch.int16).clone(), dlb.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
