"""GPU parity of Step 1 (Route) against the oracle: bit-exact expert choices
and tie-breaks, gates within the fp32 bound."""
import json
import os

import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_gates_close, cfg_for, run_dispatch, run_route, to_dev

pytestmark = pytest.mark.gpu


def _check_route(w, inp_cpu, T=None):
    cfg = cfg_for(w, T=inp_cpu["x"].shape[0])
    idx, gate = run_route(cfg, to_dev(inp_cpu))
    ridx, rgate = oracle.route(inp_cpu["x"], inp_cpu["w_router"], w.k, w.score, w.renorm,
                               inp_cpu["logit_bias"], inp_cpu["sel_bias"])
    assert torch.equal(idx, ridx), f"{int((idx != ridx).any(1).sum())} tokens differ"
    n_terms = w.k if w.renorm or w.score == "sigmoid" else w.E
    assert_gates_close(gate, rgate, n_terms)


@pytest.mark.parametrize("name", ["toy", "mixtral", "switch", "deepseek"])
@pytest.mark.parametrize("T", [1, 33, 517])
def test_route_workloads_small_T(name, T):
    w = W.WORKLOADS[name]
    _check_route(w, W.make_inputs(w, ffn=False, T=T))


@pytest.mark.parametrize("s", [0.0, 1.5])
def test_route_sweep_skew(s):
    w = W.sweep(4096, s)
    _check_route(w, W.make_inputs(w, ffn=False, T=300))


@pytest.mark.parametrize("E,k,score,renorm", [(4, 2, "softmax", True), (8, 8, "sigmoid", False),
                                               (16, 3, "softmax", False), (32, 4, "sigmoid", True),
                                               (48, 5, "softmax", True), (64, 1, "softmax", False),
                                               (128, 6, "sigmoid", True), (256, 8, "sigmoid", True),
                                               (200, 7, "softmax", True), (192, 8, "softmax", False),
                                               (64, 8, "sigmoid", False), (256, 2, "softmax", True)])
def test_route_ties_and_shapes(E, k, score, renorm):
    """A coarse weight grid makes exact ties common: the lower index must win.
    At this T the tensor-core router cuts E = 64 ... 256 into expert slices
    merged by a second kernel (96-expert slices for E = 192, with softmax
    gates over all experts); E = 200 is not cut."""
    T = 257
    d = 8 if E <= 8 else 64       # short rows keep exact ties frequent for small E
    g = W._gen(E * 100 + k, "cpu")
    x = W._grid_int((T, d), -8, 8, 8.0, g, "cpu").to(torch.bfloat16)
    wr = W._grid_int((E, d), -1, 1, 512.0, g, "cpu").to(torch.bfloat16)
    sel = (W._grid_int((E,), -1, 1, 4096.0, g, "cpu") if score == "sigmoid" else None)
    lb = W._grid_int((E,), 0, 1, 4096.0, g, "cpu")
    w = W.Workload("tie", T, d, E, 1, k, 64, "identity", "bf16", score, renorm, 0.0, 0, 0,
                   "normal512")
    inp = dict(x=x, w_router=wr, logit_bias=lb, sel_bias=sel)
    _, _, L = oracle.route(x, wr, k, score, renorm, lb, sel, return_logits=True)
    assert sum(len(set(r.tolist())) < E for r in L) > T // 8
    _check_route(w, inp)


@pytest.mark.parametrize("name", ["switch", "deepseek"])
def test_route_full_size_sampled(name):
    """The full workload through the bench's launch; the oracle scores a
    seeded sample of tokens (routing is per token)."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, ffn=False)
    cfg = cfg_for(w)
    idx, gate = run_route(cfg, to_dev(inp))
    samp = torch.randperm(w.T, generator=torch.Generator().manual_seed(7))[:384]
    samp = torch.cat([samp, torch.tensor([0, w.T - 1])])
    ridx, rgate = oracle.route(inp["x"][samp], inp["w_router"], w.k, w.score, w.renorm,
                               inp["logit_bias"], inp["sel_bias"])
    assert torch.equal(idx[samp], ridx)
    assert_gates_close(gate[samp], rgate, w.k if (w.renorm or w.score == "sigmoid") else w.E)


def test_route_sigmoid_every_grid_logit():
    """Every logit on the 1/4096 grid in [-16, 16] (131073 values) gets the
    oracle's fp32 sigmoid, bit for bit.  Tokens hit base values v/4096 with
    v = m0 + 8*m1 + 64*(sum of the rest); experts add a logit bias of 4e."""
    E, k, d = 8, 8, 256
    T = 16385
    base = torch.arange(T, dtype=torch.int64) - 65536          # v in [-65536, -49152]
    q, r = torch.div(base, 64, rounding_mode="floor"), base % 64
    x = torch.zeros((T, d), dtype=torch.float32)
    x[:, 0] = (r % 8).float() / 8
    x[:, 1] = (r // 8).float() / 8
    rest = q.abs()
    sign = torch.sign(q).float()
    for i in range(2, d):
        take = torch.clamp(rest, max=8)
        x[:, i] = sign * take.float() / 8
        rest = rest - take
    assert int(rest.abs().max()) == 0
    wr = torch.full((E, d), 64.0 / 512)
    wr[:, 0] = 1.0 / 512
    wr[:, 1] = 8.0 / 512
    lb = torch.arange(E, dtype=torch.float32) * 4.0
    x, wr = x.to(torch.bfloat16), wr.to(torch.bfloat16)
    _, _, L = oracle.route(x, wr, k, "sigmoid", False, lb, None, return_logits=True)
    grid = torch.unique(L.double() * 4096)
    assert grid.numel() == 131073 and int(grid.min()) == -65536 and int(grid.max()) == 65536
    w = W.Workload("sig", T, d, E, 1, k, 64, "identity", "bf16", "sigmoid", False, 0.0, 0, 0,
                   "normal512")
    _check_route(w, dict(x=x, w_router=wr, logit_bias=lb, sel_bias=None))
    cfg = cfg_for(w)
    _, gate = run_route(cfg, to_dev(dict(x=x, w_router=wr, logit_bias=lb, sel_bias=None)))
    _, rgate = oracle.route(x, wr, k, "sigmoid", False, lb, None)
    assert torch.equal(gate, rgate)   # no-renorm sigmoid gates are the scores themselves


@pytest.mark.parametrize("lo,hi", [(-12.0, 4.0), (-95.0, -60.0)])
def test_route_sigmoid_scores_of_arbitrary_fp32_logits(lo, hi):
    """Sigmoid scores of logits with arbitrary fp32 mantissas (a random logit
    bias per expert on top of the grid logits), bit for bit against the oracle's
    double-precision evaluation rounded to fp32: 32768 chosen scores in the
    middle of the sigmoid (bias in [-12, 4]), or far out in its tail (bias in
    [-95, -60], down to the subnormal range, where the double path decides)."""
    E, k, d, T = 256, 8, 64, 4096
    g = torch.Generator().manual_seed(int(lo * 7 + hi))
    x = torch.randint(-8, 9, (T, d), generator=g).float().div(8).to(torch.bfloat16)
    wr = torch.randint(-8, 9, (E, d), generator=g).float().div(64).to(torch.bfloat16)
    lb = (torch.rand(E, generator=g, dtype=torch.float64) * (hi - lo) + lo).float()
    w = W.Workload("sigf", T, d, E, 1, k, 64, "identity", "bf16", "sigmoid", False, 0.0, 0, 0,
                   "normal512")
    inp = dict(x=x, w_router=wr, logit_bias=lb, sel_bias=None)
    idx, gate = run_route(cfg_for(w), to_dev(inp))
    ridx, rgate = oracle.route(x, wr, k, "sigmoid", False, lb, None)
    assert torch.equal(idx, ridx.to(idx.dtype))
    assert torch.equal(gate, rgate)


def test_route_snippet_loads_on_gpu():
    """The Ultralytics routing snippet through the GPU route and dispatch:
    per-expert loads 948..1087 and per-GPU loads 1968..2139."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                    "snippet_router_loads.json")))
    torch.manual_seed(g["seed"])
    hidden = torch.randn(g["tokens"], g["d_model"])
    layer = torch.nn.Linear(g["d_model"], g["experts"])
    w = W.Workload("snippet", g["tokens"], g["d_model"], g["experts"], g["gpus"], g["top_k"], 0,
                   "identity", "f32", "softmax", True, 0.0, 0, 0, "uniform64")
    inp = dict(x=hidden, w_router=layer.weight.detach(), logit_bias=layer.bias.detach(),
               sel_bias=None)
    cfg = cfg_for(w)
    idx, _ = run_route(cfg, to_dev(inp))
    out = run_dispatch(cfg, hidden.to(DEV), idx)
    ec, rc = out["expert_counts"].cpu(), out["rank_counts"].cpu()
    assert int(ec.sum()) == g["assignments"]
    assert (int(ec.min()), int(ec.max())) == (g["expert_load_min"], g["expert_load_max"])
    assert (int(rc.min()), int(rc.max())) == (g["gpu_load_min"], g["gpu_load_max"])


def test_route_deterministic():
    w = W.WORKLOADS["deepseek"]
    inp = to_dev(W.make_inputs(w, ffn=False, T=1024))
    cfg = cfg_for(w, T=1024)
    a = run_route(cfg, inp)
    b = run_route(cfg, inp)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("E,R,M,k,score", [(8, 4, 2, 2, "softmax"), (16, 4, 1, 3, "sigmoid"),
                                            (32, 8, 2, 4, "sigmoid"), (32, 32, 3, 2, "softmax"),
                                            (64, 8, 3, 6, "softmax"), (96, 8, 2, 8, "sigmoid"),
                                            (256, 8, 4, 8, "sigmoid"), (256, 32, 5, 8, "softmax")])
def test_route_rank_limited_ties(E, R, M, k, score, dtype):
    """Rank-limited routing (at most M of R ranks per token) on a coarse grid
    with many exact ties, bit for bit against the oracle: the bf16 router on
    the tensor cores and the fp32 FFMA routers (E <= 32 and E > 32 forms)."""
    T, d = 300, 64
    g = W._gen(E * 7 + M, "cpu")
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    x = W._grid_int((T, d), -8, 8, 8.0, g, "cpu").to(dt)
    wr = W._grid_int((E, d), -1, 1, 512.0, g, "cpu").to(dt)
    sel = W._grid_int((E,), -1, 1, 4096.0, g, "cpu") if score == "sigmoid" else None
    w = W.Workload("rl", T, d, E, R, k, 64, "identity", dtype, score, True, 0.0, 0, 0,
                   "normal512", max_ranks=M)
    cfg = cfg_for(w)
    idx, gate = run_route(cfg, to_dev(dict(x=x, w_router=wr, logit_bias=None, sel_bias=sel)))
    ridx, rgate = oracle.route(x, wr, k, score, True, None, sel, R=R, max_ranks=M)
    assert torch.equal(idx, ridx), f"{int((idx != ridx).any(1).sum())} tokens differ"
    assert_gates_close(gate, rgate, k)
    per = E // R
    assert all(len(set((idx[t] // per).tolist())) <= M for t in range(T))


def test_route_rank_limited_deepseek_shape():
    """DeepSeek-V3's limit (a token's experts on at most 4 of 8 ranks) on the
    DeepSeek-shaped router, every token of a 2048-token batch."""
    w = W.WORKLOADS["deepseek"].replace(max_ranks=4)
    inp = W.make_inputs(w, ffn=False, T=2048)
    cfg = cfg_for(w, T=2048)
    idx, gate = run_route(cfg, to_dev(inp))
    ridx, rgate = oracle.route(inp["x"], inp["w_router"], w.k, w.score, w.renorm, None,
                               inp["sel_bias"], R=w.R, max_ranks=4)
    assert torch.equal(idx, ridx)
    assert_gates_close(gate, rgate, w.k)
    free, _ = oracle.route(inp["x"], inp["w_router"], w.k, w.score, w.renorm, None,
                           inp["sel_bias"])
    assert not torch.equal(free, ridx)   # the limit actually binds on this workload
