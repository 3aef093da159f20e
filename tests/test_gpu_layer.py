"""GPU parity of the whole layer (moe_layer_forward) against the oracle on
the five workloads: routing/dispatch outputs bit-exact, layer outputs within
the per-row tolerance (2e-2 bf16, 1e-4 fp32).  Small-T versions are checked
on every token; full-size versions route and dispatch every token on both
sides and compare the layer output on at least 256 tokens: a seeded sample,
the tokens at both ends of every expert's rows and at its 128-row tile
boundaries, and every fully dropped token."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_gates_close, assert_rows_close, cfg_for, to_dev

pytestmark = pytest.mark.gpu


def _run_layer(w, inp_dev, T, add_residual):
    cfg = cfg_for(w, T=T, add_residual=add_residual)
    layer = moe.MoeLayer(cfg, inp_dev["w_router"], inp_dev.get("w_up"), inp_dev.get("w_down"),
                         inp_dev.get("shared_up"), inp_dev.get("shared_down"),
                         inp_dev.get("logit_bias"), inp_dev.get("sel_bias"))
    y = layer(inp_dev["x"]).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    return layer, y


def _oracle(w, inp_cpu, add_residual, tokens=None):
    return oracle.layer_forward(
        inp_cpu["x"], inp_cpu["w_router"], k=w.k, E=w.E, R=w.R, d_ff=w.d_ff, act=w.act,
        score=w.score, renorm=w.renorm, capacity_factor=w.capacity_factor,
        logit_bias=inp_cpu["logit_bias"], sel_bias=inp_cpu["sel_bias"], w_up=inp_cpu.get("w_up"),
        w_down=inp_cpu.get("w_down"), shared_up=inp_cpu.get("shared_up"),
        shared_down=inp_cpu.get("shared_down"), add_residual=add_residual, tokens=tokens)


def _compare(w, layer, y, ref, tokens):
    b = layer.buf
    assert torch.equal(b.topk_idx.cpu(), ref["topk_idx"])
    assert_gates_close(b.topk_gate.cpu(), ref["topk_gate"],
                       w.k if (w.renorm or w.score == "sigmoid") else w.E)
    assert torch.equal(b.expert_counts.cpu(), ref["expert_counts"])
    assert torch.equal(b.expert_offsets.cpu(), ref["expert_offsets"])
    assert torch.equal(b.slot_row.cpu(), ref["slot_row"])
    assert torch.equal(b.rank_counts.cpu(), ref["rank_counts"])
    assert torch.equal(b.rank_splits.cpu(), ref["rank_splits"])
    assert int(b.n_dropped.item()) == ref["n_dropped"]
    assert torch.equal(b.row_token[: ref["rows"]].cpu(), ref["row_token"])
    tol = 1e-4 if w.dtype == "f32" else 2e-2
    return assert_rows_close(y.cpu()[tokens], ref["y"], tol)


@pytest.mark.parametrize("name,T,resid", [("toy", 4096, False), ("toy", 1000, True),
                                          ("mixtral", 48, False), ("switch", 1536, True),
                                          ("switch", 2048, False), ("deepseek", 64, True)])
def test_layer_small(name, T, resid):
    w = W.WORKLOADS[name]
    if name == "switch":
        # a tighter capacity so that small batches still drop
        w = w.replace(capacity_factor=1.0)
    inp = W.make_inputs(w, T=T)
    layer, y = _run_layer(w, to_dev(inp), T, resid)
    ref = _oracle(w, inp, resid)
    _compare(w, layer, y, ref, torch.arange(T))
    if name == "switch":
        assert ref["n_dropped"] > 0


def test_layer_rank_limited_deepseek():
    """The DeepSeek-shaped layer with rank-limited routing (4 of 8 ranks)."""
    w = W.WORKLOADS["deepseek"].replace(max_ranks=4)
    inp = W.make_inputs(w, T=128)
    layer, y = _run_layer(w, to_dev(inp), 128, True)
    ref = oracle.layer_forward(
        inp["x"], inp["w_router"], k=w.k, E=w.E, R=w.R, d_ff=w.d_ff, act=w.act, score=w.score,
        renorm=w.renorm, sel_bias=inp["sel_bias"], w_up=inp["w_up"], w_down=inp["w_down"],
        shared_up=inp["shared_up"], shared_down=inp["shared_down"], add_residual=True,
        max_ranks=4)
    _compare(w, layer, y, ref, torch.arange(128))


@pytest.mark.parametrize("s", [0.0, 1.5])
def test_layer_identity_sweep_small(s):
    w = W.sweep(4096, s)
    inp = W.make_inputs(w, T=2048)
    layer, y = _run_layer(w, to_dev(inp), 2048, False)
    ref = _oracle(w, inp, False)
    _compare(w, layer, y, ref, torch.arange(2048))


def _stratified_tokens(layer, w, n_random, seed=17):
    """Tokens whose layer outputs are compared at full size: a seeded random
    sample, plus for every expert the tokens of its first and last rows and
    (up to 64 experts) of the rows on both sides of its 128-row tile
    boundaries (every 4th boundary for long experts), where the grouped GEMM's
    tiles change."""
    g = torch.Generator().manual_seed(seed)
    picked = [torch.randperm(w.T, generator=g)[:n_random], torch.tensor([0, w.T - 1])]
    offs = layer.buf.expert_offsets.cpu().tolist()
    rt = layer.buf.row_token.cpu()
    rows = []
    for e in range(w.E):
        lo, hi = offs[e], offs[e + 1]
        if hi <= lo:
            continue
        rows += [lo, hi - 1]
        if w.E > 64:
            continue  # 256 small experts: both ends of each already give ~500 tokens
        bounds = list(range(lo + 128, hi, 128))
        step = 4 if len(bounds) > 8 else 1
        for b in bounds[::step]:
            rows += [b - 1, b]
    picked.append(rt[torch.tensor(rows, dtype=torch.long)].long())
    return torch.unique(torch.cat(picked))


@pytest.mark.parametrize("name", ["toy", "switch", "deepseek", "mixtral"])
def test_layer_full_size_sampled(name):
    w = W.WORKLOADS[name]
    inp_dev = W.make_inputs(w, device=DEV)
    inp = {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in inp_dev.items()}
    layer, y = _run_layer(w, inp_dev, w.T, False)
    n_random = {"toy": 512, "switch": 256, "deepseek": 96, "mixtral": 128}[name]
    toks = _stratified_tokens(layer, w, n_random)
    assert toks.numel() >= 256
    slot = layer.buf.slot_row.cpu()
    dropped = (slot < 0).all(1).nonzero().flatten()
    if dropped.numel():
        # fully dropped tokens: exactly zero without the residual
        assert torch.all(y[dropped.to(DEV)] == 0)
        toks = torch.unique(torch.cat([toks, dropped[:64]]))
    ref = _oracle(w, inp, False, tokens=toks)
    _compare(w, layer, y, ref, toks)


@pytest.mark.parametrize("name,T", [("deepseek", 96), ("toy", 500), ("switch", 700)])
def test_layer_forward_host_equals_device_call(name, T):
    """moe_layer_forward_host (host x in, host y out, copies enqueued by the
    library) gives the device call's output bit for bit, twice in a row."""
    w = W.WORKLOADS[name]
    if name == "deepseek":
        w = w.replace(d=512, add_residual=True)
    inp = W.make_inputs(w, T=T)
    dev = to_dev(inp)
    layer, y = _run_layer(w, dev, T, w.add_residual)
    x_host = inp["x"].contiguous().pin_memory()
    for _ in range(2):
        y_host = torch.empty(y.shape, dtype=y.dtype).pin_memory()
        layer.forward_host(x_host, y_host)
        torch.cuda.synchronize()
        assert layer.device_status() == 0
        assert torch.equal(y_host, y.cpu())
