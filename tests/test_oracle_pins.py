"""Pins for the CPU oracle: each check ties an oracle function to something
other than itself -- values the pages print, brute force on tiny inputs,
closed forms, invariants, or special cases that reduce to a library routine.
No GPU is used here.
"""
import json
import math
import os
from fractions import Fraction

import pytest
import torch
import torch.nn.functional as F

import moe_workloads as W
import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# Printed values
# --------------------------------------------------------------------------

def _snippet_router():
    """Regenerate the routing snippet's inputs: torch seed 0, hidden states
    drawn first, then a default-initialised linear router (weight, bias)."""
    g = _gold("snippet_router_loads.json")
    torch.manual_seed(g["seed"])
    hidden = torch.randn(g["tokens"], g["d_model"])
    layer = torch.nn.Linear(g["d_model"], g["experts"])
    return g, hidden, layer.weight.detach().clone(), layer.bias.detach().clone()


def test_snippet_expert_and_gpu_loads():
    """Ultralytics 'How Tokens Move Between GPUs': 8 experts, top-2, 4096
    tokens -> per-expert loads 948..1087, per-GPU loads 1968..2139."""
    g, hidden, w, b = _snippet_router()
    idx, _ = oracle.route(hidden, w, g["top_k"], "softmax", True, logit_bias=b)
    disp = oracle.dispatch(idx, g["experts"], g["gpus"], -1)
    ec, rc = disp["expert_counts"], disp["rank_counts"]
    assert int(ec.sum()) == g["assignments"]
    assert int(ec.min()) == g["expert_load_min"]
    assert int(ec.max()) == g["expert_load_max"]
    assert int(rc.min()) == g["gpu_load_min"]
    assert int(rc.max()) == g["gpu_load_max"]
    assert g["assignments"] // g["experts"] == g["even_share"]
    # the per-GPU load is the sum of its experts' loads (two per GPU, in order)
    assert rc.tolist() == ec.view(g["gpus"], -1).sum(1).tolist()


def test_capacity_example_drops_last_fifty():
    """ai360xpert 'Load Balancing and Dropped Tokens': cap 100, 150 routed -> 50 dropped."""
    g = _gold("capacity_example.json")
    T, E, R = g["routed"], 2, 1
    idx = torch.zeros((T, 1), dtype=torch.int32)  # every token picks expert 0
    C = oracle.capacity(T, 1, E, 0.0, explicit=g["capacity"])
    disp = oracle.dispatch(idx, E, R, C)
    assert disp["n_dropped"] == g["dropped"]
    assert disp["expert_counts"].tolist() == [g["routed"], 0]
    assert disp["expert_offsets"].tolist() == [0, g["capacity"], g["capacity"]]
    sr = disp["slot_row"].flatten()
    # in-order overflow: the first 100 tokens are kept in order, the last 50 skip
    assert sr[: g["capacity"]].tolist() == list(range(g["capacity"]))
    assert (sr[g["capacity"]:] == -1).all()
    # the skipped tokens reach the next layer unchanged through the residual
    x = W._grid_int((T, 16), -8, 8, 8.0, W._gen(5, "cpu"), "cpu")
    xp = oracle.permute(x, disp["slot_row"], disp["rows"])
    yp = oracle.expert_ffn(xp, None, None, "identity", 0)
    gate = torch.ones((T, 1))
    y = oracle.combine(torch.arange(T), yp, torch.arange(disp["rows"], dtype=torch.int32),
                       disp["slot_row"], gate, resid=x)
    assert torch.equal(y[g["capacity"]:], x[g["capacity"]:].double())
    assert torch.equal(y[: g["capacity"]], 2 * x[: g["capacity"]].double())


def test_capacity_factor_closed_form():
    """Ultralytics 'Load Balancing and Capacity': 1.25x the even share."""
    cf = _gold("capacity_factor.json")["capacity_factor"]
    assert oracle.capacity(32768, 1, 64, cf) == 640
    assert oracle.capacity(16, 2, 4, 0.0) == -1
    assert oracle.capacity(16, 2, 4, 0.0, explicit=3) == 3
    # exact rational ceiling over a spread of shapes
    for T, k, E, cf in [(4096, 2, 8, 1.25), (1000, 3, 7, 1.5), (33, 1, 64, 1.25), (17, 8, 256, 2.0),
                        (131072, 8, 256, 1.0), (5, 2, 3, 0.75)]:
        exact = math.ceil(Fraction(cf) * T * k / E)
        assert oracle.capacity(T, k, E, cf) == exact


# --------------------------------------------------------------------------
# Route: brute force on tiny inputs, closed forms, library special cases
# --------------------------------------------------------------------------

def _tiny_router(T, E, d, seed, grid_w=True):
    g = W._gen(seed, "cpu")
    x = W._grid_int((T, d), -8, 8, 8.0, g, "cpu")
    if grid_w:
        w = W._grid_int((E, d), -1, 1, 512.0, g, "cpu")  # coarse grid: many exact ties
    else:
        w = torch.randn((E, d), generator=g)
    return x, w


def _brute_topk(key, k):
    """Full sort on (-key, expert) -- a different procedure from the oracle's
    k rounds of selection."""
    T, E = key.shape
    out = []
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(key[t, e]), e))
        out.append(order[:k])
    return torch.tensor(out, dtype=torch.int32)


@pytest.mark.parametrize("E", [4, 8])
@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_route_softmax_bruteforce(E, k):
    if k > E:
        pytest.skip()
    x, w = _tiny_router(16, E, 4, seed=10 + E + k)
    lb = (torch.arange(E, dtype=torch.float32) % 2) / 4096.0
    idx, gate, L = oracle.route(x, w, k, "softmax", True, logit_bias=lb, return_logits=True)
    # logits through a library matmul in fp64 (exact on the grid)
    L_ref = (x.double() @ w.double().T).float() + lb
    assert torch.equal(L, L_ref)
    ties = sum(len(set(row.tolist())) < E for row in L_ref)
    assert ties > 0, "the coarse grid should produce tied logits"
    assert torch.equal(idx, _brute_topk(L_ref, k))
    # renormalised gates = library softmax over the chosen logits
    chosen = torch.gather(L_ref.double(), 1, idx.long())
    g_ref = torch.softmax(chosen, dim=1)
    assert torch.allclose(gate.double(), g_ref, rtol=1e-7, atol=0)
    assert torch.allclose(gate.double().sum(1), torch.ones(16, dtype=torch.float64), atol=k * 2 ** -23)


@pytest.mark.parametrize("k", [1, 2, 4])
def test_route_softmax_no_renorm_is_full_probability(k):
    x, w = _tiny_router(16, 8, 24, seed=3, grid_w=False)
    idx, gate, L = oracle.route(x, w, k, "softmax", False, return_logits=True)
    p = torch.softmax(L.double(), dim=1)
    assert torch.allclose(gate.double(), torch.gather(p, 1, idx.long()), rtol=1e-7, atol=0)
    # top-1 without renorm is the largest probability (Switch-style gate)
    assert torch.allclose(gate[:, 0].double(), p.max(1).values, rtol=1e-7, atol=0)


@pytest.mark.parametrize("renorm", [True, False])
@pytest.mark.parametrize("E,k", [(4, 2), (8, 3), (8, 8)])
def test_route_sigmoid_selection_bias_bruteforce(E, k, renorm):
    x, w = _tiny_router(16, E, 4, seed=20 + E + k)
    sel = torch.tensor([((e * 5) % 3 - 1) / 4096.0 for e in range(E)], dtype=torch.float32)
    idx, gate, L = oracle.route(x, w, k, "sigmoid", renorm, sel_bias=sel, return_logits=True)
    L_ref = (x.double() @ w.double().T).float()
    assert torch.equal(L, L_ref)
    s_ref = torch.sigmoid(L_ref.double()).float()       # library sigmoid, rounded to fp32
    key = s_ref + sel                                    # one fp32 add
    assert torch.equal(idx, _brute_topk(key, k))
    assert sum(len(set(row.tolist())) < E for row in key) > 0, "want tied keys"
    s_chosen = torch.gather(s_ref, 1, idx.long()).double()
    if renorm:
        g_ref = s_chosen / s_chosen.sum(1, keepdim=True)
        assert torch.allclose(gate.double(), g_ref, rtol=1e-7, atol=0)
    else:
        # the bias never reaches the gate: gate = unbiased sigmoid score
        assert torch.equal(gate, s_chosen.float())


def test_selection_bias_changes_choice_not_gate():
    """A large selection bias on one expert makes it win every token, yet the
    gate stays the plain sigmoid score."""
    x, w = _tiny_router(16, 4, 24, seed=7)
    sel = torch.tensor([0.0, 0.0, 4.0, 0.0])
    idx, gate, L = oracle.route(x, w, 1, "sigmoid", False, sel_bias=sel, return_logits=True)
    assert (idx[:, 0] == 2).all()
    assert torch.equal(gate[:, 0], torch.sigmoid(L[:, 2].double()).float())


def test_softmax_with_selection_bias_is_rejected():
    x, w = _tiny_router(4, 4, 8, seed=1)
    with pytest.raises(ValueError):
        oracle.route(x, w, 1, "softmax", True, sel_bias=torch.zeros(4))


def test_sigmoid32_against_library_on_grid():
    """fp32 sigmoid score = library sigmoid in fp64 rounded to fp32, on the
    1/4096 logit grid (sampled), plus sigma(0) = 1/2 and symmetry."""
    v = torch.arange(-16 * 4096, 16 * 4096 + 1, 97, dtype=torch.float64) / 4096.0
    ref = torch.sigmoid(v).float()
    got = torch.tensor([oracle.sigmoid32(float(a)) for a in v])
    assert torch.equal(got, ref)
    assert oracle.sigmoid32(0.0) == 0.5
    for a in [0.25, 1.0, 3.5, 9.0]:
        assert abs(oracle.sigmoid32(a) + oracle.sigmoid32(-a) - 1.0) < 2 ** -23


def test_router_logits_exact_on_grid_deepseek_shape():
    """On the dyadic grid the fp32 logit equals the exact (fp64) dot product,
    for a DeepSeek-shaped router slice (d=7168, E=256)."""
    w = W.WORKLOADS["deepseek"]
    inp = W.make_inputs(w, ffn=False, T=64)
    _, _, L = oracle.route(inp["x"], inp["w_router"], w.k, w.score, w.renorm,
                           sel_bias=inp["sel_bias"], return_logits=True)
    exact = inp["x"].double() @ inp["w_router"].double().T
    assert torch.equal(L.double(), exact)
    assert torch.equal(L.double() * 4096, torch.round(L.double() * 4096))


# --------------------------------------------------------------------------
# Dispatch: brute force (per-expert list scan) and invariants
# --------------------------------------------------------------------------

def _brute_dispatch(idx, E, R, C):
    T, k = idx.shape
    lists = [[] for _ in range(E)]          # (token, slot) per expert, token order
    for t in range(T):
        for j in range(k):
            lists[int(idx[t, j])].append((t, j))
    kept = [lst if C < 0 else lst[:C] for lst in lists]
    rows = []                               # expert-major concatenation
    for e in range(E):
        rows.extend((e, t, j) for (t, j) in kept[e])
    slot_row = torch.full((T, k), -1, dtype=torch.int32)
    row_token = torch.empty(len(rows), dtype=torch.int32)
    for r, (e, t, j) in enumerate(rows):
        slot_row[t, j] = r
        row_token[r] = t
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + len(kept[e]))
    per = E // R
    src_size = -(-T // R)
    splits = torch.zeros((R, R), dtype=torch.int32)
    for (e, t, j) in rows:
        splits[t // src_size, e // per] += 1
    return dict(expert_counts=[len(l) for l in lists], expert_offsets=offsets,
                rank_counts=splits.sum(0).tolist(), rank_splits=splits, slot_row=slot_row,
                row_token=row_token, n_dropped=T * k - len(rows))


@pytest.mark.parametrize("T,E,k,R,C,skew", [(16, 4, 2, 2, -1, 0.0), (16, 4, 1, 4, 3, 1.0),
                                             (37, 8, 3, 4, 10, 1.5), (64, 16, 4, 8, 12, 1.2),
                                             (5, 4, 4, 1, 2, 0.0), (1, 4, 2, 2, 0, 0.0)])
def test_dispatch_bruteforce(T, E, k, R, C, skew):
    idx = W.random_topk(T, E, k, seed=T + E + k, skew=skew)
    got = oracle.dispatch(idx, E, R, C)
    ref = _brute_dispatch(idx, E, R, C)
    assert got["expert_counts"].tolist() == ref["expert_counts"]
    assert got["expert_offsets"].tolist() == ref["expert_offsets"]
    assert got["rank_counts"].tolist() == ref["rank_counts"]
    assert torch.equal(got["rank_splits"], ref["rank_splits"])
    assert torch.equal(got["slot_row"], ref["slot_row"])
    assert torch.equal(got["row_token"], ref["row_token"])
    assert got["n_dropped"] == ref["n_dropped"]


def test_dispatch_invariants_medium():
    T, E, k, R = 777, 32, 4, 8
    idx = W.random_topk(T, E, k, seed=11, skew=1.3)
    C = oracle.capacity(T, k, E, 1.1)
    d = oracle.dispatch(idx, E, R, C)
    kept = (d["expert_offsets"][1:] - d["expert_offsets"][:-1])
    assert int(d["expert_counts"].sum()) == T * k
    assert int(kept.sum()) == T * k - d["n_dropped"] == d["rows"]
    assert torch.equal(kept, torch.clamp(d["expert_counts"], max=C))
    assert d["n_dropped"] > 0
    # row_token strictly increasing inside each expert segment
    off = d["expert_offsets"].tolist()
    for e in range(E):
        seg = d["row_token"][off[e]:off[e + 1]]
        assert bool((seg[1:] > seg[:-1]).all())
    # un-permute inverts permute on every kept slot
    x = W._grid_int((T, 24), -8, 8, 8.0, W._gen(3, "cpu"), "cpu").to(torch.bfloat16)
    xp = oracle.permute(x, d["slot_row"], d["rows"])
    sr = d["slot_row"]
    for t in range(T):
        for j in range(k):
            if sr[t, j] >= 0:
                assert torch.equal(xp[sr[t, j]], x[t])
    assert torch.equal(x[d["row_token"].long()], xp)
    assert int(d["rank_splits"].sum()) == d["rows"]
    assert d["rank_counts"].tolist() == d["rank_splits"].sum(0).tolist()


# --------------------------------------------------------------------------
# Compute: special cases that reduce to library routines
# --------------------------------------------------------------------------

def test_ffn_gelu_structure_matches_library_matmuls():
    """With every pre-activation above 40, erf saturates to exactly 1 in fp64
    and GELU is the identity, so the FFN is two library matmuls.  f != d
    catches a transposed operand."""
    g = torch.Generator().manual_seed(4)
    n, d, f = 5, 48, 80
    x = 1 + torch.randint(0, 9, (n, d), generator=g).float() / 8
    w1 = 1 + torch.randint(0, 9, (f, d), generator=g).float() / 8
    w2 = torch.randint(-8, 9, (d, f), generator=g).float() / 8
    out = oracle.expert_ffn(x, w1, w2, "gelu", f)
    ref = (x.double() @ w1.double().T) @ w2.double().T
    assert torch.allclose(out, ref, rtol=1e-13, atol=0)


def test_ffn_swiglu_structure_matches_library_matmuls():
    """silu(v) = v exactly in fp64 for v > 40: the SwiGLU FFN is then
    ((x Wg^T) * (x Wu^T)) Wd^T with gate rows first in w_up."""
    g = torch.Generator().manual_seed(5)
    n, d, f = 4, 48, 40
    x = 1 + torch.randint(0, 9, (n, d), generator=g).float() / 8
    wg = 1 + torch.randint(0, 9, (f, d), generator=g).float() / 8
    wu = torch.randint(-8, 9, (f, d), generator=g).float() / 8
    wd = torch.randint(-8, 9, (d, f), generator=g).float() / 8
    out = oracle.expert_ffn(x, torch.cat([wg, wu]), wd, "swiglu", f)
    xd = x.double()
    ref = ((xd @ wg.double().T) * (xd @ wu.double().T)) @ wd.double().T
    assert torch.allclose(out, ref, rtol=1e-13, atol=1e-9)


def test_ffn_activations_match_torch_functional():
    """Identity weights isolate the activations: GELU(x) and silu(x) * x."""
    d = 32
    x = torch.linspace(-6, 6, 3 * d).view(3, d)
    eye = torch.eye(d)
    out = oracle.expert_ffn(x, eye, eye, "gelu", d)
    assert torch.allclose(out, F.gelu(x.double(), approximate="none"), rtol=1e-14, atol=1e-15)
    out = oracle.expert_ffn(x, torch.cat([eye, eye]), eye, "swiglu", d)
    assert torch.allclose(out, F.silu(x.double()) * x.double(), rtol=1e-14, atol=1e-15)


def test_ffn_identity_and_bf16_widening():
    x = W._grid_int((6, 16), -8, 8, 8.0, W._gen(9, "cpu"), "cpu").to(torch.bfloat16)
    assert torch.equal(oracle.expert_ffn(x, None, None, "identity", 0), x.double())
    eye = torch.eye(16, dtype=torch.bfloat16)
    out = oracle.expert_ffn(x, eye, eye, "gelu", 16)
    assert torch.allclose(out, F.gelu(x.double()), rtol=1e-14, atol=1e-15)


# --------------------------------------------------------------------------
# Combine and the whole layer: invariants
# --------------------------------------------------------------------------

@pytest.mark.parametrize("k", [1, 2, 8])
def test_identity_experts_return_x(k):
    """Identity experts, renormalised gates, no drops: combine returns x
    (exactly for k = 1, within fp32 gate rounding otherwise)."""
    T, E, d = 64, 16, 32
    g = W._gen(31, "cpu")
    x = W._grid_int((T, d), -8, 8, 8.0, g, "cpu")
    w = W._grid_int((E, d), -8, 8, 64.0, g, "cpu")
    out = oracle.layer_forward(x, w, k=k, E=E, R=4, d_ff=0, act="identity", score="softmax",
                               renorm=True)
    if k == 1:
        assert torch.equal(out["y"], x.double())
    else:
        assert torch.allclose(out["y"], x.double(), rtol=0, atol=2 * k * 2 ** -23)


def test_layer_dropped_tokens_pass_through():
    """With a tight capacity and the residual added, every fully dropped token
    leaves the layer unchanged and its MoE part is exactly zero."""
    w = W.WORKLOADS["switch"].replace(T=512, d=64, E=8, R=2, d_ff=32, capacity_factor=0.5)
    inp = W.make_inputs(w)
    kw = dict(k=w.k, E=w.E, R=w.R, d_ff=w.d_ff, act=w.act, score=w.score, renorm=w.renorm,
              capacity_factor=w.capacity_factor, logit_bias=inp["logit_bias"], w_up=inp["w_up"],
              w_down=inp["w_down"])
    with_res = oracle.layer_forward(inp["x"], inp["w_router"], add_residual=True, **kw)
    no_res = oracle.layer_forward(inp["x"], inp["w_router"], add_residual=False, **kw)
    dropped = (with_res["slot_row"] < 0).all(1)
    assert dropped.sum() > 0 and (~dropped).sum() > 0
    assert torch.equal(with_res["y"][dropped], inp["x"][dropped].double())
    assert torch.equal(no_res["y"][dropped], torch.zeros_like(no_res["y"][dropped]))
    assert torch.allclose(with_res["y"] - no_res["y"], inp["x"].double(), atol=1e-12)


def test_layer_token_subset_equals_full():
    """Restricting compute/combine to a token subset changes nothing for those tokens."""
    w = W.WORKLOADS["deepseek"].replace(T=96, d=64, E=16, R=4, k=4, d_ff=32)
    inp = W.make_inputs(w)
    kw = dict(k=w.k, E=w.E, R=w.R, d_ff=w.d_ff, act=w.act, score=w.score, renorm=w.renorm,
              sel_bias=inp["sel_bias"], w_up=inp["w_up"], w_down=inp["w_down"],
              shared_up=inp["shared_up"], shared_down=inp["shared_down"])
    full = oracle.layer_forward(inp["x"], inp["w_router"], **kw)
    toks = [0, 5, 17, 95, 40]
    sub = oracle.layer_forward(inp["x"], inp["w_router"], tokens=toks, **kw)
    assert torch.equal(sub["y"], full["y"][toks])


def test_layer_matches_dense_mixture_definition():
    """Without drops or a shared expert, the layer equals the dense mixture
    sum_j g_j FFN_{e_j}(x), computed token by token with library matmuls (the
    special case where every pre-activation saturates GELU to the identity);
    the shared-expert term is pinned by the two tests below."""
    T, d, E, k, f = 12, 24, 4, 2, 20
    g = torch.Generator().manual_seed(8)
    x = 1 + torch.randint(0, 9, (T, d), generator=g).float() / 8
    wr = torch.randint(-8, 9, (E, d), generator=g).float() / 64
    w1 = 1 + torch.randint(0, 9, (E, f, d), generator=g).float() / 8
    w2 = torch.randint(-8, 9, (E, d, f), generator=g).float() / 8
    out = oracle.layer_forward(x, wr, k=k, E=E, R=2, d_ff=f, act="gelu", w_up=w1, w_down=w2)
    idx, gate = out["topk_idx"], out["topk_gate"]
    for t in range(T):
        ref = torch.zeros(d, dtype=torch.float64)
        for j in range(k):
            e = int(idx[t, j])
            ref += float(gate[t, j]) * ((x[t].double() @ w1[e].double().T) @ w2[e].double().T)
        assert torch.allclose(out["y"][t], ref, rtol=1e-13, atol=1e-9)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_layer_with_shared_expert_matches_dense_mixture_definition(act):
    """One always-on shared expert (the DeepSeek-V3-shaped layer): y = sum_j
    g_j FFN_{e_j}(x) + FFN_shared(x), token by token, from library matmuls.
    The shared term has gate 1, is evaluated on the token's own x (not on a
    row of the permuted buffer) and is added once.  Every pre-activation is
    >= 48, where GELU(v) = v and silu(v) = v exactly in fp64, so each FFN is
    plain matmuls (SwiGLU: the elementwise product of the gate and up
    projections); all values are dyadic, so the fp64 sums are exact."""
    T, d, E, k, f = 12, 24, 4, 2, 20
    up = 2 * f if act == "swiglu" else f
    g = torch.Generator().manual_seed(18)
    x = 2 + torch.randint(0, 9, (T, d), generator=g).float() / 8
    wr = torch.randint(-8, 9, (E, d), generator=g).float() / 64
    w1 = 1 + torch.randint(0, 9, (E, up, d), generator=g).float() / 8
    w2 = torch.randint(-8, 9, (E, d, f), generator=g).float() / 8
    s1 = 1 + torch.randint(0, 9, (1, up, d), generator=g).float() / 8
    s2 = torch.randint(-8, 9, (1, d, f), generator=g).float() / 8
    out = oracle.layer_forward(x, wr, k=k, E=E, R=2, d_ff=f, act=act, w_up=w1, w_down=w2,
                               shared_up=s1, shared_down=s2)
    idx, gate = out["topk_idx"], out["topk_gate"]
    assert (gate < 1).all()  # a shared term weighted by a routed gate would show

    def ffn(xt, wu, wd):
        pre = xt.double() @ wu.double().T
        h = pre[:f] * pre[f:] if act == "swiglu" else pre
        return h @ wd.double().T

    for t in range(T):
        ref = torch.zeros(d, dtype=torch.float64)
        for j in range(k):
            e = int(idx[t, j])
            ref += float(gate[t, j]) * ffn(x[t], w1[e], w2[e])
        ref += ffn(x[t], s1[0], s2[0])
        assert torch.allclose(out["y"][t], ref, rtol=1e-13, atol=0), t


def test_layer_shared_identity_expert_closed_form():
    """Identity experts plus a shared identity expert: y = (sum_j g_j + 1) x.
    Gates are full-softmax probabilities (no renormalisation), so sum_j g_j
    differs from 1 and from every single gate."""
    T, E, d, k = 40, 8, 16, 2
    g = W._gen(33, "cpu")
    x = W._grid_int((T, d), -8, 8, 8.0, g, "cpu")
    wr = W._grid_int((E, d), -8, 8, 16.0, g, "cpu")
    dummy = torch.zeros((1, 1, d))
    out = oracle.layer_forward(x, wr, k=k, E=E, R=4, d_ff=0, act="identity", score="softmax",
                               renorm=False, shared_up=dummy, shared_down=dummy)
    gsum = out["topk_gate"].double().sum(1, keepdim=True)
    assert (gsum < 0.99).any()
    ref = (gsum + 1) * x.double()
    assert torch.allclose(out["y"], ref, rtol=1e-14, atol=0)
    # the same tokens through the residual path instead of the shared expert
    res = oracle.layer_forward(x, wr, k=k, E=E, R=4, d_ff=0, act="identity", score="softmax",
                               renorm=False, add_residual=True)
    assert torch.allclose(res["y"], ref, rtol=1e-14, atol=0)


def test_switch_workload_drop_fraction_in_band():
    """The Switch-shaped workload's Zipf(1.1) logit skew drops 5-20% of tokens
    at capacity factor 1.25 (its stated target band)."""
    w = W.WORKLOADS["switch"]
    inp = W.make_inputs(w, ffn=False)
    idx, _ = oracle.route(inp["x"], inp["w_router"], w.k, w.score, w.renorm,
                          logit_bias=inp["logit_bias"])
    C = oracle.capacity(w.T, w.k, w.E, w.capacity_factor)
    d = oracle.dispatch(idx, w.E, w.R, C)
    frac = d["n_dropped"] / (w.T * w.k)
    assert 0.05 <= frac <= 0.20, frac


# --------------------------------------------------------------------------
# Bias-based balancing (Ultralytics "Load Balancing and Capacity", DeepSeek-V3)
# --------------------------------------------------------------------------

def _skewed_router(T=2048, E=16, k=2, d=64, seed=6):
    w = W.WORKLOADS["deepseek"].replace(T=T, d=d, E=E, R=4, k=k, d_ff=64, act="identity",
                                        n_shared=0, sel_skew=1.5, sel_bias_std=0.0)
    return w, W.make_inputs(w, ffn=False)


def test_balancing_step_direction():
    """One step lowers the bias of every expert above the even share, raises
    it for every expert below, and leaves exact-share experts alone."""
    counts = torch.tensor([5, 1, 2, 0, 2], dtype=torch.int32)   # T*k = 10, E = 5: share 2
    bias = torch.tensor([0.5, -0.25, 0.125, 0.0, 1.0])
    out = oracle.update_sel_bias(counts, bias, T=5, k=2, gamma=0.0625)
    assert out.tolist() == [0.4375, -0.1875, 0.125, 0.0625, 1.0]
    # the even share need not be an integer: T*k/E = 7/3
    out = oracle.update_sel_bias(torch.tensor([3, 2, 2], dtype=torch.int32),
                                 torch.zeros(3), T=7, k=1, gamma=0.5)
    assert out.tolist() == [-0.5, 0.5, 0.5]


def test_balancing_reduces_load_imbalance():
    """Iterating route -> count -> update on a skewed router evens out the
    load without touching the gates' scores (the purpose the pages state)."""
    w, inp = _skewed_router()
    bias = inp["sel_bias"].clone()
    T, k, E = w.T, w.k, w.E

    def spread(b):
        idx, _ = oracle.route(inp["x"], inp["w_router"], k, "sigmoid", True, None, b)
        c = oracle.dispatch(idx, E, w.R, -1)["expert_counts"].double()
        return c, float(c.max() / c.mean())

    c0, s0 = spread(bias)
    assert s0 > 1.6, s0
    for _ in range(60):
        c, _ = spread(bias)
        bias = oracle.update_sel_bias(c.int(), bias, T, k, gamma=2.0 ** -8)
    _, s1 = spread(bias)
    assert s1 < 1.25 and s1 < s0, (s0, s1)


# --------------------------------------------------------------------------
# Rank-limited routing (DeepSeek-V3: at most M devices per token)
# --------------------------------------------------------------------------

def _brute_rank_limited(key, k, R, M):
    """Sort ranks by (-best key, rank), keep the first M, then sort the
    surviving experts by (-key, expert): a different procedure from the
    oracle's rounds of selection."""
    T, E = key.shape
    per = E // R
    out = []
    for t in range(T):
        best = [max(float(key[t, e]) for e in range(r * per, (r + 1) * per)) for r in range(R)]
        ranks = sorted(range(R), key=lambda r: (-best[r], r))[:M]
        allowed = [e for e in range(E) if e // per in ranks]
        out.append(sorted(allowed, key=lambda e: (-float(key[t, e]), e))[:k])
    return torch.tensor(out, dtype=torch.int32)


@pytest.mark.parametrize("E,R,M,k,score", [(8, 4, 2, 2, "softmax"), (16, 4, 1, 3, "sigmoid"),
                                            (16, 8, 3, 4, "sigmoid"), (12, 3, 2, 5, "softmax"),
                                            (8, 8, 2, 2, "sigmoid")])
def test_rank_limited_routing_bruteforce(E, R, M, k, score):
    x, w = _tiny_router(16, E, 4, seed=40 + E + R + M)
    sel = (torch.tensor([((e * 7) % 3 - 1) / 4096.0 for e in range(E)], dtype=torch.float32)
           if score == "sigmoid" else None)
    idx, gate, L = oracle.route(x, w, k, score, True, None, sel, return_logits=True, R=R,
                                max_ranks=M)
    key = L if score == "softmax" else torch.sigmoid(L.double()).float() + (sel if sel is not None else 0)
    assert torch.equal(idx, _brute_rank_limited(key, k, R, M))
    per = E // R
    assert all(len(set((idx[t] // per).tolist())) <= M for t in range(idx.shape[0]))


def test_rank_limit_of_all_ranks_is_unlimited():
    w, inp = _skewed_router(T=256)
    a, ga = oracle.route(inp["x"], inp["w_router"], w.k, "sigmoid", True, None, inp["sel_bias"])
    b, gb = oracle.route(inp["x"], inp["w_router"], w.k, "sigmoid", True, None, inp["sel_bias"],
                         R=w.R, max_ranks=w.R)
    assert torch.equal(a, b) and torch.equal(ga, gb)


def test_rank_limit_rejects_too_few_experts():
    x, w = _tiny_router(4, 8, 4, seed=1)
    with pytest.raises(ValueError):
        oracle.route(x, w, 5, "softmax", True, R=4, max_ranks=2)   # 2 ranks x 2 experts < 5


# --------------------------------------------------------------------------
# Backward of the exchanges: adjoint identities and library autograd
# --------------------------------------------------------------------------

def _exchange_case(T=40, E=8, k=3, d=16, cap=9, seed=12):
    idx = W.random_topk(T, E, k, seed=seed, skew=1.2)
    disp = oracle.dispatch(idx, E, 2, cap)
    g = torch.Generator().manual_seed(seed)
    yp = torch.randn((disp["rows"], d), generator=g, dtype=torch.float64).float()
    dy = torch.randn((T, d), generator=g, dtype=torch.float64).float()
    gate = torch.rand((T, k), generator=g)
    return disp, yp, dy, gate


def test_combine_backward_is_the_adjoint_and_matches_autograd():
    disp, yp, dy, gate = _exchange_case()
    d_yp, d_gate = oracle.combine_backward(dy, yp, disp["slot_row"], gate)
    T = dy.shape[0]
    rows = torch.arange(disp["rows"], dtype=torch.int32)
    y = oracle.combine(torch.arange(T), yp, rows, disp["slot_row"], gate)
    # <combine(yp), dy> = <yp, d_yp>: the reverse exchange is the adjoint
    assert abs(float((y * dy.double()).sum()) - float((yp.double() * d_yp).sum())) < 1e-9
    # library autograd of the same sum (fp64)
    ypd = yp.double().clone().requires_grad_(True)
    gd = gate.double().clone().requires_grad_(True)
    sr = disp["slot_row"].long()
    kept = sr >= 0
    rows_used = ypd[sr.clamp(min=0)] * kept.unsqueeze(-1)          # [T,k,d]
    out = (gd.unsqueeze(-1) * rows_used).sum(1)
    (out * dy.double()).sum().backward()
    assert torch.allclose(d_yp, ypd.grad, rtol=1e-12, atol=1e-12)
    assert torch.allclose(d_gate, gd.grad * kept, rtol=1e-12, atol=1e-12)
    assert torch.all(d_gate[~kept] == 0)


def test_dispatch_backward_is_the_adjoint_of_permute():
    disp, yp, dy, gate = _exchange_case(T=33, k=2, cap=5)
    T, d = 33, 16
    x = torch.randn((T, d), generator=torch.Generator().manual_seed(3)).float()
    xp = oracle.permute(x, disp["slot_row"], disp["rows"])
    d_xp = torch.randn(xp.shape, generator=torch.Generator().manual_seed(4)).float()
    dx = oracle.dispatch_backward(d_xp, disp["slot_row"], T)
    assert abs(float((xp.double() * d_xp.double()).sum()) - float((x.double() * dx).sum())) < 1e-9
    # library autograd of a gather
    xd = x.double().clone().requires_grad_(True)
    (xd[disp["row_token"].long()] * d_xp.double()).sum().backward()
    assert torch.allclose(dx, xd.grad, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_expert_ffn_backward_matches_autograd(act):
    """Backward through one expert FFN against PyTorch autograd in fp64 (a
    library routine), input and weight gradients, non-square shapes."""
    g = torch.Generator().manual_seed(21)
    n, d, f = 7, 24, 40
    up_rows = 2 * f if act == "swiglu" else f
    x = torch.randn((n, d), generator=g)
    wu = torch.randn((up_rows, d), generator=g) * 0.3
    wd = torch.randn((d, f), generator=g) * 0.3
    dy = torch.randn((n, d), generator=g)
    d_in, dwu, dwd = oracle.expert_ffn_backward(x, wu, wd, dy, act, f)
    xd, wud, wdd = (t.double().clone().requires_grad_(True) for t in (x, wu, wd))
    pre = xd @ wud.T
    h = F.gelu(pre) if act == "gelu" else F.silu(pre[:, :f]) * pre[:, f:]
    ((h @ wdd.T) * dy.double()).sum().backward()
    assert torch.allclose(d_in, xd.grad, rtol=1e-10, atol=1e-12)
    assert torch.allclose(dwu, wud.grad, rtol=1e-10, atol=1e-12)
    assert torch.allclose(dwd, wdd.grad, rtol=1e-10, atol=1e-12)


# --------------------------------------------------------------------------
# Router backward: gradients through the gates (training the router)
# --------------------------------------------------------------------------

def _router_autograd(x, w, lb, idx, dg, score, renorm):
    """fp64 autograd of the forward gate definitions, with the selection fixed."""
    X = x.double().clone().requires_grad_(True)
    Wt = w.double().clone().requires_grad_(True)
    B = (lb.double() if lb is not None else torch.zeros(w.shape[0], dtype=torch.float64))
    B = B.clone().requires_grad_(True)
    L = X @ Wt.T + B
    L.retain_grad()
    ix = idx.long()
    Lc = L.gather(1, ix)
    if score == "softmax" and renorm:
        g = torch.softmax(Lc, dim=1)
    elif score == "softmax":
        g = torch.softmax(L, dim=1).gather(1, ix)
    elif renorm:
        s = torch.sigmoid(Lc)
        g = s / s.sum(1, keepdim=True)
    else:
        g = torch.sigmoid(Lc)
    (g * dg.double()).sum().backward()
    return L.grad, X.grad, Wt.grad, B.grad


@pytest.mark.parametrize("score,renorm", [("softmax", True), ("softmax", False),
                                          ("sigmoid", True), ("sigmoid", False)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_router_backward_matches_autograd(score, renorm, dtype):
    """The oracle's router backward equals fp64 autograd of the gate
    definitions on a fixed selection, for each gate form, with a logit bias;
    the selection-only bias (sigmoid) changes the selection but not the
    gradient formula."""
    T, d, E, k = 24, 32, 16, 3
    g = W._gen(41, "cpu")
    x = W._grid_int((T, d), -8, 8, 8.0, g, "cpu").to(dtype)
    w = W._grid_int((E, d), -8, 8, 64.0, g, "cpu").to(dtype)
    lb = W._grid_int((E,), -8, 8, 64.0, g, "cpu")
    sel = W._grid_int((E,), -8, 8, 256.0, g, "cpu") if score == "sigmoid" else None
    idx, _ = oracle.route(x, w, k, score, renorm, lb, sel)
    dg = torch.randn((T, k), generator=torch.Generator().manual_seed(5))
    dL, dx, dw, dlb = oracle.route_backward(x, w, idx, dg, score, renorm, lb)
    rL, rx, rw, rb = _router_autograd(x, w, lb, idx, dg, score, renorm)
    for got, ref in ((dL, rL), (dx, rx), (dw, rw), (dlb, rb)):
        assert torch.allclose(got, ref, rtol=1e-10, atol=1e-12)
    if score != "softmax" or renorm:
        # only the chosen experts' logits carry gradient
        mask = torch.zeros((T, E), dtype=torch.bool)
        mask.scatter_(1, idx.long(), True)
        assert torch.all(dL[~mask] == 0)
    if score == "softmax" and renorm:
        # renormalised softmax gates sum to 1 whatever the logits: the
        # gradient is orthogonal to a common shift of the chosen logits
        assert torch.allclose(dL.sum(1), torch.zeros(T, dtype=torch.float64), atol=1e-12)
