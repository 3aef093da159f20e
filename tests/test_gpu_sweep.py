"""The dispatch/combine bandwidth sweep at its full sizes (d=7168, E=256,
top-8, identity experts, T up to 131072, Zipf skews 0..1.5), through the same
MoeLayer call bench.py times.  Routing is checked bit for bit against the
oracle on a seeded sample of tokens; dispatch through properties that hold at
any size (counts, offsets, a valid permutation in token order, the bytes of
every row); combine through its closed form for identity experts,
y[t] = bf16(sum_j g[t,j] * x[t]), within the bf16 tolerance."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_gates_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,s", [(4096, 0.0), (16384, 0.5), (16384, 1.0), (32768, 1.5),
                                 (131072, 0.0), (131072, 1.5)])
def test_sweep_point_full_size(T, s):
    w = W.sweep(T, s)
    inp = W.make_inputs(w, device=DEV)
    cfg = moe.config_from_workload(w)
    layer = moe.MoeLayer(cfg, inp["w_router"], None, None, None, None, None, inp["sel_bias"])
    y = layer(inp["x"])
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    b = layer.buf
    k, E, R = w.k, w.E, w.R
    # routing: a seeded sample of tokens, bit for bit
    samp = torch.randperm(T, generator=torch.Generator().manual_seed(T))[:192]
    samp = torch.unique(torch.cat([samp, torch.tensor([0, T - 1])]))
    x_s = inp["x"][samp.to(DEV)].cpu()
    ridx, rgate = oracle.route(x_s, inp["w_router"].cpu(), k, w.score, w.renorm, None,
                               inp["sel_bias"].cpu())
    idx = b.topk_idx.cpu()
    assert torch.equal(idx[samp], ridx)
    assert_gates_close(b.topk_gate.cpu()[samp], rgate, k)
    # dispatch properties (no capacity: nothing dropped)
    counts = torch.bincount(idx.flatten().long(), minlength=E)
    assert torch.equal(b.expert_counts.cpu().long(), counts)
    offs = b.expert_offsets.cpu().long()
    assert torch.equal(offs, torch.cat([torch.zeros(1, dtype=torch.long), counts.cumsum(0)]))
    assert int(b.n_dropped.item()) == 0
    sr = b.slot_row.long()
    rows = T * k
    assert bool((sr >= 0).all())
    seen = torch.zeros(rows, dtype=torch.int32, device=DEV)
    seen.index_add_(0, sr.flatten(), torch.ones(rows, dtype=torch.int32, device=DEV))
    assert bool((seen == 1).all())                                    # a permutation
    rt = b.row_token[:rows].long()
    tok = torch.arange(T, device=DEV).unsqueeze(1).expand(T, k)
    assert torch.equal(rt[sr.flatten()], tok.flatten())               # row -> its token
    exp_of_row = torch.repeat_interleave(torch.arange(E, device=DEV), counts.to(DEV))
    assert torch.equal(exp_of_row[sr.flatten()], idx.to(DEV).long().flatten())
    same = exp_of_row[1:] == exp_of_row[:-1]
    assert bool((rt[1:][same] > rt[:-1][same]).all())                 # token order per expert
    assert torch.equal(b.xp[:rows], inp["x"][rt])                     # bytes of every row
    per = E // R
    rc = counts.view(R, per).sum(1)
    assert torch.equal(b.rank_counts.cpu().long(), rc)
    src = (torch.arange(T) // ((T + R - 1) // R)).unsqueeze(1).expand(T, k).flatten()
    splits = torch.zeros((R, R), dtype=torch.long)
    splits.index_put_((src, idx.flatten().long() // per), torch.ones(T * k, dtype=torch.long),
                      accumulate=True)
    assert torch.equal(b.rank_splits.cpu().long(), splits)
    # combine for identity experts
    gsum = b.topk_gate.sum(1, keepdim=True)
    ref = inp["x"].float() * gsum
    err = (y.float() - ref).abs().amax(1)
    bound = 2.0 ** -7 * ref.abs().amax(1) + 1e-6
    assert bool((err <= bound).all())
