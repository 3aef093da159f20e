"""GPU parity of the bias-based balancing update (moe_update_sel_bias) with the
oracle, one step and a 30-step route -> dispatch -> update loop run entirely
on the device."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, run_dispatch, run_route, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("E,T,k", [(5, 5, 2), (256, 8192, 8), (64, 3001, 3)])
def test_update_one_step(E, T, k):
    g = torch.Generator().manual_seed(E)
    counts = torch.randint(0, 2 * T * k // E + 2, (E,), generator=g, dtype=torch.int32)
    bias = torch.round(torch.randn(E, generator=g) * 4096) / 4096
    cfg = moe.make_config(T, 64, E, k, 1, 0, 0, "bf16", "sigmoid", True, 0.0, 0, "identity")
    b_dev = bias.to(DEV)
    moe.moe_update_sel_bias(cfg, counts.to(DEV), b_dev, 2.0 ** -10)
    torch.cuda.synchronize()
    ref = oracle.update_sel_bias(counts, bias, T, k, 2.0 ** -10)
    assert torch.equal(b_dev.cpu(), ref)


def test_balancing_loop_on_device_matches_oracle():
    w = W.WORKLOADS["deepseek"].replace(T=2048, d=256, E=32, R=4, k=4, d_ff=64, act="identity",
                                        n_shared=0, sel_skew=1.5, sel_bias_std=0.0)
    inp = W.make_inputs(w, ffn=False)
    cfg = moe.config_from_workload(w)
    dev = to_dev(inp)
    bias_dev = dev["sel_bias"].clone()
    bias_ref = inp["sel_bias"].clone()
    gamma = 2.0 ** -8
    first = last = None
    for step in range(30):
        idx, _ = run_route(cfg, dict(dev, sel_bias=bias_dev))
        out = run_dispatch(cfg, dev["x"], idx)
        moe.moe_update_sel_bias(cfg, out["expert_counts"], bias_dev, gamma)
        ridx, _ = oracle.route(inp["x"], inp["w_router"], w.k, "sigmoid", True, None, bias_ref)
        assert torch.equal(idx, ridx), step
        rc = oracle.dispatch(ridx, w.E, w.R, -1)["expert_counts"]
        assert torch.equal(out["expert_counts"].cpu(), rc)
        bias_ref = oracle.update_sel_bias(rc, bias_ref, w.T, w.k, gamma)
        torch.cuda.synchronize()
        assert torch.equal(bias_dev.cpu(), bias_ref), step
        spread = float(rc.max()) / (w.T * w.k / w.E)
        first = spread if first is None else first
        last = spread
    assert last < first
