"""The whole layer enqueues only device work on the caller's stream (no host
synchronisation inside the calls), so it can be captured into a CUDA graph:
capture once, replay on new inputs written into the same buffers, and match
eager execution bit for bit."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
from gpu_util import DEV

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,T", [("deepseek", 512), ("switch", 4096), ("toy", 1024)])
def test_layer_forward_graph_replay_matches_eager(name, T):
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device=DEV, T=T)
    cfg = moe.config_from_workload(w, T=T, add_residual=True)
    layer = moe.MoeLayer(cfg, inp["w_router"], inp.get("w_up"), inp.get("w_down"),
                         inp.get("shared_up"), inp.get("shared_down"), inp.get("logit_bias"),
                         inp.get("sel_bias"))
    x = inp["x"].clone()
    layer(x)                                   # eager warm-up (one-time host set-up)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            y_graph = layer(x)
    torch.cuda.current_stream().wait_stream(s)
    for seed in (11, 12):
        new_x = W._grid_int(tuple(x.shape), -8, 8, 8.0, W._gen(seed, DEV), DEV).to(x.dtype)
        x.copy_(new_x)
        graph.replay()
        torch.cuda.synchronize()
        got = y_graph.clone()
        eager = layer(x).clone()
        torch.cuda.synchronize()
        assert torch.equal(got, eager)
        assert layer.device_status() == 0
