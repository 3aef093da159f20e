"""The range-checked debugging build (libmoe_b300_checked.so, MOE_CHECKED):
indices read from callers' buffers that are out of range are reported as
MOE_DEV_BOUNDS and the access is skipped, with no fault; clean inputs give
the release build's results and no report.  Each case runs in a child
process that loads the checked build and confirms it (moe_build_checked)
before it plants any bad index: the release build does not check."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import torch
import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_rows_close
assert moe.moe_build_checked(), "not the checked build: stop before planting bad indices"

# 1. a clean layer: no report, same routing and outputs as the oracle
w = W.WORKLOADS["deepseek"].replace(T=64, d=256, E=16, R=4, k=4, d_ff=128, add_residual=True)
inp = W.make_inputs(w)
dev = {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
cfg = moe.config_from_workload(w)
layer = moe.MoeLayer(cfg, dev["w_router"], dev["w_up"], dev["w_down"], dev["shared_up"],
                     dev["shared_down"], dev["logit_bias"], dev["sel_bias"])
y = layer(dev["x"]).clone()
torch.cuda.synchronize()
assert layer.device_status() == 0
ref = oracle.layer_forward(inp["x"], inp["w_router"], k=w.k, E=w.E, R=w.R, d_ff=w.d_ff, act=w.act,
                           score=w.score, renorm=w.renorm, sel_bias=inp["sel_bias"],
                           w_up=inp["w_up"], w_down=inp["w_down"], shared_up=inp["shared_up"],
                           shared_down=inp["shared_down"], add_residual=True)
assert torch.equal(layer.buf.slot_row.cpu(), ref["slot_row"])
assert_rows_close(y.cpu(), ref["y"], 2e-2)

# 2. combine with kept rows out of range: reported, counted as dropped
b = layer.buf
rows = moe.moe_max_rows(cfg)
bad = b.slot_row.clone()
bad[3, 0] = rows + 7
bad[9, 1] = -5
y2 = torch.empty_like(y)
moe.moe_combine(cfg, b.yp, bad, b.topk_gate, b.shared_out, dev["x"], y2)
assert layer.device_status() == moe.MOE_DEV_BOUNDS
fixed = bad.cpu().clone()
fixed[3, 0] = -1
fixed[9, 1] = -1
ref2 = oracle.combine(torch.arange(w.T), b.yp.cpu(), torch.arange(rows, dtype=torch.int32), fixed,
                      b.topk_gate.cpu(), b.shared_out.cpu().double(), inp["x"])
assert_rows_close(y2.cpu(), ref2, 2e-2)
# the same bad rows through the backward of combine and of dispatch
d_yp = torch.zeros_like(b.yp)
d_gate = torch.zeros_like(b.topk_gate)
moe.moe_combine_backward(cfg, y2, b.yp, bad, b.topk_gate, d_yp, d_gate)
assert layer.device_status() == moe.MOE_DEV_BOUNDS
assert float(d_gate[3, 0]) == 0.0 and float(d_gate[9, 1]) == 0.0
dx = torch.empty_like(y2)
moe.moe_dispatch_backward(cfg, d_yp, bad, dx)
assert layer.device_status() == moe.MOE_DEV_BOUNDS

# 3. expert FFN with expert_offsets that decrease and run past the rows
offs = b.expert_offsets.clone()
offs[5] = offs[4] - 3
offs[-1] = rows + 100
moe.moe_expert_ffn(cfg, b.xp, offs, dev["w_up"], dev["w_down"], b.h, b.yp, dev["x"],
                   dev["shared_up"], dev["shared_down"], b.shared_h, b.shared_out, b.ws)
torch.cuda.synchronize()
assert layer.device_status() == moe.MOE_DEV_BOUNDS
# ... and its backward
scratch = torch.empty(moe.moe_expert_ffn_backward_scratch_size(cfg, True), dtype=torch.uint8,
                      device=DEV)
moe.moe_expert_ffn_backward(cfg, b.xp, offs, dev["w_up"], dev["w_down"], b.yp, torch.empty_like(b.xp),
                            torch.empty_like(dev["w_up"]), torch.empty_like(dev["w_down"]), scratch,
                            b.ws)
torch.cuda.synchronize()
assert layer.device_status() == moe.MOE_DEV_BOUNDS
# 4. after all of that, a clean call on the same context is still right
y3 = layer(dev["x"]).clone()
torch.cuda.synchronize()
assert layer.device_status() == 0
assert torch.equal(y3, y)
print("checked build ok")
'''


def test_checked_build_reports_out_of_range_indices():
    env = dict(os.environ, MOE_B300_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True, env=env,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "checked build ok" in r.stdout
