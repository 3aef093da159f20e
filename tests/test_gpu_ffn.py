"""GPU parity of Step 3 (expert FFN, grouped GEMM) against the oracle:
ragged groups (empty, 1 row, tile edges, several tiles), GELU and SwiGLU,
the bf16 tensor-core path and the fp32 FFMA path, plus the shared expert."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import Guarded, DEV, assert_rows_close

pytestmark = pytest.mark.gpu


def _weights(E, rows_up, d, f, dtype, seed):
    g = W._gen(seed, "cpu")
    w_up = W._grid_normal((E, rows_up, d), 0.02 * 4, 2.0 ** -9, 0.125, g, "cpu").to(dtype)
    w_dn = W._grid_normal((E, d, f), 0.02 * 4, 2.0 ** -9, 0.125, g, "cpu").to(dtype)
    return w_up, w_dn


def _run_ffn(counts, d, f, act, dtype, seed, rows_cap=None, shared=False):
    E = len(counts)
    offs = torch.zeros(E + 1, dtype=torch.int32)
    offs[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32), 0)
    N = int(offs[-1])
    rows_cap = rows_cap or max(N, 1)
    T = max(N, 1)
    rows_up = 2 * f if act == "swiglu" else f
    w_up, w_dn = _weights(E, rows_up, d, f, dtype, seed)
    g = W._gen(seed + 1, "cpu")
    xp = W._grid_int((rows_cap, d), -8, 8, 8.0, g, "cpu").to(dtype)
    cfg = moe.make_config(T, d, E, 1, 1, f, 1 if shared else 0,
                          "bf16" if dtype == torch.bfloat16 else "f32", "softmax", True, 0.0,
                          0, act)
    hg = Guarded((rows_cap, f), dtype, 0)
    ypg = Guarded((rows_cap, d), dtype, 7.0)
    h, yp = hg.t, ypg.t
    ws = moe.alloc_workspace(cfg)
    sh_args = {}
    if shared:
        su, sd = _weights(1, rows_up, d, f, dtype, seed + 7)
        sx = xp[:T]
        sh_h = torch.empty((T, f), dtype=dtype, device=DEV)
        sh_out = torch.empty((T, d), dtype=dtype, device=DEV)
        sh_args = dict(shared_x=sx.to(DEV), shared_up=su.to(DEV), shared_down=sd.to(DEV),
                       shared_h=sh_h, shared_out=sh_out)
    moe.moe_expert_ffn(cfg, xp.to(DEV), offs.to(DEV), w_up.to(DEV), w_dn.to(DEV), h, yp, ws=ws,
                       **sh_args)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    hg.check("h")
    ypg.check("yp")
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-4
    worst = 0.0
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        ref = oracle.expert_ffn(xp[lo:hi], w_up[e], w_dn[e], act, f)
        worst = max(worst, assert_rows_close(yp[lo:hi], ref, tol))
    # rows past the last group are untouched
    if rows_cap > N:
        assert torch.all(yp[N:].float() == 7.0)
    if shared:
        ref = oracle.expert_ffn(xp[:T], su[0], sd[0], act, f)
        assert_rows_close(sh_args["shared_out"], ref, tol)
    return worst


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("counts,d,f", [
    ([128], 128, 128),
    ([1], 64, 64),
    ([0, 1, 127, 128, 129, 300, 0, 513], 256, 384),
    ([40, 0, 0, 250], 512, 1024),
    ([700, 3], 1024, 256),
    ([1500, 1100], 256, 256),
    ([2000, 0, 1], 128, 384),
    ([17, 33, 250, 5, 300, 1], 512, 512),
])
def test_ffn_bf16_tensor_cores(act, counts, d, f):
    _run_ffn(counts, d, f, act, torch.bfloat16, seed=sum(counts) + d + f)


def test_ffn_bf16_many_groups_and_spare_rows():
    counts = [int(c) for c in torch.randint(0, 40, (256,), generator=torch.Generator().manual_seed(2))]
    _run_ffn(counts, 128, 128, "swiglu", torch.bfloat16, seed=11, rows_cap=sum(counts) + 200)


def test_ffn_bf16_shared_expert():
    _run_ffn([100, 60, 0, 96], 256, 128, "swiglu", torch.bfloat16, seed=4, shared=True)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("counts,d,f", [([0, 1, 63, 64, 65, 200], 68, 36), ([1024, 1000], 512, 1024)])
def test_ffn_fp32(act, counts, d, f):
    _run_ffn(counts, d, f, act, torch.float32, seed=len(counts) + d)
