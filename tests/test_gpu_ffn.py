"""GPU parity of Step 3 (expert FFN, grouped GEMM) against the oracle:
ragged groups (empty, 1 row, tile edges, several tiles), GELU and SwiGLU,
the bf16 tensor-core path, the fp32 tensor-core path (three tf32 products per
fp32 product; d and d_ff multiples of 16) and the fp32 FFMA path (other fp32
shapes), plus the shared expert."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import Guarded, DEV, assert_rows_close

pytestmark = pytest.mark.gpu


# A positive value whose tf32 split is (v, v * 2^-12): v has at most 7
# significant bits (exact in tf32, and v (1 + 2^-12) exact in fp32) and
# v * 2^-12 is below half of v's tf32 spacing, so rn_tf32(v (1 + 2^-12)) = v
# and the remainder v * 2^-12 is exact.  With all
# operands of this form and positive, each cross term a_lo*b_hi and a_hi*b_lo
# carries 2^-12 (2.4e-4) of every product with the same sign: an fp32 GEMM
# that dropped either would miss the 1e-4 budget, while the term a_lo*b_lo
# that three tf32 products leave out is 2^-24.
def _lo_heavy(shape, step, top, g):
    v = torch.randint(1, top + 1, shape, generator=g, dtype=torch.int32).to(torch.float64) * step
    return (v * (1.0 + 2.0 ** -12)).to(torch.float32)


def _values(shape, kind, g, scale):
    if kind == "normal":  # arbitrary fp32: every operand has a non-zero low part
        return torch.randn(shape, generator=g, dtype=torch.float32) * scale
    # positive multiples of 1/8 (x) or of 2^-9 up to 2^-3 (weights)
    return _lo_heavy(shape, 0.125, 8, g) if scale == 1.0 else _lo_heavy(shape, 2.0 ** -9, 64, g)


def _weights(E, rows_up, d, f, dtype, seed, values="grid"):
    g = W._gen(seed, "cpu")
    if values != "grid":
        return _values((E, rows_up, d), values, g, 0.05), _values((E, d, f), values, g, 0.05)
    w_up = W._grid_normal((E, rows_up, d), 0.02 * 4, 2.0 ** -9, 0.125, g, "cpu").to(dtype)
    w_dn = W._grid_normal((E, d, f), 0.02 * 4, 2.0 ** -9, 0.125, g, "cpu").to(dtype)
    return w_up, w_dn


def _run_ffn(counts, d, f, act, dtype, seed, rows_cap=None, shared=False, values="grid"):
    E = len(counts)
    offs = torch.zeros(E + 1, dtype=torch.int32)
    offs[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32), 0)
    N = int(offs[-1])
    rows_cap = rows_cap or max(N, 1)
    T = max(N, 1)
    rows_up = 2 * f if act == "swiglu" else f
    w_up, w_dn = _weights(E, rows_up, d, f, dtype, seed, values)
    g = W._gen(seed + 1, "cpu")
    if values == "grid":
        xp = W._grid_int((rows_cap, d), -8, 8, 8.0, g, "cpu").to(dtype)
    else:
        xp = _values((rows_cap, d), values, g, 1.0)
    cfg = moe.make_config(T, d, E, 1, 1, f, 1 if shared else 0,
                          "bf16" if dtype == torch.bfloat16 else "f32", "softmax", True, 0.0,
                          0, act)
    hg = Guarded((rows_cap, f), dtype, 0)
    ypg = Guarded((rows_cap, d), dtype, 7.0)
    h, yp = hg.t, ypg.t
    ws = moe.alloc_workspace(cfg)
    sh_args = {}
    if shared:
        su, sd = _weights(1, rows_up, d, f, dtype, seed + 7, values)
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


# d = 68, f = 36 and d = 64, f = 36: FFMA path; the others: tensor cores (three
# tf32 products), d = 48, f = 80 with contraction lengths of 3 and 5 K stages
@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("counts,d,f", [
    ([0, 1, 63, 64, 65, 200], 68, 36),
    ([5, 130], 64, 36),
    ([0, 1, 63, 64, 65, 200], 48, 80),
    ([1024, 1000], 512, 1024),
    ([0, 1, 63, 64, 65, 127, 128, 129, 300], 128, 96),
    ([40, 0, 0, 250], 256, 416),
    ([700, 3], 96, 512),
])
def test_ffn_fp32(act, counts, d, f):
    _run_ffn(counts, d, f, act, torch.float32, seed=len(counts) + d)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("counts,d,f", [([1, 64, 65, 300, 0, 129], 128, 256), ([500], 512, 96)])
def test_ffn_fp32_tensor_cores_arbitrary_values(act, counts, d, f):
    """Normal fp32 operands (non-zero low parts everywhere): within 1e-4 of the
    fp64 oracle and, asserted, within 2e-5 (one tf32 product per fp32 product
    would be off by ~2^-11 of each product)."""
    worst = _run_ffn(counts, d, f, act, torch.float32, seed=3 + d, values="normal")
    assert worst < 2e-5, worst


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_ffn_fp32_tensor_cores_keep_both_cross_terms(act):
    """Operands whose low parts are 2^-12 of their high parts, all positive: a
    missing a_lo*b_hi or a_hi*b_lo pass would be off by 2.4e-4."""
    worst = _run_ffn([1, 63, 64, 200, 130], 128, 160, act, torch.float32, seed=5, values="lo_heavy")
    assert worst < 2e-5, worst


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_ffn_fp32_tensor_cores_smallest_shape_and_no_rows(act):
    """d = d_ff = 16 (one 16-column K stage, 16 of a tile's 256 columns stored)
    and a call whose experts received no rows."""
    _run_ffn([3, 0, 130], 16, 16, act, torch.float32, seed=21, values="normal")
    _run_ffn([0, 0], 64, 64, act, torch.float32, seed=22, rows_cap=40)


def test_ffn_fp32_tensor_cores_shared_expert_and_many_groups():
    counts = [int(c) for c in torch.randint(0, 40, (256,), generator=torch.Generator().manual_seed(9))]
    _run_ffn(counts, 64, 64, "swiglu", torch.float32, seed=12, rows_cap=sum(counts) + 70)
    _run_ffn([100, 60, 0, 96], 128, 64, "gelu", torch.float32, seed=13, shared=True, values="normal")
