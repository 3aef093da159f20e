"""GPU parity of the expert-FFN backward (moe_expert_ffn_backward) against the
oracle: input gradient d_xp and both weight gradients, GELU and SwiGLU, the
bf16 tensor-core path (including the K-grouped weight-gradient GEMM) and the
fp32 paths (input-gradient GEMMs on the tensor cores as three tf32 products
per product when d and d_ff are multiples of 16, else FFMA), over ragged
groups (empty, one row, tile edges, several tiles).

Tolerances.  d_xp: per row, relative to the row's max |ref| (as the forward
FFN test): bf16 2e-2 -- pre, dh and d_pre are each rounded to bf16 once
(2^-9 relative each) before the next contraction, and the result is rounded
once more; fp32 1e-4.  Weight gradients: max |err| over an expert's matrix
relative to that matrix's max |ref| (the scale one learning rate applies to),
same tol.  Per-row scaling does not fit them: with few rows a row of dW is
d_pre[:, m] times activations, and the relative error of one d_pre element is
unbounded where act' crosses zero (GELU' at a = -0.75, silu' at g = -1.28),
because pre is stored in bf16 before act' is taken.  Outputs whose reference
is exactly zero must be exactly zero."""
import pytest
import torch

import expert_dispatch_top_b300 as moe
import moe_workloads as W
import oracle
from gpu_util import DEV, assert_rows_close

pytestmark = pytest.mark.gpu


def assert_matrix_close(got, ref, tol):
    got = got.double().cpu()
    ref = ref.double().cpu()
    scale = float(ref.abs().max()) if ref.numel() else 0.0
    err = (got - ref).abs()
    if scale == 0.0:
        assert torch.all(err == 0), "a zero weight gradient must be exactly zero"
        return 0.0
    worst = float(err.max()) / scale
    assert worst <= tol, f"worst matrix error {worst:.3e} > {tol:.1e}"
    return worst


def _offsets(counts):
    offs = torch.zeros(len(counts) + 1, dtype=torch.int32)
    offs[1:] = torch.cumsum(torch.tensor(counts, dtype=torch.int32), 0)
    return offs


def _inputs(counts, d, f, act, dtype, seed, sparse_rows=None, normal=False):
    E = len(counts)
    offs = _offsets(counts)
    N = int(offs[-1])
    rows_up = 2 * f if act == "swiglu" else f
    g = W._gen(seed, "cpu")
    if normal:  # arbitrary fp32 values: every operand has a non-zero tf32 low part
        w_up = torch.randn((E, rows_up, d), generator=g) * 0.08
        w_dn = torch.randn((E, d, f), generator=g) * 0.08
        xp = torch.randn((max(N, 1), d), generator=g)
        d_yp = torch.randn((max(N, 1), d), generator=g) * 0.5
    else:
        w_up = W._grid_normal((E, rows_up, d), 0.08, 2.0 ** -9, 0.125, g, "cpu").to(dtype)
        w_dn = W._grid_normal((E, d, f), 0.08, 2.0 ** -9, 0.125, g, "cpu").to(dtype)
        xp = W._grid_int((max(N, 1), d), -8, 8, 8.0, g, "cpu").to(dtype)
        d_yp = W._grid_normal((max(N, 1), d), 0.5, 2.0 ** -9, 4.0, g, "cpu").to(dtype)
    if sparse_rows is not None:
        keep = torch.zeros(max(N, 1), dtype=torch.bool)
        keep[sparse_rows] = True
        d_yp[~keep] = 0
    cfg = moe.make_config(max(N, 1), d, E, 1, 1, f, 0,
                          "bf16" if dtype == torch.bfloat16 else "f32", "softmax", True, 0.0, 0,
                          act)
    return cfg, offs, w_up, w_dn, xp, d_yp


def _run(cfg, offs, w_up, w_dn, xp, d_yp, weight_grads=True):
    E = offs.numel() - 1
    dtype = xp.dtype
    rows = xp.shape[0]
    d_xp = torch.full((rows, xp.shape[1]), 5.0, dtype=dtype, device=DEV)
    d_wu = torch.full(tuple(w_up.shape), 9.0, dtype=dtype, device=DEV) if weight_grads else None
    d_wd = torch.full(tuple(w_dn.shape), 9.0, dtype=dtype, device=DEV) if weight_grads else None
    nbytes = moe.moe_expert_ffn_backward_scratch_size(cfg, weight_grads)
    assert nbytes > 0
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    ws = moe.alloc_workspace(cfg)
    moe.moe_expert_ffn_backward(cfg, xp.to(DEV), offs.to(DEV), w_up.to(DEV), w_dn.to(DEV),
                                d_yp.to(DEV), d_xp, d_wu, d_wd, scratch, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    assert E == w_up.shape[0]
    return d_xp, d_wu, d_wd


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("counts,d,f", [
    ([128], 128, 128),
    ([1], 64, 64),
    ([0, 1, 63, 64, 65, 300, 0, 513], 256, 384),
    ([40, 0, 0, 250], 512, 1024),
    ([700, 3], 1024, 256),
    ([17, 33, 250, 5, 300, 1], 512, 512),
])
def test_ffn_backward(dtype, act, counts, d, f):
    cfg, offs, w_up, w_dn, xp, d_yp = _inputs(counts, d, f, act, dtype, seed=sum(counts) + d + f)
    d_xp, d_wu, d_wd = _run(cfg, offs, w_up, w_dn, xp, d_yp)
    tol = 2e-2 if dtype == torch.bfloat16 else 1e-4
    for e in range(len(counts)):
        lo, hi = int(offs[e]), int(offs[e + 1])
        ref_in, ref_wu, ref_wd = oracle.expert_ffn_backward(xp[lo:hi], w_up[e], w_dn[e],
                                                            d_yp[lo:hi], act, f)
        if hi > lo:
            assert_rows_close(d_xp[lo:hi], ref_in, tol)
        # an expert with no rows has exactly zero weight gradients
        assert_matrix_close(d_wu[e], ref_wu, tol)
        assert_matrix_close(d_wd[e], ref_wd, tol)
    n = int(offs[-1])
    if d_xp.shape[0] > n:
        assert torch.all(d_xp[n:].float().cpu() == 5.0)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
@pytest.mark.parametrize("counts,d,f,normal", [
    ([0, 1, 63, 64, 65, 200], 68, 36, False),   # FFMA (d, d_ff not multiples of 16)
    ([1, 64, 65, 300, 0, 129], 128, 96, True),  # tensor cores, non-dyadic operands
    ([40, 0, 250], 48, 80, True),
])
def test_ffn_backward_fp32_paths(act, counts, d, f, normal):
    cfg, offs, w_up, w_dn, xp, d_yp = _inputs(counts, d, f, act, torch.float32, seed=d + f,
                                              normal=normal)
    d_xp, d_wu, d_wd = _run(cfg, offs, w_up, w_dn, xp, d_yp)
    for e in range(len(counts)):
        lo, hi = int(offs[e]), int(offs[e + 1])
        ref_in, ref_wu, ref_wd = oracle.expert_ffn_backward(xp[lo:hi], w_up[e], w_dn[e],
                                                            d_yp[lo:hi], act, f)
        if hi > lo:
            assert_rows_close(d_xp[lo:hi], ref_in, 1e-4)
        assert_matrix_close(d_wu[e], ref_wu, 1e-4)
        assert_matrix_close(d_wd[e], ref_wd, 1e-4)


@pytest.mark.parametrize("act", ["gelu", "swiglu"])
def test_ffn_backward_input_grad_only(act):
    counts, d, f = [300, 0, 77, 129], 256, 256
    cfg, offs, w_up, w_dn, xp, d_yp = _inputs(counts, d, f, act, torch.bfloat16, seed=11)
    assert (moe.moe_expert_ffn_backward_scratch_size(cfg, False) <
            moe.moe_expert_ffn_backward_scratch_size(cfg, True))
    d_xp, _, _ = _run(cfg, offs, w_up, w_dn, xp, d_yp, weight_grads=False)
    for e in range(len(counts)):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            ref, _, _ = oracle.expert_ffn_backward(xp[lo:hi], w_up[e], w_dn[e], d_yp[lo:hi], act,
                                                   f, weight_grads=False)
            assert_rows_close(d_xp[lo:hi], ref, 2e-2)


@pytest.mark.parametrize("shape", ["mixtral", "deepseek"])
def test_ffn_backward_layer_sized(shape):
    """Full layer widths: Mixtral-8x7B-shaped experts (8 x SwiGLU 4096 -> 14336)
    over 4096 rows and DeepSeek-V3-shaped experts (d = 7168, d_ff = 2048) on 32
    ragged groups.  d_yp is zero except on a few sampled rows per expert, so
    every other row's d_xp is exactly zero and the weight gradients are sums
    over the sampled rows alone, which the oracle computes; the GPU still runs
    every GEMM over all rows."""
    if shape == "mixtral":
        counts, d, f = [700, 380, 510, 640, 300, 520, 449, 597], 4096, 14336
    else:
        g = torch.Generator().manual_seed(5)
        counts = [int(c) for c in torch.randint(0, 160, (32,), generator=g)]
        counts[3] = 0
        d, f = 7168, 2048
    offs = _offsets(counts)
    g = torch.Generator().manual_seed(17)
    sample = []
    for e in range(len(counts)):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi > lo:
            pick = torch.randperm(hi - lo, generator=g)[:3] + lo
            sample += sorted(int(r) for r in pick)
    cfg, offs, w_up, w_dn, xp, d_yp = _inputs(counts, d, f, "swiglu", torch.bfloat16, seed=23,
                                              sparse_rows=sample)
    d_xp, d_wu, d_wd = _run(cfg, offs, w_up, w_dn, xp, d_yp)
    samp = torch.tensor(sample, dtype=torch.long)
    others = torch.ones(d_xp.shape[0], dtype=torch.bool)
    others[samp] = False
    assert torch.all(d_xp[others.to(DEV)] == 0)
    gw = torch.Generator().manual_seed(29)
    # weight gradients of a few experts (each oracle call forms a whole dW in fp64),
    # an empty one among them for the DeepSeek shape
    wg_experts = {0, 5} if shape == "mixtral" else {0, 3, 17, 30}
    for e in range(len(counts)):
        lo, hi = int(offs[e]), int(offs[e + 1])
        rows = samp[(samp >= lo) & (samp < hi)]
        ref_in, ref_wu, ref_wd = oracle.expert_ffn_backward(xp[rows], w_up[e], w_dn[e], d_yp[rows],
                                                            "swiglu", f,
                                                            weight_grads=e in wg_experts)
        if rows.numel():
            assert_rows_close(d_xp[rows.to(DEV)], ref_in, 2e-2)
        if e not in wg_experts:
            continue
        # weight-gradient rows checked on a sample (the full matrices are large),
        # against the whole matrix's scale
        ru = torch.randperm(ref_wu.shape[0], generator=gw)[:96]
        rd = torch.randperm(ref_wd.shape[0], generator=gw)[:96]
        su, sd = float(ref_wu.abs().max()), float(ref_wd.abs().max())
        for got, ref, sc in ((d_wu[e][ru.to(DEV)], ref_wu[ru], su),
                             (d_wd[e][rd.to(DEV)], ref_wd[rd], sd)):
            err = (got.double().cpu() - ref).abs()
            assert float(err.max()) <= 2e-2 * sc if sc else torch.all(err == 0)
