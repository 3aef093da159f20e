"""Helpers shared by the GPU parity tests: run one step of the CUDA library
through the C ABI, and compare with the oracle under the tolerances below.

Tolerances:
  * indices, counts, offsets, rows, drop decisions, xp bytes: exact;
  * gates (fp32): |g - g_ref| <= (4 + n_terms) * 2^-23 * |g_ref|, n_terms = k
    (renormalised) or E (full softmax);
  * layer / FFN outputs, per token row: max|y - ref| <= tol * max|ref row|,
    tol = 2e-2 (bf16 experts) or 1e-4 (fp32); a row whose reference is all
    zeros must be exactly zero.
"""
from __future__ import annotations

import torch

import expert_dispatch_top_b300 as moe

DEV = "cuda"


def gate_tol(n_terms: int) -> float:
    return (4 + n_terms) * 2.0 ** -23


def assert_gates_close(got, ref, n_terms):
    got = got.double().cpu()
    ref = ref.double().cpu()
    err = (got - ref).abs()
    bound = gate_tol(n_terms) * ref.abs()
    bad = err > bound
    assert not bad.any(), f"{int(bad.sum())} gates off; worst {float((err - bound).max()):.3e}"


def assert_rows_close(got, ref, tol):
    """Per-row relative check against the row's max |ref|; zero rows exact."""
    got = got.double().cpu()
    ref = ref.double().cpu()
    rmax = ref.abs().amax(dim=1)
    err = (got - ref).abs().amax(dim=1)
    zero = rmax == 0
    assert torch.all(err[zero] == 0), "rows whose reference is zero must be exactly zero"
    nz = ~zero
    ratio = err[nz] / rmax[nz]
    assert ratio.numel() == 0 or float(ratio.max()) <= tol, \
        f"worst row error {float(ratio.max()):.3e} > {tol:.1e}"
    return float(ratio.max()) if ratio.numel() else 0.0


def cfg_for(w, T=None, **kw):
    return moe.config_from_workload(w, T=T, **kw)


def run_route(cfg, inp):
    T, k = cfg.T, cfg.k
    idx = torch.full((T, k), -7, dtype=torch.int32, device=DEV)
    gate = torch.full((T, k), float("nan"), dtype=torch.float32, device=DEV)
    ws = moe.alloc_workspace(cfg)
    moe.moe_route(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), inp.get("sel_bias"), idx,
                  gate, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    return idx.cpu(), gate.cpu()


def run_dispatch(cfg, x, topk_idx, rank_splits=True, ws=None):
    T, k, E, R = cfg.T, cfg.k, cfg.E, cfg.R
    rows = max(moe.moe_max_rows(cfg), 1)
    i32 = dict(dtype=torch.int32, device=DEV)
    out = dict(
        xp=torch.zeros((rows, cfg.d), dtype=x.dtype, device=DEV),
        row_token=torch.full((rows,), -5, **i32),
        slot_row=torch.full((T, k), -9, **i32),
        expert_counts=torch.full((E,), -1, **i32),
        expert_offsets=torch.full((E + 1,), -1, **i32),
        rank_counts=torch.full((R,), -1, **i32),
        rank_splits=torch.full((R, R), -1, **i32) if rank_splits else None,
        n_dropped=torch.full((1,), -1, **i32),
    )
    ws = moe.alloc_workspace(cfg) if ws is None else ws
    moe.moe_dispatch(cfg, x, topk_idx.to(DEV), out["xp"], out["row_token"], out["slot_row"],
                     out["expert_counts"], out["expert_offsets"], out["rank_counts"],
                     out["rank_splits"], out["n_dropped"], ws)
    torch.cuda.synchronize()
    out["status"] = moe.moe_read_device_status(ws)
    return out


def to_dev(inp):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
