"""Helpers shared by the GPU parity tests: run one step of the CUDA library
through the C ABI, and compare with the oracle under the tolerances below.

Every output buffer these helpers hand to the library sits between guard
bands that are checked after the call (Guarded).

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


CANARY = 4096  # guard elements on each side of an output buffer


class Guarded:
    """An output tensor placed inside a larger buffer whose guard bands (CANARY
    elements before and after) hold a fixed bit pattern; check() asserts that
    no kernel wrote outside the tensor.  Stands in for a memory checker."""

    def __init__(self, shape, dtype, fill):
        n = 1
        for s_ in shape:
            n *= s_
        self.buf = torch.empty(n + 2 * CANARY, dtype=dtype, device=DEV)
        self.pattern = torch.full((CANARY,), -12345 if not dtype.is_floating_point else -1.5e4,
                                  dtype=dtype, device=DEV)
        self.buf[:CANARY] = self.pattern
        self.buf[CANARY + n:] = self.pattern
        self.t = self.buf[CANARY:CANARY + n].view(shape)
        self.t.fill_(fill)
        self.n = n

    def check(self, what=""):
        head = self.buf[:CANARY]
        tail = self.buf[CANARY + self.n:]
        assert torch.equal(head, self.pattern) and torch.equal(tail, self.pattern), \
            f"write outside the output buffer {what}"


def cfg_for(w, T=None, **kw):
    return moe.config_from_workload(w, T=T, **kw)


def run_route(cfg, inp):
    T, k = cfg.T, cfg.k
    idx = Guarded((T, k), torch.int32, -7)
    gate = Guarded((T, k), torch.float32, float("nan"))
    ws = moe.alloc_workspace(cfg)
    moe.moe_route(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), inp.get("sel_bias"),
                  idx.t, gate.t, ws)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(ws) == 0
    idx.check("topk_idx")
    gate.check("topk_gate")
    return idx.t.cpu(), gate.t.cpu()


def run_dispatch(cfg, x, topk_idx, rank_splits=True, ws=None):
    T, k, E, R = cfg.T, cfg.k, cfg.E, cfg.R
    rows = max(moe.moe_max_rows(cfg), 1)
    i32 = torch.int32
    g = dict(
        xp=Guarded((rows, cfg.d), x.dtype, 0),
        row_token=Guarded((rows,), i32, -5),
        slot_row=Guarded((T, k), i32, -9),
        expert_counts=Guarded((E,), i32, -1),
        expert_offsets=Guarded((E + 1,), i32, -1),
        rank_counts=Guarded((R,), i32, -1),
        rank_splits=Guarded((R, R), i32, -1) if rank_splits else None,
        n_dropped=Guarded((1,), i32, -1),
    )
    out = {key: (v.t if v is not None else None) for key, v in g.items()}
    ws = moe.alloc_workspace(cfg) if ws is None else ws
    moe.moe_dispatch(cfg, x, topk_idx.to(DEV), out["xp"], out["row_token"], out["slot_row"],
                     out["expert_counts"], out["expert_offsets"], out["rank_counts"],
                     out["rank_splits"], out["n_dropped"], ws)
    torch.cuda.synchronize()
    out["status"] = moe.moe_read_device_status(ws)
    for key, v in g.items():
        if v is not None:
            v.check(key)
    return out


def to_dev(inp):
    return {k: (v.to(DEV) if torch.is_tensor(v) else v) for k, v in inp.items()}
