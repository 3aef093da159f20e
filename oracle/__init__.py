"""CPU oracle for one mixture-of-experts layer forward pass.

TEST INFRASTRUCTURE ONLY.  This package is imported by ``tests/``,
``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` -- nothing else.  It shares no code with the CUDA library
(``expert_dispatch_top_b300``) and never touches a GPU.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 sums in index order,
built with ``-O2 -ffp-contract=off``; OpenMP over independent tokens only).
This module only marshals CPU tensors into that library and composes the four
steps of the Ultralytics glossary page "Expert Parallelism", section "How
Tokens Move Between GPUs": route, dispatch, compute, combine.

Pins: every function here is checked in ``tests/test_oracle_pins.py`` against
something other than itself (the routing snippet's printed loads, the
capacity example of the ai360xpert page, brute force, closed forms and
library special cases).  The pages print no whole-layer output: the layer's
composition is pinned against the dense-mixture definition computed with
library matmuls (with and without a shared expert, where the activations are
exactly the identity) and through the per-step pins.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_SO = os.path.join(_HERE, "_build", "libmoe_oracle.so")

F32, BF16 = 0, 1
SOFTMAX, SIGMOID = 0, 1
GELU, SWIGLU, IDENTITY = 0, 1, 2
_ACTS = {"gelu": GELU, "swiglu": SWIGLU, "identity": IDENTITY}
_SCORES = {"softmax": SOFTMAX, "sigmoid": SIGMOID}

_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/_build/libmoe_oracle.so (gcc)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_SO), exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
             "-shared", "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        i64, i32, vp, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_double
        lib.oracle_num_threads.restype = i32
        lib.oracle_sigmoid32.argtypes = [ctypes.c_float]
        lib.oracle_sigmoid32.restype = ctypes.c_float
        lib.oracle_route.argtypes = [i64, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, i32, i32,
                                     vp, vp, vp]
        lib.oracle_route.restype = i32
        lib.oracle_capacity.argtypes = [i64, i32, i32, dbl, i64]
        lib.oracle_capacity.restype = i64
        lib.oracle_dispatch.argtypes = [i64, i32, i32, i32, i64, vp, vp, vp, vp, vp, vp, vp, vp]
        lib.oracle_dispatch.restype = i64
        lib.oracle_permute.argtypes = [i64, i32, i64, vp, vp, vp]
        lib.oracle_permute.restype = None
        lib.oracle_expert_ffn.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp]
        lib.oracle_expert_ffn.restype = None
        lib.oracle_combine.argtypes = [i64, vp, i32, i32, vp, vp, vp, vp, vp, i32, vp, vp]
        lib.oracle_combine.restype = None
        lib.oracle_update_sel_bias.argtypes = [i64, i32, i32, vp, vp, ctypes.c_float]
        lib.oracle_update_sel_bias.restype = None
        lib.oracle_expert_ffn_backward.argtypes = [i64, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                                   vp]
        lib.oracle_route_backward.argtypes = [i64, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                              vp, vp, vp, vp]
        lib.oracle_route_backward.restype = None
        lib.oracle_expert_ffn_backward.restype = None
        lib.oracle_combine_backward.argtypes = [i64, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        lib.oracle_combine_backward.restype = None
        lib.oracle_dispatch_backward.argtypes = [i64, i32, i32, i32, vp, vp, vp]
        lib.oracle_dispatch_backward.restype = None
        _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle uses (the core count reported with timings)."""
    return int(_load().oracle_num_threads())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"oracle supports float32 and bfloat16 storage, got {t.dtype}")


def _cpu(t, dtype=None):
    if t is None:
        return None
    t = t.detach().to("cpu")
    if dtype is not None:
        t = t.to(dtype)
    return t.contiguous()


def sigmoid32(L: float) -> float:
    """fp32 sigmoid score: fp32(1 / (1 + exp(-L))) evaluated in double."""
    return float(_load().oracle_sigmoid32(ctypes.c_float(L)))


def route(x, w_router, k, score="softmax", renorm=True, logit_bias=None, sel_bias=None,
          return_logits=False, R=0, max_ranks=0):
    """Step 1 (Route).  Returns (topk_idx int32 [T,k], topk_gate fp32 [T,k][, logits fp32 [T,E]]).
    max_ranks > 0 limits every token to experts on at most that many of the R
    virtual ranks (contiguous blocks of E/R experts)."""
    x = _cpu(x)
    w = _cpu(w_router, x.dtype)
    T, d = x.shape
    E = w.shape[0]
    lb = _cpu(logit_bias, torch.float32)
    sb = _cpu(sel_bias, torch.float32)
    idx = torch.empty((T, k), dtype=torch.int32)
    gate = torch.empty((T, k), dtype=torch.float32)
    logits = torch.empty((T, E), dtype=torch.float32) if return_logits else None
    rc = _load().oracle_route(T, d, E, k, _dtype_code(x), _SCORES[score], int(bool(renorm)),
                              _ptr(x), _ptr(w), _ptr(lb), _ptr(sb), int(R), int(max_ranks),
                              _ptr(idx), _ptr(gate), _ptr(logits))
    if rc != 0:
        raise ValueError("oracle_route: unsupported arguments")
    return (idx, gate, logits) if return_logits else (idx, gate)


def capacity(T, k, E, capacity_factor=0.0, explicit=0) -> int:
    """Per-expert capacity: explicit, else ceil(cf*T*k/E), else -1 (no limit)."""
    return int(_load().oracle_capacity(T, k, E, float(capacity_factor), int(explicit)))


def dispatch(topk_idx, E, R, C):
    """Step 2 (Dispatch) metadata.  C < 0 means no capacity limit."""
    idx = _cpu(topk_idx, torch.int32)
    T, k = idx.shape
    out = {
        "expert_counts": torch.zeros(E, dtype=torch.int32),
        "expert_offsets": torch.zeros(E + 1, dtype=torch.int32),
        "rank_counts": torch.zeros(R, dtype=torch.int32),
        "rank_splits": torch.zeros((R, R), dtype=torch.int32),
        "slot_row": torch.empty((T, k), dtype=torch.int32),
        "row_token": torch.full((max(T * k, 1),), -1, dtype=torch.int32),
    }
    nd = ctypes.c_int64(0)
    rows = _load().oracle_dispatch(T, E, k, R, int(C), _ptr(idx), _ptr(out["expert_counts"]),
                                   _ptr(out["expert_offsets"]), _ptr(out["rank_counts"]),
                                   _ptr(out["rank_splits"]), _ptr(out["slot_row"]),
                                   _ptr(out["row_token"]), ctypes.byref(nd))
    if rows < 0:
        raise MemoryError("oracle_dispatch")
    out["row_token"] = out["row_token"][:rows].clone()
    out["n_dropped"] = int(nd.value)
    out["rows"] = int(rows)
    out["capacity"] = int(C)
    return out


def permute(x, slot_row, rows):
    """The dispatch permutation: xp[slot_row[t,j]] = x[t] (raw element copy)."""
    x = _cpu(x)
    sr = _cpu(slot_row, torch.int32)
    T, d = x.shape
    xp = torch.zeros((rows, d), dtype=x.dtype)
    _load().oracle_permute(T, sr.shape[1], d * x.element_size(), _ptr(x), _ptr(sr), _ptr(xp))
    return xp


def expert_ffn(rows, w_up, w_down, act, d_ff):
    """Step 3 (Compute) for one expert: fp64 output [n_rows, d]."""
    rows = _cpu(rows)
    n, d = rows.shape
    out = torch.empty((n, d), dtype=torch.float64)
    if n == 0:
        return out
    a = _ACTS[act] if isinstance(act, str) else int(act)
    wu = _cpu(w_up, rows.dtype) if a != IDENTITY else None
    wd = _cpu(w_down, rows.dtype) if a != IDENTITY else None
    _load().oracle_expert_ffn(n, d, int(d_ff), a, _dtype_code(rows), _ptr(rows), _ptr(wu),
                              _ptr(wd), _ptr(out))
    return out


def combine(tokens, yp_rows, row_map, slot_row, topk_gate, shared=None, resid=None):
    """Step 4 (Combine) for the listed tokens: fp64 [n_tok, d]."""
    toks = torch.as_tensor(tokens, dtype=torch.int64).contiguous()
    yp_rows = _cpu(yp_rows, torch.float64)
    row_map = _cpu(row_map, torch.int32)
    sr = _cpu(slot_row, torch.int32)
    g = _cpu(topk_gate, torch.float32)
    sh = _cpu(shared, torch.float64)
    rs = _cpu(resid)
    d = yp_rows.shape[1]
    k = sr.shape[1]
    y = torch.empty((toks.numel(), d), dtype=torch.float64)
    _load().oracle_combine(toks.numel(), _ptr(toks), d, k, _ptr(yp_rows), _ptr(row_map), _ptr(sr),
                           _ptr(g), _ptr(sh), _dtype_code(rs) if rs is not None else F32, _ptr(rs),
                           _ptr(y))
    return y


def update_sel_bias(expert_counts, sel_bias, T, k, gamma):
    """Bias-based balancing step: returns the updated fp32 selection bias."""
    counts = _cpu(expert_counts, torch.int32)
    out = _cpu(sel_bias, torch.float32).clone()
    _load().oracle_update_sel_bias(int(T), int(k), counts.numel(), _ptr(counts), _ptr(out),
                                   ctypes.c_float(gamma))
    return out


def expert_ffn_backward(rows, w_up, w_down, d_out, act, d_ff, weight_grads=True):
    """Backward through one expert FFN: (d_in fp64 [n,d], d_w_up fp64, d_w_down fp64)."""
    rows = _cpu(rows)
    n, d = rows.shape
    a = _ACTS[act] if isinstance(act, str) else int(act)
    up_rows = 2 * d_ff if a == SWIGLU else d_ff
    wu = _cpu(w_up, rows.dtype)
    wd = _cpu(w_down, rows.dtype)
    dy = _cpu(d_out, rows.dtype)
    d_in = torch.zeros((n, d), dtype=torch.float64)
    dwu = torch.zeros((up_rows, d), dtype=torch.float64) if weight_grads else None
    dwd = torch.zeros((d, d_ff), dtype=torch.float64) if weight_grads else None
    if n:
        _load().oracle_expert_ffn_backward(n, d, int(d_ff), a, _dtype_code(rows), _ptr(rows),
                                           _ptr(wu), _ptr(wd), _ptr(dy), _ptr(d_in), _ptr(dwu),
                                           _ptr(dwd))
    return d_in, dwu, dwd


def combine_backward(dy, yp, slot_row, topk_gate):
    """Backward of combine: (d_yp fp64 [rows,d] (zero where no slot points),
    d_gate fp64 [T,k])."""
    dy = _cpu(dy)
    yp = _cpu(yp, dy.dtype)
    sr = _cpu(slot_row, torch.int32)
    g = _cpu(topk_gate, torch.float32)
    T, d = dy.shape
    k = sr.shape[1]
    d_yp = torch.zeros((max(yp.shape[0], 1), d), dtype=torch.float64)
    d_gate = torch.zeros((T, k), dtype=torch.float64)
    _load().oracle_combine_backward(T, d, k, _dtype_code(dy), _ptr(dy), _ptr(yp), _ptr(sr), _ptr(g),
                                    _ptr(d_yp), _ptr(d_gate))
    return d_yp[: yp.shape[0]], d_gate


def dispatch_backward(d_xp, slot_row, T):
    """Backward of dispatch: dx fp64 [T,d] = sum of the kept rows' gradients."""
    d_xp = _cpu(d_xp)
    sr = _cpu(slot_row, torch.int32)
    d = d_xp.shape[1]
    dx = torch.empty((T, d), dtype=torch.float64)
    _load().oracle_dispatch_backward(T, d, sr.shape[1], _dtype_code(d_xp), _ptr(d_xp), _ptr(sr),
                                     _ptr(dx))
    return dx


def route_backward(x, w_router, topk_idx, d_gate, score="softmax", renorm=True, logit_bias=None):
    """Backward of the router through its gates: (d_logits fp64 [T,E], dx fp64 [T,d],
    dw fp64 [E,d], d_logit_bias fp64 [E]).  The selection itself carries no gradient."""
    x = _cpu(x)
    w = _cpu(w_router, x.dtype)
    T, d = x.shape
    E = w.shape[0]
    idx = _cpu(topk_idx, torch.int32)
    k = idx.shape[1]
    dg = _cpu(d_gate, torch.float32)
    lb = _cpu(logit_bias, torch.float32)
    dL = torch.zeros((T, E), dtype=torch.float64)
    dx = torch.zeros((T, d), dtype=torch.float64)
    dw = torch.zeros((E, d), dtype=torch.float64)
    dlb = torch.zeros(E, dtype=torch.float64)
    _load().oracle_route_backward(T, d, E, k, _dtype_code(x), _SCORES[score], int(bool(renorm)),
                                  _ptr(x), _ptr(w), _ptr(lb), _ptr(idx), _ptr(dg), _ptr(dL),
                                  _ptr(dx), _ptr(dw), _ptr(dlb))
    return dL, dx, dw, dlb


def layer_forward(x, w_router, *, k, E, R, d_ff, act, score="softmax", renorm=True,
                  capacity_factor=0.0, explicit_capacity=0, logit_bias=None, sel_bias=None,
                  w_up=None, w_down=None, shared_up=None, shared_down=None,
                  add_residual=False, tokens=None, max_ranks=0):
    """The four steps in the pages' order.  ``tokens`` restricts the expert
    compute and the combine to a subset of tokens (routing and dispatch always
    cover every token, since capacity decisions depend on all of them); each
    token's output depends only on its own rows, so the subset is exact.

    Returns a dict with the routing/dispatch metadata, ``y`` (fp64, one row per
    listed token) and ``tokens``.
    """
    x = _cpu(x)
    T, d = x.shape
    idx, gate = route(x, w_router, k, score, renorm, logit_bias, sel_bias, R=R,
                      max_ranks=max_ranks)
    C = capacity(T, k, E, capacity_factor, explicit_capacity)
    disp = dispatch(idx, E, R, C)
    toks = torch.arange(T, dtype=torch.int64) if tokens is None else \
        torch.as_tensor(tokens, dtype=torch.int64)
    sr = disp["slot_row"]
    # Rows the listed tokens use, grouped by expert (expert-major).
    used = sr[toks].flatten()
    used = torch.unique(used[used >= 0])
    row_map = torch.full((max(disp["rows"], 1),), -1, dtype=torch.int32)
    row_map[used.long()] = torch.arange(used.numel(), dtype=torch.int32)
    yp_rows = torch.zeros((max(used.numel(), 1), d), dtype=torch.float64)
    offs = disp["expert_offsets"]
    xp_used = x[disp["row_token"][used.long()].long()] if used.numel() else x[:0]
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        sel = ((used >= lo) & (used < hi)).nonzero().flatten()
        if sel.numel() == 0:
            continue
        wu = w_up[e] if w_up is not None else None
        wd = w_down[e] if w_down is not None else None
        yp_rows[sel] = expert_ffn(xp_used[sel], wu, wd, act, d_ff)
    shared = None
    if shared_up is not None and shared_down is not None and len(shared_up) > 0:
        shared = torch.zeros((toks.numel(), d), dtype=torch.float64)
        for s in range(len(shared_up)):
            shared += expert_ffn(x[toks], shared_up[s], shared_down[s], act, d_ff)
    y = combine(toks, yp_rows, row_map, sr, gate, shared, x if add_residual else None)
    out = dict(disp)
    out.update(topk_idx=idx, topk_gate=gate, y=y, tokens=toks)
    return out
