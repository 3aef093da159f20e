"""Seeded synthetic inputs for the MoE-layer workloads.

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic (no routing, counting, permutation, FFN or combine).  Both
the oracle-side tests and the CUDA-side tests/bench take their inputs from
here, so the two sides see bit-identical tensors.

All values lie on a dyadic grid so that router logits are exact in fp32
whatever the summation order:

* hidden states x: integers in [-8, 8] divided by 8;
* "uniform64" weights (the toy layer): integers in [-8, 8] divided by 64,
  i.e. multiples of 1/8 in [-1, 1] scaled by 1/8;
* "normal512" weights (all larger layers): N(0, 0.02) rounded to multiples of
  2**-9 and clamped to +-1/8 (at most 7 significant bits: exact in bf16);
* selection bias (DeepSeek-V3-style routers): N(0, 0.1) rounded to multiples
  of 2**-12;
* Zipf-shaped skew: for a seeded permutation rho of the experts, expert e
  gets -beta * s * ln(rho(e) + 1), rounded to a multiple of 2**-12.

Every product x*w is a multiple of 2**-12 and every partial sum of a logit is
bounded by d/8 <= 896 < 2**10, so 22 bits hold it exactly in fp32.

Workload shapes follow the pages' examples: the Ultralytics routing snippet
(8 experts, 4 GPUs, top-2, 4096 x 512), a Mixtral-8x7B-shaped layer, a
Switch-style top-1 layer with a capacity factor of 1.25, a DeepSeek-V3-shaped
layer (256 routed experts, top-8, 8 ranks, one shared expert) and a
dispatch/combine bandwidth sweep with identity experts.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass
from typing import Optional

import torch

SKEW_BETA = 0.06  # strength of the Zipf-shaped per-expert skew


@dataclass(frozen=True)
class Workload:
    name: str
    T: int          # tokens
    d: int          # d_model
    E: int          # routed experts
    R: int          # virtual expert-parallel ranks
    k: int          # experts per token
    d_ff: int       # expert hidden size
    act: str        # "gelu" | "swiglu" | "identity"
    dtype: str      # "f32" | "bf16" (activations and weights)
    score: str      # "softmax" | "sigmoid"
    renorm: bool    # gates renormalised over the chosen k
    capacity_factor: float  # <= 0: no capacity limit
    n_shared: int   # always-on shared experts
    seed: int
    weights: str    # "uniform64" | "normal512"
    logit_skew: float = 0.0    # Zipf exponent of a per-expert logit bias (0: none)
    sel_bias_std: float = 0.0  # std of the selection-only bias (0: none)
    sel_skew: float = 0.0      # Zipf exponent added to the selection-only bias
    add_residual: bool = False
    max_ranks: int = 0         # rank-limited routing: at most this many ranks per token (0: none)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def up_rows(self) -> int:
        return 2 * self.d_ff if self.act == "swiglu" else self.d_ff

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    # Ultralytics routing snippet scale: 4096 x 512, 8 experts on 4 ranks, top-2.
    "toy": Workload("toy", 4096, 512, 8, 4, 2, 1024, "gelu", "f32", "softmax", True, 0.0, 0, 0,
                    "uniform64"),
    # Mixtral-8x7B-shaped: 8 experts top-2, SwiGLU 4096 -> 14336.
    "mixtral": Workload("mixtral", 16384, 4096, 8, 8, 2, 14336, "swiglu", "bf16", "softmax", True,
                        0.0, 0, 1, "normal512"),
    # Switch-style top-1, capacity factor 1.25, Zipf(1.1)-skewed logits, gate = probability.
    "switch": Workload("switch", 32768, 1024, 64, 8, 1, 4096, "gelu", "bf16", "softmax", False,
                       1.25, 0, 2, "normal512", logit_skew=1.1),
    # DeepSeek-V3-shaped: 256 experts top-8, sigmoid + selection-only bias, 1 shared expert.
    "deepseek": Workload("deepseek", 8192, 7168, 256, 8, 8, 2048, "swiglu", "bf16", "sigmoid",
                         True, 0.0, 1, 3, "normal512", sel_bias_std=0.1),
}


def sweep(T: int, s: float) -> Workload:
    """Dispatch/combine bandwidth sweep point: identity experts, DeepSeek-style
    routing with an extra Zipf(s) selection skew (s=0: random-router spread)."""
    return Workload(f"sweep_T{T}_s{s:g}", T, 7168, 256, 8, 8, 0, "identity", "bf16", "sigmoid",
                    True, 0.0, 0, 4, "normal512", sel_bias_std=0.1, sel_skew=s)


SWEEP_T = [4096 * 2 ** i for i in range(6)]
SWEEP_S = [0.0, 0.5, 1.0, 1.5]


def get(name: str) -> Workload:
    if name.startswith("sweep"):
        # sweep_T<T>_s<s>
        parts = dict(p[0:1] and (p[0], p[1:]) for p in name.split("_")[1:])
        return sweep(int(parts["T"]), float(parts["s"]))
    return WORKLOADS[name]


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _grid_int(shape, lo, hi, denom, g, device):
    v = torch.randint(lo, hi + 1, shape, generator=g, device=device, dtype=torch.int32)
    return v.to(torch.float32) / denom


def _grid_normal(shape, std, step, clamp, g, device, chunk=1 << 26):
    out = torch.empty(shape, dtype=torch.float32, device=device)
    flat = out.view(-1)
    lim = clamp / step
    for s in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - s)
        v = torch.randn((n,), generator=g, device=device, dtype=torch.float32)
        flat[s:s + n] = torch.round(v * (std / step)).clamp_(-lim, lim) * step
    return out


def _weights(w: Workload, shape, g, device):
    if w.weights == "uniform64":
        return _grid_int(shape, -8, 8, 64.0, g, device)
    return _grid_normal(shape, 0.02, 2.0 ** -9, 0.125, g, device)


def _zipf_skew(E, s, g, device):
    rho = torch.randperm(E, generator=g, device=device).to(torch.float64)
    v = -SKEW_BETA * s * torch.log(rho + 1.0)
    return (torch.round(v * 4096.0) / 4096.0).to(torch.float32)


def make_inputs(w: Workload, device="cpu", ffn: bool = True, T: Optional[int] = None) -> dict:
    """Draw every input of workload ``w`` (optionally with a different T).

    Returns a dict: x [T,d], w_router [E,d] (activation dtype), logit_bias [E]
    fp32 or None, sel_bias [E] fp32 or None, and when ``ffn`` and the experts
    are not identity: w_up [E, up_rows, d], w_down [E, d, d_ff], shared_up
    [n_shared, up_rows, d], shared_down [n_shared, d, d_ff].  Draw order is
    fixed: x, router, biases, expert weights, shared weights.
    """
    T = w.T if T is None else T
    g = _gen(w.seed, device)
    dt = w.torch_dtype
    out = {}
    out["x"] = _grid_int((T, w.d), -8, 8, 8.0, g, device).to(dt)
    out["w_router"] = _weights(w, (w.E, w.d), g, device).to(dt)
    out["logit_bias"] = _zipf_skew(w.E, w.logit_skew, g, device) if w.logit_skew else None
    sb = None
    if w.sel_bias_std > 0:
        v = torch.randn((w.E,), generator=g, device=device, dtype=torch.float32) * w.sel_bias_std
        sb = torch.round(v * 4096.0) / 4096.0
    if w.sel_skew:
        sk = _zipf_skew(w.E, w.sel_skew, g, device)
        sb = sk if sb is None else sb + sk
    out["sel_bias"] = sb
    if ffn and w.act != "identity":
        out["w_up"] = _weights(w, (w.E, w.up_rows, w.d), g, device).to(dt)
        out["w_down"] = _weights(w, (w.E, w.d, w.d_ff), g, device).to(dt)
        if w.n_shared:
            out["shared_up"] = _weights(w, (w.n_shared, w.up_rows, w.d), g, device).to(dt)
            out["shared_down"] = _weights(w, (w.n_shared, w.d, w.d_ff), g, device).to(dt)
    return out


def random_topk(T: int, E: int, k: int, seed: int, skew: float = 0.0, device="cpu"):
    """Seeded expert choices without a router: k distinct experts per token,
    drawn with Zipf(skew)-shaped popularity (skew=0: uniform).  Used to drive
    the dispatch step on its own."""
    g = _gen(seed, device)
    rank = torch.randperm(E, generator=g, device=device).to(torch.float64)
    weight = (rank + 1.0) ** (-skew)
    p = (weight / weight.sum()).to(torch.float32).expand(T, E).contiguous()
    return torch.multinomial(p, k, replacement=False, generator=g).to(torch.int32)


def seed_everything_info(w: Workload) -> str:
    """One-line description of the draw recipe (for bench output)."""
    return (f"seed={w.seed}; x=U{{-8..8}}/8; weights={w.weights}; "
            f"logit_skew={w.logit_skew}; sel_bias_std={w.sel_bias_std}; sel_skew={w.sel_skew}")


__all__ = ["Workload", "WORKLOADS", "SWEEP_T", "SWEEP_S", "sweep", "get", "make_inputs",
           "random_topk", "seed_everything_info", "math"]
