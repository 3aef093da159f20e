#!/usr/bin/env python
"""MoE-layer throughput on B300: route -> dispatch -> expert FFN -> combine.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: the Mixtral-8x7B-shaped layer (T=16384 tokens, d=4096, 8
experts top-2, SwiGLU d_ff=14336, bf16, no dropping) on seeded synthetic
inputs.  One JSON line is printed by rank 0.

`value` is tokens/s of the whole layer with inputs resident in HBM: K
back-to-back steps, each the four C-ABI calls that moe_layer_forward makes
(moe_route, moe_dispatch, moe_expert_ffn, moe_combine) with CUDA events
between them, so the per-kernel times in `kernels` come from the same timed
pass and add up to the step.  Inputs are larger than L2 (x 134 MB, weights
2.8 GB), so no explicit L2 flush is needed.  `layer_forward` repeats the K
steps through the single moe_layer_forward call as a cross-check, with its
own clock record.  `e2e` is the same metric through the C-ABI call with HOST
buffers (moe_layer_forward_host: the pinned host->device copy of x, the
layer and the device->host copy of y, every step; two layer instances
alternate on two streams, as a serving loop would run them).  `roofline` is for the dominant kernel (the
tcgen05 grouped GEMM): algorithmic FLOPs / its measured time, against the
measured bf16 burst peak.  `configs` holds one record per other workload
(the toy, Switch- and DeepSeek-shaped layers and the sweep's end points),
each with its own timed steps, L2 flushed before every step, per-kernel
rates and clock record.  `cpu_baseline` is the CPU oracle timed on a bounded
sample of the same workload on this host's cores (N=1, rank 0).

With --impl reference the CPU oracle itself is timed (on the host cores,
rank 0 only) on a bounded sample of the workload per step.

Multi-GPU (torchrun, N>1): replicas only -- every rank runs the whole layer on
its own tokens with no collective on the data path; value = all ranks'
tokens / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s on 1 B300; expert GEMM % bf16 peak; permute GB/s % HBM"
UNIT = "tokens/s"

# DRAM traffic of one tc_gemm_kernel launch pair (up + down) per workload from
# an ncu capture (dram__bytes_read.sum + dram__bytes_write.sum), with the
# hash of ffn_tc.cu at capture time: reported only while the kernel source is
# unchanged.  See profiles/ for the commands.
TRAFFIC = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum (1 pass) on the full
    # Mixtral-shaped step: up 2.192 GB read + 0.929 GB written, down (banded tile
    # order) 4.459 GB + 0.266 GB.  Valid while the kernel's device code (ffn_tc.cu
    # and its tile schedule, gemm_tiles.cuh) is unchanged.
    "mixtral": {"bytes": 2.1918e9 + 0.9288e9 + 4.4590e9 + 0.2657e9, "src_hash": "8ea23d976567afdd",
                "per": "step (up + down launches)"},
}
GEMM_SRC = [os.path.join(ROOT, "expert_dispatch_top_b300", "csrc", f)
            for f in ("ffn_tc.cu", "gemm_tiles.cuh")]


def _src_hash(paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured", sm_mhz=d.get("sm_max_mhz", 2032.0))
    return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, src="fallback", sm_mhz=2032.0)


def fp32_ffma_peak_tflops(sm_count, sm_mhz):
    """FP32 FFMA roofline: SMs x 128 FP32 lanes x 2 flops x clock."""
    return sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12


# Dense tf32 : bf16 tensor rate on B300, nominal (1.1 vs 2.25 PFLOP/s): the
# tf32 roofline is the measured bf16 burst peak times this ratio.
TF32_PER_BF16 = 1.1 / 2.25


def ffn_on_tf32(w):
    """fp32 experts whose d and d_ff are multiples of 16 run on the tensor cores
    as three tf32 products per fp32 product (split pass + up + down)."""
    return w.dtype == "f32" and w.act != "identity" and w.d % 16 == 0 and w.d_ff % 16 == 0


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid):
        self.uuid = gpu_uuid
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"] + (["-i", self.uuid] if self.uuid else []),
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [r for r in rows if r[2] > 200.0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3][1:5])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(loaded), "power_w_max": max(r[2] for r in rows)}


def replica_throughput(local_ms, tokens_per_rank, world, device="cpu"):
    """Replicas-only scaling: every rank runs the whole layer on its own tokens.
    The job's time is the slowest rank's (all_reduce MAX) and its throughput
    counts every rank's tokens.  Returns (max_ms, tokens/s)."""
    import torch
    import torch.distributed as dist
    ms = float(local_ms)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_per_rank / (ms / 1e3)


def layer_work(w, n_kept):
    """Algorithmic work of one layer step (counted once, nothing dense over E)."""
    b = 4 if w.dtype == "f32" else 2
    T, d, f, k = w.T, w.d, w.d_ff, w.k
    mult = 3 if w.act == "swiglu" else (2 if w.act == "gelu" else 0)
    ffn_flops = 2.0 * n_kept * d * f * mult + w.n_shared * 2.0 * T * d * f * mult
    route_bytes = T * d * b + w.E * d * b
    permute_bytes = T * d * b + n_kept * d * b
    combine_bytes = n_kept * d * b + T * d * b * (1 + w.n_shared + int(w.add_residual))
    weight_bytes = (w.E + w.n_shared) * (w.up_rows * d + d * f) * b if mult else 0
    return dict(ffn_flops=ffn_flops, route_bytes=route_bytes, permute_bytes=permute_bytes,
                combine_bytes=combine_bytes, weight_bytes=weight_bytes,
                route_flops=2.0 * T * d * w.E)


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and --impl reference)
# ---------------------------------------------------------------------------
def oracle_layer_sample(w, inp, n_tokens, seed):
    """One oracle step: the whole layer (route, dispatch, expert FFN, combine)
    with the workload's weights on `n_tokens` seeded tokens of its batch.
    Every step of the oracle costs time in proportion to the tokens it
    processes (capacity, if any, is computed for the sample's own size), so
    tokens / seconds is its measured throughput on this workload.  Returns
    seconds."""
    import torch

    import oracle
    g = torch.Generator().manual_seed(seed)
    toks = torch.sort(torch.randperm(w.T, generator=g)[:max(1, min(w.T, n_tokens))]).values
    x = inp["x"][toks]
    t0 = time.perf_counter()
    oracle.layer_forward(x, inp["w_router"], k=w.k, E=w.E, R=w.R, d_ff=w.d_ff, act=w.act,
                         score=w.score, renorm=w.renorm, capacity_factor=w.capacity_factor,
                         logit_bias=inp.get("logit_bias"), sel_bias=inp.get("sel_bias"),
                         w_up=inp.get("w_up"), w_down=inp.get("w_down"),
                         shared_up=inp.get("shared_up"), shared_down=inp.get("shared_down"),
                         add_residual=w.add_residual, max_ranks=w.max_ranks)
    return time.perf_counter() - t0


def oracle_tokens_for(w, inp, seconds):
    """Tokens per oracle step so that one step takes about `seconds` (from a
    calibration step on one token per oracle thread)."""
    import oracle
    n0 = max(1, min(w.T, oracle.num_threads()))
    t = oracle_layer_sample(w, inp, n0, 12345)
    return int(max(1, min(w.T, seconds * n0 / max(t, 1e-6))))


def oracle_sample_desc(w, n):
    return (f"the whole layer (route, dispatch, expert FFN, combine) on {n} seeded tokens of "
            f"the {w.T}-token batch per step, with the workload's full weights; measured, not "
            f"extrapolated (the oracle's work is linear in tokens)")


def cpu_inputs(w):
    import moe_workloads as W
    return W.make_inputs(w, device="cpu")


def run_reference(args, w):
    """The oracle as it stands, on the host cores: each step is the whole layer
    on a seeded token sample, sized so that all warm-up and timed steps take
    about --ref-budget-s seconds together."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = cpu_inputs(w)
    per_step = args.ref_budget_s / max(1, args.steps + args.warmup)
    n = oracle_tokens_for(w, inp, per_step)
    for i in range(max(0, args.warmup - 1)):  # the calibration step was the first warm-up
        oracle_layer_sample(w, inp, n, 100 + i)
    times = []
    t_wall = time.perf_counter()
    for i in range(args.steps):
        times.append(oracle_layer_sample(w, inp, n, 1000 + i))
    wall = time.perf_counter() - t_wall
    ms = statistics.mean(times) * 1e3
    value = n / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded dyadic grid; no dataset)",
        "config": workload_config(w, None, 1),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": oracle_sample_desc(w, n),
                         "tokens_per_step": n},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "sample_wall_s": wall,
    }
    print(json.dumps(line), flush=True)


def workload_config(w, n_kept, world):
    return {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "R": w.R,
            "d_ff": w.d_ff, "act": w.act, "score": w.score, "max_ranks": w.max_ranks,
            "capacity_factor": w.capacity_factor, "n_shared": w.n_shared,
            "parallelism": f"replicas x{world}" if world > 1 else "none",
            "l2": "inputs larger than L2 (x and expert weights); no flush"}


# ---------------------------------------------------------------------------
# GPU path
# ---------------------------------------------------------------------------
def time_ffn_backward(args, w, cfg, b, inp, stream, peaks):
    """Opt-in (--backward): time moe_expert_ffn_backward (input and both weight
    gradients) over the forward's dispatched rows, with a seeded d_yp.

    Tensor flops per call: the recomputed up projection (2 rows d up), dh
    (2 rows d f), d_xp (2 rows up d), dW_down (2 rows d f), dW_up (2 rows up d);
    the bf16 weight and activation transposes are HBM traffic, not flops."""
    import torch

    import expert_dispatch_top_b300 as moe
    import moe_workloads as W

    rows = int(b.expert_offsets[-1].item())
    up = w.up_rows
    g = W._gen(w.seed + 100, b.xp.device)
    d_yp = W._grid_normal(tuple(b.yp.shape), 0.5, 2.0 ** -9, 4.0, g, b.xp.device).to(b.yp.dtype)
    d_xp = torch.empty_like(b.xp)
    d_wu = torch.empty_like(inp["w_up"])
    d_wd = torch.empty_like(inp["w_down"])
    nbytes = moe.moe_expert_ffn_backward_scratch_size(cfg, True)
    scratch = torch.empty(nbytes, dtype=torch.uint8, device=b.xp.device)

    def call():
        moe.moe_expert_ffn_backward(cfg, b.xp, b.expert_offsets, inp["w_up"], inp["w_down"], d_yp,
                                    d_xp, d_wu, d_wd, scratch, b.ws)

    for _ in range(max(args.warmup, 1)):
        call()
    torch.cuda.synchronize()
    n = max(args.steps // 4, 3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(b.ws) == 0
    ms = e0.elapsed_time(e1) / n
    flops = 2.0 * rows * w.d * (3 * up + 2 * w.d_ff)
    tf = flops / (ms * 1e-3) / 1e12
    out = {"ms": ms, "calls": n, "rows": rows, "tensor_flops_per_call": flops, "TFLOP/s": tf,
           "scratch_bytes": nbytes}
    if w.dtype == "bf16":
        out["frac_bf16_sustained"] = tf / peaks["bf16_sus"]
    return out


def _phase_calls(moe, cfg, w, inp, b, x):
    """The layer step as its four C-ABI calls (what moe_layer_forward enqueues),
    so that events can sit between them."""
    ident = w.act == "identity"

    def route():
        moe.moe_route(cfg, x, inp["w_router"], inp.get("logit_bias"), inp.get("sel_bias"),
                      b.topk_idx, b.topk_gate, b.ws)

    def dispatch():
        moe.moe_dispatch(cfg, x, b.topk_idx, b.xp, b.row_token, b.slot_row, b.expert_counts,
                         b.expert_offsets, b.rank_counts, b.rank_splits, b.n_dropped, b.ws)

    def ffn():
        if not ident:
            moe.moe_expert_ffn(cfg, b.xp, b.expert_offsets, inp["w_up"], inp["w_down"], b.h, b.yp,
                               x if w.n_shared else None, inp.get("shared_up"),
                               inp.get("shared_down"), b.shared_h, b.shared_out, b.ws)

    def combine():
        moe.moe_combine(cfg, b.xp if ident else b.yp, b.slot_row, b.topk_gate, b.shared_out,
                        x if w.add_residual else None, b.y)

    return [("route", route), ("dispatch", dispatch), ("ffn", ffn), ("combine", combine)]


def timed_steps(steps, phases, stream, flush=None, barrier=lambda: None):
    """K steps of the layer, each its four calls with a CUDA event before the
    first and after each one, on the launching stream.  With `flush`, a
    buffer larger than L2 is written before every step (outside the step's
    events).  Returns (bracket ms over all K steps, per-step ms, per-phase
    mean ms)."""
    import torch
    n = len(phases)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n + 1)] for _ in range(steps)]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    ev0.record(stream)
    for s in range(steps):
        if flush is not None:
            flush()
        e = evs[s]
        e[0].record(stream)
        for i, (_, f) in enumerate(phases):
            f()
            e[i + 1].record(stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    per_step = [evs[s][0].elapsed_time(evs[s][n]) for s in range(steps)]
    phase = {name: statistics.mean(evs[s][i].elapsed_time(evs[s][i + 1]) for s in range(steps))
             for i, (name, _) in enumerate(phases)}
    return ev0.elapsed_time(ev1), per_step, phase


def kernel_report(w, work, phase, peaks, sms):
    """Per-kernel times of one timed pass, with rates against their bounds."""
    ident = w.act == "identity"
    k = {
        "route": {"ms": phase["route"],
                  "GB/s": work["route_bytes"] / (phase["route"] * 1e-3) / 1e9,
                  "TFLOP/s": work["route_flops"] / (phase["route"] * 1e-3) / 1e12},
        "dispatch": {"ms": phase["dispatch"],
                     "GB/s": work["permute_bytes"] / (phase["dispatch"] * 1e-3) / 1e9},
        "combine": {"ms": phase["combine"],
                    "GB/s": work["combine_bytes"] / (phase["combine"] * 1e-3) / 1e9},
    }
    for name in ("route", "dispatch", "combine"):
        k[name]["frac_hbm"] = k[name]["GB/s"] / peaks["hbm"]
    # bf16 routers run on the tensor cores (a short kernel: burst peak), fp32 ones on FFMA
    if w.dtype == "bf16":
        k["route"]["pipe"] = "tensor (bf16)"
        k["route"]["frac_tensor"] = k["route"]["TFLOP/s"] / peaks["bf16"]
    else:
        k["route"]["pipe"] = "FFMA (fp32)"
        k["route"]["frac_fp32_ffma"] = k["route"]["TFLOP/s"] / \
            fp32_ffma_peak_tflops(sms, peaks["sm_mhz"])
    if not ident:
        tf = work["ffn_flops"] / (phase["ffn"] * 1e-3) / 1e12
        x3 = ffn_on_tf32(w)
        k["ffn"] = {"ms": phase["ffn"], "TFLOP/s": tf,
                    "launches_per_step": (3 if x3 else 2) * (1 + w.n_shared)}
        if w.dtype == "bf16":
            k["ffn"]["frac_bf16_burst"] = tf / peaks["bf16"]
            k["ffn"]["frac_bf16_sustained"] = tf / peaks["bf16_sus"]
        elif x3:
            # three tf32 products per fp32 product; the phase includes the split pass
            k["ffn"]["pipe"] = "tensor (fp32 as three tf32 products)"
            k["ffn"]["tf32_TFLOP/s"] = 3 * tf
            k["ffn"]["frac_tf32_burst"] = 3 * tf / (peaks["bf16"] * TF32_PER_BF16)
        else:
            k["ffn"]["pipe"] = "FFMA (fp32)"
            k["ffn"]["frac_fp32_ffma"] = tf / fp32_ffma_peak_tflops(sms, peaks["sm_mhz"])
    else:
        moved = work["route_bytes"] + work["permute_bytes"] + work["combine_bytes"]
        ms = phase["route"] + phase["dispatch"] + phase["combine"]
        k["route_permute_unpermute"] = {"ms": ms, "GB/s": moved / (ms * 1e-3) / 1e9,
                                        "frac_hbm": moved / (ms * 1e-3) / 1e9 / peaks["hbm"]}
    return k


class L2Flush:
    """Before each timed step: writes a 512 MiB buffer (over 4x the 126 MB L2),
    then reads a second 256 MiB buffer, so that the step finds none of its
    inputs in L2 and no dirty line of the flush left to write back (a write-only
    flush leaves up to ~126 MB of dirty lines whose write-back the step's first
    kernel would pay for)."""

    DESC = ("flushed before every step: 512 MiB written, then 256 MiB of a second buffer read "
            "(no dirty flush lines left); outside the step's events")

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.rbuf = torch.zeros(64 << 20, dtype=torch.float32, device=dev)
        self.v = 0

    def __call__(self):
        self.v ^= 1
        self.buf.fill_(self.v)
        self.rbuf.sum()


def measure_config(moe, W, w, dev, stream, peaks, sms, uuid, target_ms=400.0):
    """One per-config record for the bench line: inputs drawn on the device, a
    1 s pause and ~0.2 s of warm-up steps (the clocks settle after the previous
    workload), then K steps (K sized to ~target_ms of step time, 20..200) with
    L2 flushed before each step; the four calls timed with events, clocks
    sampled during the timed steps."""
    import torch
    inp = W.make_inputs(w, device=dev)
    cfg = moe.config_from_workload(w)
    b = moe.alloc_buffers(cfg, dev)
    x = inp["x"]
    phases = _phase_calls(moe, cfg, w, inp, b, x)
    flush = L2Flush(dev)
    # let the clocks and power settle after the previous workload, then warm up
    # for ~0.2 s of this workload's own steps before timing
    torch.cuda.synchronize()
    time.sleep(1.0)
    _, per, _ = timed_steps(3, phases, stream, flush)
    warm = int(max(3, min(400, 200.0 / max(statistics.median(per), 1e-3))))
    timed_steps(warm, phases, stream, flush)
    assert moe.moe_read_device_status(b.ws) == 0
    steps = int(max(20, min(200, target_ms / max(statistics.median(per), 1e-3))))
    n0 = moe.moe_launch_count()
    with ClockSampler(uuid) as clk:
        _, per, phase = timed_steps(steps, phases, stream, flush)
    launches = moe.moe_launch_count() - n0
    assert moe.moe_read_device_status(b.ws) == 0
    n_kept = int(b.expert_offsets[-1].item())
    ms = statistics.mean(per)
    work = layer_work(w, n_kept)
    rec = {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "d_ff": w.d_ff,
           "act": w.act, "dtype": w.dtype, "score": w.score, "n_shared": w.n_shared,
           "capacity_factor": w.capacity_factor, "kept_rows": n_kept,
           "dropped_frac": 1.0 - n_kept / (w.T * w.k), "steps": steps, "warmup": 3 + warm,
           "ms_per_step": ms, "value": w.T / (ms * 1e-3), "unit": UNIT,
           "l2": L2Flush.DESC,
           "kernels": kernel_report(w, work, phase, peaks, sms), "clocks": clk.summary(),
           "gpu_launches": launches, "launches_per_step": launches / steps}
    del inp, b, phases, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


DEFAULT_CONFIGS = ["toy", "switch", "deepseek", "sweep_T4096_s0", "sweep_T4096_s1.5",
                   "sweep_T131072_s0", "sweep_T131072_s1.5"]


def time_route_backward(args, w, cfg, b, inp, stream):
    """Opt-in (--backward): time moe_route_backward (logit, input, weight and
    logit-bias gradients) on the forward's choices with a seeded d_gate."""
    import torch

    import expert_dispatch_top_b300 as moe
    import moe_workloads as W

    g = W._gen(w.seed + 200, b.xp.device)
    d_gate = torch.randn(tuple(b.topk_gate.shape), generator=g, device=b.xp.device)
    d_logits = torch.empty((w.T, w.E), dtype=torch.float32, device=b.xp.device)
    dx = torch.empty_like(inp["x"])
    dw = torch.empty_like(inp["w_router"])
    dlb = torch.empty(w.E, dtype=torch.float32, device=b.xp.device)

    def call(weights=True):
        moe.moe_route_backward(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), b.topk_idx,
                               d_gate, d_logits, dx, dw if weights else None,
                               dlb if weights else None)

    def timed(weights):
        for _ in range(max(args.warmup, 1)):
            call(weights)
        torch.cuda.synchronize()
        n = max(args.steps // 4, 3)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            call(weights)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n, n

    ms, n = timed(True)
    # without weight and bias gradients only the per-token kernel (dL, dx) runs
    ms_tok, _ = timed(False)
    return {"ms": ms, "calls": n, "token_kernel_ms": ms_tok, "weight_kernel_ms": ms - ms_tok}


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import expert_dispatch_top_b300 as moe
    import moe_workloads as W

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    peaks = _peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count

    inp = W.make_inputs(w, device=dev)
    cfg = moe.config_from_workload(w)
    layer = moe.MoeLayer(cfg, inp["w_router"], inp.get("w_up"), inp.get("w_down"),
                         inp.get("shared_up"), inp.get("shared_down"), inp.get("logit_bias"),
                         inp.get("sel_bias"), device=dev)
    x = inp["x"]
    stream = torch.cuda.current_stream()
    ident = w.act == "identity"

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v):
        return replica_throughput(v, w.T, world, dev)[0]

    for _ in range(max(args.warmup, 1)):
        layer(x)
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    n_kept = int(layer.buf.expert_offsets[-1].item())
    work = layer_work(w, n_kept)

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass

    # ---- timed region: K layer steps, inputs resident in HBM.  Each step is
    # the four C-ABI calls moe_layer_forward makes, with events between them,
    # so the per-kernel times come from this same pass and add up to the step.
    b = layer.buf
    phases = _phase_calls(moe, cfg, w, inp, b, x)
    # the library counts its own kernel launches: the timed region's are the difference
    n0 = moe.moe_launch_count()
    with ClockSampler(uuid if rank == 0 else None) as clk:
        total_ms, per_step, phase = timed_steps(args.steps, phases, stream, None, barrier)
    launches = moe.moe_launch_count() - n0
    ms = max_over_ranks(total_ms) / args.steps
    clocks = clk.summary() if rank == 0 else None
    value = world * w.T / (ms / 1e3)
    assert layer.device_status() == 0

    # ---- cross-check: the same K steps through moe_layer_forward (one call) ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(uuid if rank == 0 else None) as clk2:
        barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            layer(x)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
    lf_ms = max_over_ranks(ev0.elapsed_time(ev1)) / args.steps
    lf_clocks = clk2.summary() if rank == 0 else None
    assert layer.device_status() == 0

    # ---- e2e: the C-ABI call with HOST buffers, every step ----
    # moe_layer_forward_host copies the step's x in from pinned host memory, runs
    # the layer and copies its y back out, all enqueued by the library.  Two
    # layer instances (separate buffers, workspaces and staging) alternate on
    # two streams, so one step's copies overlap the other step's kernels, as a
    # serving loop would run them; each step still moves its own x and y.
    layers = [layer, moe.MoeLayer(cfg, inp["w_router"], inp.get("w_up"), inp.get("w_down"),
                                  inp.get("shared_up"), inp.get("shared_down"),
                                  inp.get("logit_bias"), inp.get("sel_bias"), device=dev)]
    e2e_streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    xh = x.cpu().pin_memory()
    yh = [torch.empty(b.y.shape, dtype=b.y.dtype, pin_memory=True) for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]

    def e2e_run(n):
        start = torch.cuda.Event()
        start.record(stream)
        for st in e2e_streams:
            st.wait_event(start)
        for i in range(n):
            j = i % 2
            layers[j].forward_host(xh, yh[j], xd[j], e2e_streams[j])
        for st in e2e_streams:
            stream.wait_stream(st)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    ev0.record(stream)
    e2e_run(args.steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1)) / args.steps
    assert all(lay.device_status() == 0 for lay in layers)
    bytes_in = x.numel() * x.element_size()
    bytes_out = b.y.numel() * b.y.element_size()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    kernels = kernel_report(w, work, phase, peaks, sms)
    phase_sum = sum(phase.values())
    if not ident:
        achieved = kernels["ffn"]["TFLOP/s"]
        if w.dtype == "bf16":
            tr = TRAFFIC.get(w.name)
            traffic = None
            if tr and tr["src_hash"] == _src_hash(GEMM_SRC):
                traffic = tr["bytes"]
            # the FFN runs in ms-long windows between the other kernels: burst peak
            roofline = {"kernel": "tc_gemm_kernel (expert FFN, up+down per step)",
                        "bound": "tensor", "achieved": achieved, "peak": peaks["bf16"],
                        "unit": "TFLOP/s", "frac": achieved / peaks["bf16"],
                        "traffic": traffic, "peak_kind": f"bf16 burst ({peaks['src']})",
                        "frac_of_sustained": achieved / peaks["bf16_sus"],
                        "algorithmic_flops_per_step": work["ffn_flops"]}
        elif ffn_on_tf32(w):
            # tensor work: three tf32 products per fp32 product, over the phase's
            # time (the split pass included); the FFN runs in sub-ms windows: burst
            pk = peaks["bf16"] * TF32_PER_BF16
            roofline = {"kernel": "tc_gemm_x3_kernel (fp32 expert FFN as three tf32 products: "
                                  "split pass + up + down per step)",
                        "bound": "tensor", "achieved": 3 * achieved, "peak": pk, "unit": "TFLOP/s",
                        "frac": 3 * achieved / pk, "traffic": None,
                        "peak_kind": f"tf32 dense = bf16 burst ({peaks['src']}) x 1.1/2.25 nominal",
                        "fp32_TFLOP/s": achieved,
                        "algorithmic_flops_per_step": work["ffn_flops"],
                        "tensor_flops_per_step": 3 * work["ffn_flops"]}
        else:
            pk = fp32_ffma_peak_tflops(sms, peaks["sm_mhz"])
            roofline = {"kernel": "gemm_simt_kernel (fp32 expert FFN, up+down per step)",
                        "bound": "alu", "achieved": achieved, "peak": pk, "unit": "TFLOP/s",
                        "frac": achieved / pk, "traffic": None,
                        "peak_kind": f"FP32 FFMA: {sms} SMs x 128 lanes x 2 x {peaks['sm_mhz']:.0f} MHz",
                        "algorithmic_flops_per_step": work["ffn_flops"]}
    else:
        gbs = kernels["dispatch"]["GB/s"]
        roofline = {"kernel": "place_kernel (permute)", "bound": "hbm", "achieved": gbs,
                    "peak": peaks["hbm"], "unit": "GB/s", "frac": gbs / peaks["hbm"],
                    "traffic": None, "peak_kind": f"HBM copy ({peaks['src']})",
                    "algorithmic_bytes_per_step": work["permute_bytes"]}
    if args.backward and not ident:
        kernels["ffn_backward"] = time_ffn_backward(args, w, cfg, b, inp, stream, peaks)
    if args.backward:
        kernels["route_backward"] = time_route_backward(args, w, cfg, b, inp, stream)

    configs = None
    if world == 1 and args.configs:
        del layer, layers, phases, xd
        inp = {kk: v for kk, v in inp.items() if kk == "x"}
        torch.cuda.empty_cache()
        configs = []
        for name in [c for c in args.configs.split(",") if c]:
            configs.append(measure_config(moe, W, W.get(name), dev, stream, peaks, sms, uuid))

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        inp_cpu = cpu_inputs(w)
        n = oracle_tokens_for(w, inp_cpu, args.cpu_step_s)
        ts = [oracle_layer_sample(w, inp_cpu, n, 7 + i) for i in range(2)]
        cpu = {"value": n / statistics.mean(ts), "unit": UNIT, "cores": oracle.num_threads(),
               "kind": "oracle", "sample": oracle_sample_desc(w, n) + "; 2 steps",
               "tokens_per_step": n, "s_per_step": statistics.mean(ts)}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded dyadic grid; no dataset)",
        "config": dict(workload_config(w, n_kept, world), kept_rows=n_kept,
                       timed_step="moe_route, moe_dispatch, moe_expert_ffn, moe_combine with CUDA "
                                  "events between them (the calls moe_layer_forward makes)"),
        "e2e": {"value": world * w.T / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": bytes_in, "d2h_bytes_per_step": bytes_out,
                "via": "moe_layer_forward_host (host x in, host y out; copies enqueued by the library)",
                "overlap": "two layer instances alternate on two streams: one step's copies "
                           "overlap the other's kernels"},
        "gpu_launches": launches,
        "launches_per_step": launches / args.steps,
        "roofline": roofline,
        "kernels": kernels,
        "phase_sum_ms": phase_sum,
        "layer_forward": {"ms_per_step": lf_ms, "value": world * w.T / (lf_ms / 1e3),
                          "unit": UNIT, "clocks": lf_clocks,
                          "note": "same K steps through the single moe_layer_forward call"},
        "configs": configs,
        "cpu_baseline": cpu,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mixtral")
    ap.add_argument("--tokens", type=int, default=0, help="override T (small profiling cases)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override E (small profiling cases with the same rows per expert)")
    ap.add_argument("--max-ranks", type=int, default=-1, help="rank-limited routing (0: off)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", default=",".join(DEFAULT_CONFIGS),
                    help="comma-separated workloads measured after the main line, each with its "
                         "own timed steps and clocks ('' to skip)")
    ap.add_argument("--backward", action="store_true",
                    help="also time the expert-FFN and router backwards (kernels.ffn_backward, "
                         "kernels.route_backward)")
    ap.add_argument("--cpu-step-s", type=float, default=8.0,
                    help="host seconds per cpu_baseline step (the token sample is sized to fit)")
    ap.add_argument("--ref-budget-s", type=float, default=150.0,
                    help="host seconds for all --impl reference steps (samples are sized to fit)")
    args = ap.parse_args()
    import moe_workloads as W
    w = W.get(args.workload)
    if args.tokens:
        w = w.replace(T=args.tokens)
    if args.experts:
        w = w.replace(E=args.experts)
    if args.max_ranks >= 0:
        w = w.replace(max_ranks=args.max_ranks)
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
