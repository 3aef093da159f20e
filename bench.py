#!/usr/bin/env python
"""MoE-layer throughput on B300: route -> dispatch -> expert FFN -> combine.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Default workload: the Mixtral-8x7B-shaped layer (T=16384 tokens, d=4096, 8
experts top-2, SwiGLU d_ff=14336, bf16, no dropping) on seeded synthetic
inputs.  One JSON line is printed by rank 0.

`value` is tokens/s of the whole layer with inputs resident in HBM (CUDA
events around K back-to-back moe_layer_forward calls).  Inputs are larger
than L2 (x 134 MB, weights 2.8 GB), so no explicit L2 flush is needed.
`e2e` adds, every step, the pinned host->device copy of x and the
device->host copy of y (double-buffered on a copy stream, as a serving loop
would run them).  `roofline` is for the dominant kernel (the tcgen05
grouped GEMM): algorithmic FLOPs / its measured time, against the measured
sustained bf16 peak.  `cpu_baseline` is the CPU oracle timed on a bounded
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
    # Mixtral-shaped step: up 2.18 GB read + 0.928 GB written, down 5.20 GB + 0.265 GB.
    "mixtral": {"bytes": 2.18e9 + 0.92834e9 + 5.20e9 + 0.2649e9, "src_hash": "aaa35b3fa1d43b50",
                "per": "step (up + down launches)"},
}


def _src_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


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
def oracle_step(w, inp, rng_seed, route_tokens, ffn_experts, disp_tokens=None, comb_tokens=256):
    """Time the oracle on a bounded sample and extrapolate to the workload:
    route `route_tokens` tokens; dispatch and permute `disp_tokens` tokens
    (all T by default); the expert FFN of `ffn_experts` experts with as many of
    their rows as the oracle has threads (it parallelises one call over its
    rows, and every expert of the full workload has far more rows than
    threads); combine `comb_tokens` tokens.  Each phase is scaled linearly to
    the full workload (the FFN by rows).  Returns (seconds for the whole
    workload, description, per-phase seconds)."""
    import torch

    import moe_workloads as W
    import oracle
    T = w.T
    g = torch.Generator().manual_seed(rng_seed)
    rs = torch.randperm(T, generator=g)[:route_tokens]
    t0 = time.perf_counter()
    oracle.route(inp["x"][rs], inp["w_router"], w.k, w.score, w.renorm, inp["logit_bias"],
                 inp["sel_bias"])
    t_route = (time.perf_counter() - t0) * T / len(rs)
    # dispatch needs every sampled token's choice: take seeded choices of the same shape
    nd = T if disp_tokens is None else max(1, min(T, disp_tokens))
    ds = torch.sort(torch.randperm(T, generator=g)[:nd]).values
    idx = W.random_topk(nd, w.E, w.k, seed=rng_seed)
    C = oracle.capacity(nd, w.k, w.E, w.capacity_factor)
    xs = inp["x"] if nd == T else inp["x"][ds]
    t0 = time.perf_counter()
    disp = oracle.dispatch(idx, w.E, w.R, C)
    xp = oracle.permute(xs, disp["slot_row"], disp["rows"])
    t_disp = (time.perf_counter() - t0) * T / nd
    full_rows = disp["rows"] * T / nd  # kept rows of the whole workload, estimated
    t_ffn = 0.0
    n_rows_s = 0
    n_exp = 0
    off = disp["expert_offsets"]
    rows_per_call = oracle.num_threads()
    yp = torch.zeros((max(disp["rows"], 1), w.d), dtype=torch.float64)
    if w.act != "identity":
        order = torch.randperm(w.E, generator=g).tolist()
        t0 = time.perf_counter()
        for e in order:
            lo, hi = int(off[e]), int(off[e + 1])
            if hi == lo:
                continue
            n = min(rows_per_call, hi - lo)
            yp[lo:lo + n] = oracle.expert_ffn(xp[lo:lo + n], inp["w_up"][e], inp["w_down"][e],
                                              w.act, w.d_ff)
            n_rows_s += n
            n_exp += 1
            if n_exp == ffn_experts:
                break
        t_ffn = (time.perf_counter() - t0) * full_rows / max(n_rows_s, 1)
    else:
        yp = xp.double()
    row_map = torch.arange(max(disp["rows"], 1), dtype=torch.int32)
    fs = torch.randperm(nd, generator=g)[:max(1, min(nd, comb_tokens))]
    t0 = time.perf_counter()
    oracle.combine(fs, yp, row_map, disp["slot_row"], torch.rand((nd, w.k), generator=g))
    t_comb = (time.perf_counter() - t0) * T / len(fs)
    total = t_route + t_disp + t_ffn + t_comb
    desc = (f"route {len(rs)} of {T} tokens, dispatch+permute {nd} of {T}, expert FFN on "
            f"{n_rows_s} rows ({n_exp} experts x up to {rows_per_call} rows, one row per oracle "
            f"thread), combine {len(fs)} tokens; each phase extrapolated linearly to the full "
            f"workload")
    return total, desc, dict(route=t_route, dispatch=t_disp, ffn=t_ffn, combine=t_comb)


def cpu_inputs(w, dev_inp=None):
    import torch

    import moe_workloads as W
    if dev_inp is not None:
        return {k: (v.cpu() if torch.is_tensor(v) else v) for k, v in dev_inp.items()}
    return W.make_inputs(w, device="cpu")


def run_reference(args, w):
    """The oracle as it stands, on the host cores, one bounded sample per step,
    sized so that all warm-up and timed steps together take about
    --ref-budget-s seconds (or one minimal sample per step, if even that is
    over budget)."""
    import oracle
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    inp = cpu_inputs(w)
    # Calibration step (one of the warm-up steps) with one expert's FFN sample;
    # the FFN is nearly all of the oracle's time, so only the number of sampled
    # experts grows to fill the per-step budget.
    rt, dt, fe = min(w.T, 256), min(w.T, 2048), 1
    t0 = time.perf_counter()
    oracle_step(w, inp, 99, rt, fe, dt)
    cal = time.perf_counter() - t0
    per_step = args.ref_budget_s / max(1, args.steps + args.warmup)
    if cal < per_step:
        fe = int(max(1, min(args.ref_ffn_experts, w.E, per_step / cal)))
    for i in range(max(0, args.warmup - 1)):
        oracle_step(w, inp, 100 + i, rt, fe, dt)
    times = []
    desc = ""
    t_wall = time.perf_counter()
    for i in range(args.steps):
        t, desc, _ = oracle_step(w, inp, 1000 + i, rt, fe, dt)
        times.append(t)
    wall = time.perf_counter() - t_wall
    per_step = statistics.mean(times)
    value = w.T / per_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded dyadic grid)",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "d_ff": w.d_ff,
                   "act": w.act},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "sample_wall_s": wall,
    }
    print(json.dumps(line), flush=True)


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

    inp = W.make_inputs(w, device=dev)
    cfg = moe.config_from_workload(w)
    layer = moe.MoeLayer(cfg, inp["w_router"], inp.get("w_up"), inp.get("w_down"),
                         inp.get("shared_up"), inp.get("shared_down"), inp.get("logit_bias"),
                         inp.get("sel_bias"), device=dev)
    x = inp["x"]
    stream = torch.cuda.current_stream()
    ident = w.act == "identity"
    # route 1, dispatch 3 (count, scan, place), combine 1, FFN 2 per expert set
    per_step_launches = 5 + (0 if ident else 2 * (1 + w.n_shared))

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

    # ---- timed region: K whole-layer calls, inputs resident in HBM ----
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(uuid if rank == 0 else None) as clk:
        barrier()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            layer(x)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = max_over_ranks(ev0.elapsed_time(ev1)) / args.steps
    clocks = clk.summary() if rank == 0 else None
    value = world * w.T / (ms / 1e3)

    # ---- per-step breakdown: the same four C-ABI calls with events between ----
    b = layer.buf
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    torch.cuda.synchronize()
    for s in range(args.steps):
        e = evs[s]
        e[0].record(stream)
        moe.moe_route(cfg, x, inp["w_router"], inp.get("logit_bias"), inp.get("sel_bias"),
                      b.topk_idx, b.topk_gate, b.ws)
        e[1].record(stream)
        moe.moe_dispatch(cfg, x, b.topk_idx, b.xp, b.row_token, b.slot_row, b.expert_counts,
                         b.expert_offsets, b.rank_counts, b.rank_splits, b.n_dropped, b.ws)
        e[2].record(stream)
        if not ident:
            moe.moe_expert_ffn(cfg, b.xp, b.expert_offsets, inp["w_up"], inp["w_down"], b.h, b.yp,
                               x if w.n_shared else None, inp.get("shared_up"),
                               inp.get("shared_down"), b.shared_h, b.shared_out, b.ws)
        e[3].record(stream)
        moe.moe_combine(cfg, b.xp if ident else b.yp, b.slot_row, b.topk_gate, b.shared_out,
                        x if w.add_residual else None, b.y)
        e[4].record(stream)
    torch.cuda.synchronize()
    phase = {}
    for i, name in enumerate(["route", "dispatch", "ffn", "combine"]):
        phase[name] = statistics.mean(evs[s][i].elapsed_time(evs[s][i + 1])
                                      for s in range(args.steps))
    assert layer.device_status() == 0

    # ---- e2e: pinned host x in, y out, every step ----
    # Double-buffered like a serving loop: the H2D copy of step i+1 and the
    # D2H copy of step i-1 run on a copy stream while step i computes.  Each
    # step still moves its own x in and its own y out.
    xh = x.cpu().pin_memory()
    yh = [torch.empty(b.y.shape, dtype=b.y.dtype, pin_memory=True) for _ in range(2)]
    xd = [torch.empty_like(x) for _ in range(2)]
    yd = [torch.empty_like(b.y) for _ in range(2)]
    copy_s = torch.cuda.Stream(device=dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    y_ready = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]
    in_free = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(n):
        with torch.cuda.stream(copy_s):
            xd[0].copy_(xh, non_blocking=True)
            h2d_done[0].record(copy_s)
        for i in range(n):
            cur, nxt = i % 2, (i + 1) % 2
            if i + 1 < n:
                with torch.cuda.stream(copy_s):
                    if i >= 1:
                        copy_s.wait_event(in_free[nxt])  # step i-1 finished reading xd[nxt]
                    xd[nxt].copy_(xh, non_blocking=True)
                    h2d_done[nxt].record(copy_s)
            stream.wait_event(h2d_done[cur])
            if i >= 2:
                stream.wait_event(d2h_done[cur])       # yd[cur] drained by step i-2's D2H
            y = layer(xd[cur])
            yd[cur].copy_(y, non_blocking=True)
            in_free[cur].record(stream)
            y_ready[cur].record(stream)
            with torch.cuda.stream(copy_s):
                copy_s.wait_event(y_ready[cur])
                yh[cur].copy_(yd[cur], non_blocking=True)
                d2h_done[cur].record(copy_s)
        stream.wait_stream(copy_s)

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    ev0.record(stream)
    e2e_run(args.steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1)) / args.steps
    bytes_in = x.numel() * x.element_size()
    bytes_out = b.y.numel() * b.y.element_size()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    ffn_ms = phase["ffn"]
    kernels = {
        "route": {"ms": phase["route"],
                  "GB/s": work["route_bytes"] / (phase["route"] * 1e-3) / 1e9,
                  "TFLOP/s": work["route_flops"] / (phase["route"] * 1e-3) / 1e12},
        "dispatch": {"ms": phase["dispatch"],
                     "GB/s": work["permute_bytes"] / (phase["dispatch"] * 1e-3) / 1e9},
        "combine": {"ms": phase["combine"],
                    "GB/s": work["combine_bytes"] / (phase["combine"] * 1e-3) / 1e9},
    }
    for kname in ("dispatch", "combine"):
        kernels[kname]["frac_hbm"] = kernels[kname]["GB/s"] / peaks["hbm"]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if not ident:
        kernels["ffn"] = {"ms": ffn_ms, "TFLOP/s": work["ffn_flops"] / (ffn_ms * 1e-3) / 1e12,
                          "launches_per_step": 2 * (1 + w.n_shared)}
        achieved = kernels["ffn"]["TFLOP/s"]
        if w.dtype == "bf16":
            tr = TRAFFIC.get(w.name)
            traffic = None
            if tr and tr["src_hash"] == _src_hash(os.path.join(ROOT, "expert_dispatch_top_b300",
                                                               "csrc", "ffn_tc.cu")):
                traffic = tr["bytes"]
            roofline = {"kernel": "tc_gemm_kernel (expert FFN, up+down per step)",
                        "bound": "tensor", "achieved": achieved, "peak": peaks["bf16_sus"],
                        "unit": "TFLOP/s", "frac": achieved / peaks["bf16_sus"],
                        "traffic": traffic, "peak_kind": f"bf16 sustained ({peaks['src']})",
                        "frac_of_burst": achieved / peaks["bf16"],
                        "algorithmic_flops_per_step": work["ffn_flops"]}
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
    # bf16 routers run on the tensor cores (a short kernel: burst peak), fp32 ones on FFMA
    if w.dtype == "bf16":
        kernels["route"]["pipe"] = "tensor (bf16)"
        kernels["route"]["frac_tensor"] = kernels["route"]["TFLOP/s"] / peaks["bf16"]
    else:
        kernels["route"]["pipe"] = "FFMA (fp32)"
        kernels["route"]["frac_fp32_ffma"] = kernels["route"]["TFLOP/s"] / \
            fp32_ffma_peak_tflops(sms, peaks["sm_mhz"])
    kernels["route"]["frac_hbm"] = kernels["route"]["GB/s"] / peaks["hbm"]

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        import oracle
        inp_cpu = cpu_inputs(w, inp)
        t, desc, parts = oracle_step(w, inp_cpu, 7, args.ref_route_tokens, args.ref_ffn_experts)
        cpu = {"value": w.T / t, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
               "sample": desc, "phase_s": parts}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded dyadic grid; no dataset)",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "R": w.R,
                   "d_ff": w.d_ff, "act": w.act, "score": w.score, "max_ranks": w.max_ranks,
                   "capacity_factor": w.capacity_factor, "n_shared": w.n_shared,
                   "kept_rows": n_kept, "parallelism": f"replicas x{world}" if world > 1 else "none",
                   "l2": "inputs larger than L2 (x and expert weights); no flush"},
        "e2e": {"value": world * w.T / (e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": bytes_in, "d2h_bytes_per_step": bytes_out,
                "overlap": "double-buffered: H2D(i+1) and D2H(i-1) on a copy stream during step i"},
        "gpu_launches": per_step_launches * args.steps,
        "roofline": roofline,
        "kernels": kernels,
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
    ap.add_argument("--backward", action="store_true",
                    help="also time the expert-FFN backward (kernels.ffn_backward)")
    ap.add_argument("--ref-route-tokens", type=int, default=256)
    ap.add_argument("--ref-ffn-experts", type=int, default=8,
                    help="experts whose FFN the oracle sample runs (rows: one per oracle thread)")
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
