#!/usr/bin/env python3
"""Throughput of the MoE-layer forward pass on B300 (libmoe, sm_103a).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-per-config]
                    [--pass forward|backward]

A step is one forward pass of the layer (route, dispatch, expert FFN,
combine) over one batch of seeded synthetic inputs of the named workload
(default: the large-FFN layer, bf16, T=16384 tokens, d=4096, d_ff=14336,
E=8, top-2).  The inputs and the expert weights are resident in HBM when the
timed region starts; L2 is flushed (a 256 MiB write, untimed) before every
timed step.  Each timed iteration replays a CUDA graph of one moe_forward
call and then, after a second flush, the graphs of the stage calls (route +
dispatch, expert FFN, combine), so the step and its stages are timed under
the same clocks; the expert FFN's stage time gives the dominant kernel's
roofline (against the measured bf16 burst peak, the sustained one as a
note).  The same steps back to back without a flush give the warm-L2
figure.  The end-to-end figure (`e2e`) runs the steps through the host-buffer
executor (moe_pipeline_*): pinned host batch in, y and the loss out, the
copies of neighbouring steps overlapping the forward pass.  With the default
workload, `per_config` adds the other graded workloads (the T=4096 layer,
Switch routing with the capacity drop, the decode-sized batch), timed the
same way.  Rank 0 prints one JSON line.

Under torchrun (N > 1) every rank runs an independent replica of the layer
on its own GPU (the layer has no cross-GPU step); the line reports the tokens
of all ranks over the slowest rank's time.

--impl reference times the CPU oracle (fp64, numpy) on the host cores on a
bounded token sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mixture_experts_71_b300 import inputs as I  # noqa: E402

DEFAULT_WORKLOAD = I.LARGE.name
L2_BYTES = 126 << 20  # B300 L2
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
METRIC = "MoE-layer fwd tokens/s and achieved TFLOP/s (or HBM GB/s) vs B300 roofline"

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def algorithmic_work(wl, kept_per_expert):
    """FLOPs and minimum HBM bytes of one forward pass.

    FLOPs: router 2*T*d*E plus 4*d*d_ff per kept assignment (two GEMMs).
    Bytes: x, y, W_r, and the weights and biases of every expert that kept at
    least one assignment.
    """
    es = 4 if wl.dtype == "f32" else 2
    kept = int(sum(kept_per_expert))
    used = int(sum(1 for c in kept_per_expert if c > 0))
    flops_router = 2.0 * wl.T * wl.d * wl.E
    flops_ffn = 4.0 * kept * wl.d * wl.F
    w_bytes = used * (2 * wl.d * wl.F + wl.F + wl.d) * es
    io_bytes = 2 * wl.T * wl.d * es + wl.E * wl.d * 4
    return dict(flops=flops_router + flops_ffn, flops_ffn=flops_ffn, bytes=w_bytes + io_bytes,
                ffn_bytes=w_bytes + kept * wl.d * (es + 4), kept=kept, experts_used=used)


class ClockSampler:
    """Samples SM clock and throttle reasons while the timed region runs.

    Uses NVML through pynvml when it is importable, else an
    ``nvidia-smi --query-gpu ... -lms`` subprocess (reading settings only)."""

    REASONS = {  # NVML clocks-event-reason bits
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
        0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
        0x100: "display_clock_setting"}
    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown")

    def __init__(self, index: int, period_s: float = 0.01):
        self.index, self.period = index, period_s
        self.samples, self.reasons = [], set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None
        self.mode = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception:
            import shutil
            if shutil.which("nvidia-smi"):
                self.mode = "smi"

    def _run_nvml(self):
        nv = self._nv
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(self._h)
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.mode == "nvml":
            self._t = threading.Thread(target=self._run_nvml, daemon=True)
            self._t.start()
        elif self.mode == "smi":
            import subprocess
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.SMI_FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)  # let the first sample land before the timed region
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._t is not None:
            self._t.join()
        if self._proc is not None:
            time.sleep(0.05)
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            names = ("sw_power_cap", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")
            for line in out.splitlines():
                f = [v.strip() for v in line.split(",")]
                if len(f) < 6 or not f[0].isdigit():
                    continue
                self.samples.append(int(f[0]))
                self.max_mhz = int(f[1]) if f[1].isdigit() else self.max_mhz
                for name, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(name)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "samples": 0, "source": self.mode}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons - {"gpu_idle"}), "samples": len(self.samples),
                "source": self.mode}


def slowest_rank_ms(ms: float, world: int, device=None) -> float:
    """The job's time: the largest of the ranks' timings (an all-reduce MAX
    over the process group when there is more than one rank; NCCL on the GPU
    box, gloo in the CPU tests)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens: int, steps: int, total_ms: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time
    (each rank runs an independent replica on a batch of `tokens`)."""
    return world * tokens * steps / (total_ms * 1e-3)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def blas_threads() -> int:
    """Threads the oracle's BLAS calls use (numpy's OpenBLAS)."""
    try:
        from threadpoolctl import threadpool_info
        n = [p.get("num_threads", 1) for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return max(n)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def oracle_layer(wl, inp):
    """fn(n): the oracle's layer on the first n tokens as a batch of their own."""
    from oracle import moe_oracle as O
    x = inp.as_f32("x")
    W1, b1, W2, b2 = (inp.as_f32(n) for n in ("W1", "b1", "W2", "b2"))
    if wl.routing == "expert":
        return lambda n: O.expert_choice_forward(x[:n], inp.W_r, W1, b1, W2, b2, k=wl.k,
                                                 capacity=wl.capacity,
                                                 logit_bias=inp.logit_bias)
    return lambda n: O.moe_forward(x[:n], inp.W_r, W1, b1, W2, b2, k=wl.k,
                                   renormalize=wl.renormalize, capacity=wl.capacity,
                                   logit_bias=inp.logit_bias, layout=False,
                                   reroute=wl.overflow == "reroute")


def cpu_oracle_rate(wl, inp, budget_s: float, probe: int = 256):
    """Tokens/s of the oracle on a token sample sized to the time budget.

    The sample is the first n tokens of the batch taken as a batch of their own
    (routing, experts, combine and loss all run on it).  The oracle has a fixed
    cost per call (per-expert weight conversion), so n grows until one run
    takes at least half the budget (or covers the batch)."""
    layer = oracle_layer(wl, inp)

    def run(n):
        t0 = time.perf_counter()
        layer(n)
        return time.perf_counter() - t0

    run(min(wl.T, 4))  # first call: imports, page faults of the widened weights
    n = min(wl.T, probe)
    t = run(n)
    for _ in range(5):
        if t >= 0.5 * budget_s or n >= wl.T:
            break
        n = int(min(wl.T, max(2 * n, 0.9 * n * budget_s / max(t, 1e-6))))
        t = run(n)
    return n / t, n, t, blas_threads()


def bench_reference(args, wl):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    inp = I.make_inputs(wl, seed=0)
    per_step = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    layer = oracle_layer(wl, inp)
    # size the per-step sample from one probe step
    rate, n, _, threads = cpu_oracle_rate(wl, inp, per_step)
    n = max(1, min(wl.T, int(rate * per_step)))

    def step():
        layer(n)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = n * args.steps / total
    sample = f"first {n} of {wl.T} tokens as a batch of their own, per step"
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "d_ff": wl.F, "E": wl.E,
                       "k": wl.k, "capacity": wl.capacity},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _stats(ms):
    return {"mean": statistics.mean(ms), "median": statistics.median(ms), "min": min(ms)}


def ffn_roofline(wl, work, ffn_ms, pk, pk_kind):
    """Roofline of the expert FFN (the grouped GEMM1 + GEMM2 launch pair, the
    dominant kernel): against the measured bf16 burst peak when its arithmetic
    intensity is above the ridge (the stage is timed on its own, in its own
    graph), else its algorithmic bytes against the measured HBM copy rate."""
    ffn_s = ffn_ms * 1e-3
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)  # flop per byte
    traffic, traffic_src = committed_traffic(wl.name)
    if wl.dtype == "bf16" and work["flops_ffn"] / work["ffn_bytes"] >= ridge:
        achieved = work["flops_ffn"] / ffn_s / 1e12
        peak = pk["bf16_tflops"]
        roof = {"bound": "tensor", "unit": "TFLOP/s", "peak_source": pk_kind + " bf16 burst",
                "frac_of_sustained": achieved / pk["bf16_tflops_sustained"],
                "frac_of_2250_nominal": achieved / 2250.0,
                "algorithmic": f"4*d*d_ff*kept = {work['flops_ffn']:.4g} flop per launch pair"}
    else:
        achieved = work["ffn_bytes"] / ffn_s / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "unit": "GB/s", "peak_source": pk_kind + " HBM copy",
                "frac_of_8tbs_nominal": achieved / 8000.0,
                "algorithmic": f"used-expert weights + kept rows in and out = "
                               f"{work['ffn_bytes']:.4g} B per launch pair"}
    fused = (wl.dtype == "bf16" and wl.T * wl.k >= 96 * wl.E and
             wl.T * wl.k * wl.d * wl.F <= 2 ** 39)  # the library's rule (csrc/gemm_tc.cu)
    kern = ("expert FFN (ffn_pair_kernel: both grouped GEMMs in one launch)" if fused
            else "expert FFN (grouped GEMM1 + GEMM2)")
    roof.update({"kernel": kern, "achieved": achieved,
                 "peak": peak, "frac": achieved / peak, "traffic": traffic,
                 "traffic_source": traffic_src})
    return roof


def call_roofline(wl, work, step_ms, pk, pk_kind):
    """Roofline of a decode-sized forward call that moe_forward runs as one
    fused expert-FFN kernel between the router and the combine: the call's
    algorithmic bytes (used-expert weights, x, y, W_r) over the timed step,
    against the measured HBM copy rate."""
    achieved = work["bytes"] / (step_ms * 1e-3) / 1e9
    traffic, traffic_src = committed_traffic(wl.name)
    return {"bound": "hbm", "unit": "GB/s", "peak_source": pk_kind + " HBM copy",
            "kernel": "whole moe_forward call (router, fused expert-FFN kernel, combine)",
            "achieved": achieved, "peak": pk["hbm_gbs"], "frac": achieved / pk["hbm_gbs"],
            "frac_of_8tbs_nominal": achieved / 8000.0,
            "algorithmic": f"used-expert weights + x + y + W_r = {work['bytes']:.4g} B per call",
            "traffic": traffic, "traffic_source": traffic_src}


TRAFFIC_SUMMARY = os.path.join("profiles", "grouped_gemm_dram_traffic.md")


def committed_traffic(workload):
    """DRAM bytes (read + write) of one expert-FFN launch pair of `workload`
    from the committed ncu summary - its forward GEMM1 and GEMM2 rows, or the
    row of the fused decode kernel when it has one - with the summary's path;
    (None, None) when it has no capture of the workload."""
    path = os.path.join(ROOT, TRAFFIC_SUMMARY)
    if not os.path.exists(path):
        return None, None
    pair, fused = [], None
    with open(path) as f:
        for line in f:
            cols = [c.strip() for c in line.strip().strip("|").split("|")]
            if len(cols) < 5 or cols[0].strip("`") != workload:
                continue
            try:
                b = (float(cols[3]) + float(cols[4])) * 1e6
            except ValueError:
                continue
            if "GEMM1 + GEMM2" in cols[1]:
                fused = b
            elif re.search(r"\bGEMM[12]\b", cols[1]) and "staged" not in cols[1]:
                pair.append(b)
    if fused is not None:
        return fused, TRAFFIC_SUMMARY
    if len(pair) != 2:
        return None, None
    return sum(pair), TRAFFIC_SUMMARY


def dense_decode(wl) -> bool:
    """Whether moe_forward takes its dense decode path on this workload (every
    expert on all T tokens in one fused kernel; the library's condition, see
    dense_decode in csrc/moe_api.cu)."""
    return (wl.dtype == "bf16" and wl.routing == "token" and wl.overflow == "drop"
            and wl.n_shared == 0 and 0 < wl.T <= 64 and wl.T * wl.k < 96 * wl.E
            and wl.T * wl.k >= 4 * wl.E)


def measure_workload(args, wl, dev, stream, flush, world, e2e=True):
    """Device-timed forward steps of one workload: W warm-up steps, then K
    timed steps in which each iteration replays the moe_forward graph and,
    after a second L2 flush, the stage graphs (route + dispatch, expert FFN,
    combine), so both see the same clocks; then K steps back to back without a
    flush (warm L2); then, optionally, K end-to-end steps through the
    host-buffer executor.  Returns the per-workload record."""
    import torch
    import torch.distributed as dist
    from sparse_mixture_experts_71_b300 import binding as B
    from sparse_mixture_experts_71_b300.layer import MoELayer, capture_graph, device_inputs

    inp = I.make_inputs(wl, seed=0)
    D = device_inputs(inp, dev)
    layer = MoELayer(D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], k=wl.k, capacity=wl.capacity,
                     renormalize=wl.renormalize, logit_bias=D["logit_bias"], routing=wl.routing,
                     overflow=wl.overflow)
    cfg = layer.config(wl.T)
    ws = layer.workspace(wl.T)
    T, k, E, d = wl.T, wl.k, wl.E, wl.d
    ec = wl.routing == "expert"
    n = E * B.expert_choice_capacity(cfg) if ec else T * k  # permuted rows
    i32, f32 = torch.int32, torch.float32
    dt = D["x"].dtype
    kr = B.ranked_columns(cfg)  # router columns (rerouting: the next-best experts too)
    buf = dict(idx=torch.empty((T, kr), dtype=i32, device=dev),
               w=torch.empty((T, kr), dtype=f32, device=dev),
               counts=torch.empty(E, dtype=i32, device=dev),
               aux=torch.empty(1, dtype=f32, device=dev),
               offsets=torch.empty(E + 1, dtype=i32, device=dev),
               slot_of=torch.empty((T, E if ec else k), dtype=i32, device=dev),
               perm_token=torch.empty(n, dtype=i32, device=dev),
               perm_w=torch.empty(n, dtype=f32, device=dev),
               x_perm=torch.empty((n, d), dtype=dt, device=dev),
               y_perm=torch.empty((n, d), dtype=f32, device=dev),
               y=torch.empty((T, d), dtype=dt, device=dev))

    def stage_route(st):
        b = buf
        if ec:
            B.route_expert_choice(cfg, D["x"], D["W_r"], b["offsets"], b["perm_token"],
                                  b["perm_w"], b["slot_of"], ws, x_perm=b["x_perm"],
                                  logit_bias=D["logit_bias"], expert_counts=b["counts"],
                                  stream=st)
            return
        B.route(cfg, D["x"], D["W_r"], b["idx"], b["w"], ws, logit_bias=D["logit_bias"],
                expert_counts=b["counts"], aux_out=b["aux"], stream=st)
        B.dispatch(cfg, D["x"], b["idx"], b["offsets"], b["slot_of"], b["perm_token"],
                   b["x_perm"], ws, topk_w=b["w"], perm_w=b["perm_w"], stream=st)

    def stage_ffn(st):
        b = buf
        B.expert_ffn(cfg, b["x_perm"], b["offsets"], D["W1"], D["b1"], D["W2"], D["b2"],
                     b["y_perm"], ws, perm_w=b["perm_w"], stream=st)

    def stage_combine(st):
        B.combine(cfg, buf["y_perm"], buf["slot_of"], buf["y"], stream=st)

    y_f = torch.empty_like(D["x"])
    aux_f = torch.empty(1, dtype=f32, device=dev)

    def full_forward(st):
        layer.forward(D["x"], y=y_f, aux=aux_f, stream=st)

    # every step is one CUDA-graph replay of the layer call (no host launch cost
    # inside the timed region); the stage graphs time the stages separately
    graphs, kernels = {}, {}
    stages = ("route+dispatch", "expert_ffn", "combine")
    for name, fn in (("forward", full_forward), ("route+dispatch", stage_route),
                     ("expert_ffn", stage_ffn), ("combine", stage_combine)):
        c0 = B.launch_count()
        for _ in range(2):
            fn(stream)
        torch.cuda.synchronize(dev)
        c1 = B.launch_count()
        graphs[name] = capture_graph(fn, warmup=0)
        kernels[name] = B.launch_count() - c1  # kernels the graph holds
        assert 2 * kernels[name] == c1 - c0, "a graph must hold the eager launches"
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        graphs["forward"].replay()
        flush.fill_(1)
        for name in stages:
            graphs[name].replay()
    torch.cuda.synchronize(dev)
    kept = [int(v) for v in torch.diff(buf["offsets"]).cpu().tolist()]
    work = algorithmic_work(wl, kept)

    K = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev_f = [[mk(), mk()] for _ in range(K)]
    evs = [[mk() for _ in range(4)] for _ in range(K)]
    ev_w = [[mk(), mk()] for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device())
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        for s in range(K):
            flush.fill_(s & 0xFF)
            ev_f[s][0].record(stream)
            graphs["forward"].replay()
            ev_f[s][1].record(stream)
            flush.fill_((s + 1) & 0xFF)
            evs[s][0].record(stream)
            for j, name in enumerate(stages):
                graphs[name].replay()
                evs[s][j + 1].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    for s in range(K):  # warm L2: the same steps back to back, no flush
        ev_w[s][0].record(stream)
        graphs["forward"].replay()
        ev_w[s][1].record(stream)
    torch.cuda.synchronize(dev)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev_f]
    stage_ms = {name: [e[j].elapsed_time(e[j + 1]) for e in evs] for j, name in enumerate(stages)}
    warm_ms = [e[0].elapsed_time(e[1]) for e in ev_w]
    total_ms = slowest_rank_ms(sum(step_ms), world, dev)
    ms_per_step = total_ms / K
    pk, pk_kind = peaks()
    rec = {"workload": wl.name, "T": T, "d": d, "d_ff": wl.F, "E": E, "k": k,
           "capacity": wl.capacity, "routing": wl.routing, "overflow": wl.overflow,
           "value": job_tokens_per_s(world, T, K, total_ms), "unit": "tokens/s",
           "ms_per_step": ms_per_step, "ms_per_step_stats": _stats(step_ms),
           "tflops": work["flops"] / (ms_per_step * 1e-3) / 1e12 * world,
           "hbm_gbs_algorithmic": work["bytes"] / (ms_per_step * 1e-3) / 1e9 * world,
           "whole_call": {"algorithmic_bytes": work["bytes"], "algorithmic_flops": work["flops"],
                          "gbs": work["bytes"] / (ms_per_step * 1e-3) / 1e9,
                          "frac_of_measured_hbm": work["bytes"] / (ms_per_step * 1e-3) / 1e9
                          / pk["hbm_gbs"],
                          "frac_of_8tbs_nominal": work["bytes"] / (ms_per_step * 1e-3) / 8e12,
                          "frac_of_bf16_burst": work["flops"] / (ms_per_step * 1e-3) / 1e12
                          / pk["bf16_tflops"]},
           "warm_l2": {"ms_per_step": statistics.mean(warm_ms),
                       "ms_per_step_median": statistics.median(warm_ms),
                       "value": T * world / (statistics.mean(warm_ms) * 1e-3)},
           "kernels_per_step": kernels["forward"],
           "stages_ms": {name: statistics.mean(v) for name, v in stage_ms.items()},
           "stages_ms_median": {name: statistics.median(v) for name, v in stage_ms.items()},
           "kept_assignments": work["kept"], "experts_used": work["experts_used"],
           "roofline": (call_roofline(wl, work, ms_per_step, pk, pk_kind) if dense_decode(wl)
                        else ffn_roofline(wl, work, statistics.mean(stage_ms["expert_ffn"]), pk,
                                          pk_kind)),
           "gpu_launches": K * sum(kernels.values()) + (3 if e2e else 2) * K * kernels["forward"],
           "clocks": sampler.summary(),
           "l2": "flushed before every timed step and before every stage-graph step "
                 "(256 MiB write, untimed); warm_l2: no flush"}
    if e2e:
        rec["e2e"] = measure_e2e(args, wl, inp, layer, dev, stream, flush, world, dt)
    rec["_inputs"] = inp
    return rec


def measure_e2e(args, wl, inp, layer, dev, stream, flush, world, dt):
    """End to end through the host-buffer executor of the C ABI
    (moe_pipeline_*): per step the pinned host batch is copied in, the layer
    runs, y and the loss are copied out; neighbouring steps' copies overlap
    the forward pass."""
    import torch
    import torch.distributed as dist
    T, d, E = wl.T, wl.d, wl.E
    es = 2 if dt == torch.bfloat16 else 4
    x_np = inp.x.view(np.int16) if inp.x.dtype == np.uint16 else inp.x
    x_host = []
    for _ in range(2):
        t = torch.from_numpy(x_np.copy())
        x_host.append((t.view(torch.bfloat16) if inp.x.dtype == np.uint16 else t).pin_memory())
    y_host = [torch.empty((T, d), dtype=dt).pin_memory() for _ in range(2)]
    aux_host = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
    pipe = layer.host_pipeline(T, depth=2, stream=stream)
    # the expert weights are the data a step could find in L2 from the step
    # before; below twice the L2 size the L2 is flushed between steps (on the
    # compute stream, so inside the timed region)
    w_bytes = 2 * E * d * wl.F * es
    e2e_flush = w_bytes <= 2 * L2_BYTES
    for s in range(max(args.warmup, 3)):
        pipe.submit(x_host[s & 1], y_host[s & 1], aux_host[s & 1])
    pipe.join()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.join()  # the first input copy starts after e0
    for s in range(args.steps):
        if e2e_flush:
            flush.fill_(s & 0xFF)
        pipe.submit(x_host[s & 1], y_host[s & 1], aux_host[s & 1])
    pipe.join()
    e1.record(stream)
    e1.synchronize()
    e2e_ms = slowest_rank_ms(e0.elapsed_time(e1), world, dev)
    pipe.close()
    return {"value": job_tokens_per_s(world, T, args.steps, e2e_ms), "unit": "tokens/s",
            "ms_per_step": e2e_ms / args.steps,
            "h2d_bytes_per_step": T * d * es, "d2h_bytes_per_step": T * d * es + 4,
            "path": "moe_pipeline_submit (pinned host x in, y and loss out; copies of "
                    "neighbouring steps overlap the forward pass)",
            "l2": ("flushed before every step, inside the timed region" if e2e_flush
                   else f"not flushed: expert weights ({w_bytes / 2**20:.0f} MiB) exceed "
                        "twice the L2")}


def cpu_baselines(wl, inp, budget_s=10.0):
    """The oracle on the host cores, with every BLAS thread (this process) and
    single-threaded (a child process started with the BLAS and OpenMP thread
    counts set to 1), each on a token sample sized to about budget_s."""
    import subprocess
    rate, n, t, threads = cpu_oracle_rate(wl, inp, budget_s, probe=64)
    out = {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
           "sample": f"first {n} of {wl.T} tokens as a batch of their own, {t:.1f} s "
                     f"({threads} BLAS threads)",
           "host_cores": os.cpu_count()}
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-rate-only",
                            str(budget_s), "--workload", wl.name], env=env, capture_output=True,
                           text=True, timeout=20 * budget_s + 120)
        one = json.loads(r.stdout.strip().splitlines()[-1])
        out["single_thread"] = {"value": one["value"], "cores": one["cores"],
                                "sample": one["sample"]}
    except Exception as exc:  # the multi-threaded figure stands on its own
        out["single_thread"] = {"value": None, "error": f"{type(exc).__name__}: {exc}"[:200]}
    return out


def oracle_rate_only(args, wl):
    """--oracle-rate-only BUDGET: the oracle's tokens/s on a sample sized to
    BUDGET seconds, as one JSON line (the single-thread CPU baseline's child)."""
    inp = I.make_inputs(wl, seed=0)
    rate, n, t, threads = cpu_oracle_rate(wl, inp, args.oracle_rate_only, probe=16)
    print(json.dumps({"value": rate, "cores": threads,
                      "sample": f"first {n} of {wl.T} tokens as a batch of their own, {t:.1f} s"}))
    return 0


PER_CONFIG = ("bf16-T4096-d1024-F4096-E8-top2", "switch-bf16-T32768-d2048-F8192-E64-top1-cap640",
              "decode-bf16-T64-d4096-F14336-E8-top2")


def bench_ours(args, wl):
    import torch
    import torch.distributed as dist

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    rec = measure_workload(args, wl, dev, stream, flush, world)
    inp = rec.pop("_inputs")
    line = {"metric": METRIC, "value": rec["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": rec["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "d_ff": wl.F, "E": wl.E,
                       "k": wl.k, "capacity": wl.capacity, "routing": wl.routing,
                       "overflow": wl.overflow, "parallelism": f"replicas{world}",
                       "l2": rec["l2"]}}
    for key in ("ms_per_step_stats", "tflops", "hbm_gbs_algorithmic", "whole_call", "warm_l2",
                "kernels_per_step", "stages_ms", "stages_ms_median", "kept_assignments",
                "roofline", "e2e", "gpu_launches", "clocks"):
        line[key] = rec[key]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baselines(wl, inp)
    del inp
    if args.per_config and wl.name == DEFAULT_WORKLOAD:
        # the other graded workloads, device-timed the same way (no CPU baseline)
        per = {}
        for name in PER_CONFIG:
            torch.cuda.empty_cache()
            r = measure_workload(args, I.WORKLOADS[name], dev, stream, flush, world)
            r.pop("_inputs")
            per[name] = {key: r[key] for key in (
                "value", "unit", "ms_per_step", "ms_per_step_stats", "tflops",
                "hbm_gbs_algorithmic", "whole_call", "warm_l2", "stages_ms", "stages_ms_median",
                "kept_assignments", "experts_used", "roofline", "e2e", "kernels_per_step",
                "clocks")}
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def kept_per_expert(cfg, wl, D, dev):
    """Rows each expert keeps on this batch (the stage calls' offsets)."""
    import torch
    from sparse_mixture_experts_71_b300 import binding as B
    T, E, d = wl.T, wl.E, wl.d
    ec = wl.routing == "expert"
    k = wl.k + wl.n_shared
    n = max(E * B.expert_choice_capacity(cfg) if ec else T * k, 1)
    i32, f32 = torch.int32, torch.float32
    kr = B.ranked_columns(cfg)
    ws = B.workspace(cfg, device=dev)
    offsets = torch.empty(E + 1, dtype=i32, device=dev)
    slot_of = torch.empty((T, E if ec else k), dtype=i32, device=dev)
    perm_token = torch.empty(n, dtype=i32, device=dev)
    perm_w = torch.empty(n, dtype=f32, device=dev)
    x_perm = torch.empty((n, d), dtype=D["x"].dtype, device=dev)
    if ec:
        B.route_expert_choice(cfg, D["x"], D["W_r"], offsets, perm_token, perm_w, slot_of, ws,
                              x_perm=x_perm, logit_bias=D["logit_bias"])
    else:
        idx = torch.empty((T, kr), dtype=i32, device=dev)
        w = torch.empty((T, kr), dtype=f32, device=dev)
        B.route(cfg, D["x"], D["W_r"], idx, w, ws, logit_bias=D["logit_bias"])
        B.dispatch(cfg, D["x"], idx, offsets, slot_of, perm_token, x_perm, ws, topk_w=w,
                   perm_w=perm_w)
    torch.cuda.synchronize(dev)
    return [int(v) for v in torch.diff(offsets).cpu().tolist()]


def backward_roofline(wl, achieved, kernels, pk, pk_kind, clocks):
    """bf16 layers: the whole call's GEMM flops against the measured bf16
    burst peak.  fp32 layers run every product as fp32 FMA on the CUDA cores:
    against 148 SMs x 128 fp32 lanes x 2 flop x the SM clock (the maximum
    the clock sampler reports, 2032 MHz if none)."""
    roof = {"kernel": f"whole backward call ({kernels} launches)", "achieved": achieved,
            "unit": "TFLOP/s", "traffic": None}
    if wl.dtype == "bf16":
        roof.update(bound="tensor", peak=pk["bf16_tflops"], peak_source=pk_kind + " burst")
    else:
        mhz = (clocks or {}).get("sm_max_mhz") or 2032.0
        roof.update(bound="alu", peak=148 * 128 * 2 * mhz * 1e6 / 1e12,
                    peak_source=f"148 SMs x 128 fp32 FMA lanes x 2 flop x {mhz:.0f} MHz")
    roof["frac"] = achieved / roof["peak"]
    return roof


def bench_backward(args, wl):
    """One step = one moe_backward call (it recomputes the forward
    intermediates it needs) on the workload's inputs and a seeded dy."""
    import torch
    import torch.distributed as dist
    from sparse_mixture_experts_71_b300 import binding as B
    from sparse_mixture_experts_71_b300.layer import MoELayer, capture_graph, device_inputs

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    inp = I.make_inputs(wl, seed=0)
    D = device_inputs(inp, dev)
    layer = MoELayer(D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], k=wl.k, capacity=wl.capacity,
                     renormalize=wl.renormalize, logit_bias=D["logit_bias"], routing=wl.routing,
                     overflow=wl.overflow, n_shared=wl.n_shared)
    cfg = layer.config(wl.T)
    T, d, F, E = wl.T, wl.d, wl.F, wl.E
    ws = B.backward_workspace(cfg, device=dev)
    dy = torch.from_numpy(I.router_noise(T, d, 1.0, seed=1)).to(D["x"].dtype).to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dx=torch.empty_like(D["x"]), dW_r=torch.empty(tuple(D["W_r"].shape), **f32),
             dW1=torch.empty((E, F, d), **f32), db1=torch.empty((E, F), **f32),
             dW2=torch.empty((E, d, F), **f32), db2=torch.empty((E, d), **f32))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(st):
        B.backward(cfg, D["x"], D["W_r"], D["W1"], D["b1"], D["W2"], D["b2"], dy, g["dx"],
                   g["dW_r"], g["dW1"], g["db1"], g["dW2"], g["db2"], ws,
                   logit_bias=D["logit_bias"], aux_grad=0.01, z_grad=0.001, stream=st)

    c0 = B.launch_count()
    step(stream)
    torch.cuda.synchronize(dev)
    kernels = B.launch_count() - c0
    graph = capture_graph(step, warmup=1)
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        graph.replay()
    torch.cuda.synchronize(dev)
    kept = sum(kept_per_expert(cfg, wl, D, dev))  # kept assignments of this batch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with sampler:
        for s_ in range(args.steps):
            flush.fill_(s_ & 0xFF)
            ev[s_][0].record(stream)
            graph.replay()
            ev[s_][1].record(stream)
        torch.cuda.synchronize(dev)
    total_ms = slowest_rank_ms(sum(e0.elapsed_time(e1) for e0, e1 in ev), world, dev)
    ms = total_ms / args.steps
    # the GEMMs the call runs: the first forward GEMM recomputed (bf16 layers
    # take the slot scores from the dH product's epilogue; fp32 layers also
    # recompute the second), dH, dX and the two weight-gradient GEMMs; the
    # router's logits, dx and dW_r products over the routed experts
    gemms = 5 if wl.dtype == "bf16" else 6
    flops = gemms * 2.0 * kept * d * F + 3 * 2.0 * T * d * (E - wl.n_shared)
    pk, pk_kind = peaks()
    clocks = sampler.summary()
    achieved = flops / (ms * 1e-3) / 1e12
    line = {"metric": "MoE-layer backward tokens/s (gradients of x, W_r, W1, b1, W2, b2)",
            "value": job_tokens_per_s(world, T, 1, ms), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if wl.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "pass": "backward", "T": T, "d": d, "d_ff": F,
                       "E": E, "k": wl.k, "capacity": wl.capacity,
                       "routing": wl.routing, "overflow": wl.overflow,
                       "n_shared": wl.n_shared, "parallelism": f"replicas{world}",
                       "l2": "flushed before every timed step (256 MiB write, untimed)"},
            "kernels_per_step": kernels, "kept_assignments": kept,
            "roofline": backward_roofline(wl, achieved, kernels, pk, pk_kind, clocks),
            "gpu_launches": kernels * args.steps, "clocks": clocks}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(I.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="skip the per_config block (the other graded workloads)")
    ap.add_argument("--oracle-rate-only", type=float, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--pass", dest="pass_", choices=("forward", "backward"), default="forward",
                    help="backward: time moe_backward instead of the forward pass")
    args = ap.parse_args()
    wl = I.WORKLOADS[args.workload]
    if args.oracle_rate_only is not None:
        return oracle_rate_only(args, wl)
    if args.impl == "reference":
        return bench_reference(args, wl)
    if args.pass_ == "backward":
        return bench_backward(args, wl)
    return bench_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
