"""Benchmark of the fused-linear JSD forward + backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload headline]
    python bench.py --impl reference ...   # the float64 CPU oracle on host cores

One step is fljsd_forward + fljsd_backward (upstream gradient 1) over one batch
of synthetic inputs resident in HBM: both logits GEMMs, the three passes over
the vocabulary, grad_input and grad_weight, the loss reduction and the
backward scaling. Prints one JSON line (rank 0). Under torchrun each rank runs
an independent replica on its own GPU (the loss shards by rows, but this build
runs replicas only: no collective), and the value is the tokens all ranks
processed divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused-linear-JSD fwd+bwd tokens/s at H=4096,V=128256 bf16; % bf16 TC roofline"
# The pages' own number for this workload (H100 80GB HBM3, BT=8192, one chunk,
# 60.62 ms per full pass): context on another machine, not the target.
PAGES_MS_ONE_CHUNK = 60.62


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


GEMM_SOURCES = ("gemm_tc.cuh", "gemm_tc_kernel.cuh", "gemm_tc.cu", "gemm_tc_kk.cu",
                "gemm_tc_kmn.cu", "gemm_tc_mnmn.cu", "gemm_tc_mnk.cu")
ROWS_SOURCES = ("rows.cu", "jsd_math.cuh")


def sources_hash(sources) -> str | None:
    """First 16 hex digits of the SHA-256 of the named kernel sources, in order."""
    import hashlib

    h = hashlib.sha256()
    try:
        for name in sources:
            h.update(open(os.path.join(ROOT, "lm_head_jsd_gb300", "csrc", name), "rb").read())
    except OSError:
        return None
    return h.hexdigest()[:16]


def _profiled_traffic(kernel: str, sources, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    figures (profiles/dram_traffic.json), or None when there are none for that
    workload or the kernel's sources have changed since the counters were
    taken."""
    h = sources_hash(sources)
    if h is None:
        return None
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel, {}).get(workload)
    if not e or e.get("source_sha256_16") != h:
        return None
    return int(e["traffic_bytes_per_launch"])


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []
        self._t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._t = threading.Thread(target=self._read, daemon=True)
        self._t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self._t:
            self._t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def _gpu_index(torch, dev) -> str:
    """nvidia-smi identifier of the device: its PCI address when torch exposes
    it, else its index among the visible devices."""
    try:
        pr = torch.cuda.get_device_properties(dev)
        return f"{int(pr.pci_domain_id):08X}:{int(pr.pci_bus_id):02X}:{int(pr.pci_device_id):02X}.0"
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        return vis.split(",")[dev.index or 0]
    return str(dev.index or 0)


# ---------------------------------------------------------------------------
# multi-rank host logic (replicas: no collective on the data path)
# ---------------------------------------------------------------------------
def reduce_max(value: float, dist, device) -> float:
    """Largest `value` over all ranks (the slowest replica's time)."""
    if dist is None:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world: int, bt: int, ms_per_step: float) -> float:
    """Tokens all replicas processed per second: each rank runs the full batch."""
    return world * bt / (ms_per_step / 1e3)


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of the same workload
# ---------------------------------------------------------------------------
def cpu_baseline(w, x_s, w_s, x_t, w_t, labels, budget_s: float, block: int = 16):
    """Times the float64 oracle, as it stands, on blocks of rows of the workload
    until about `budget_s` seconds of CPU work; returns tokens (rows) / s."""
    import numpy as np

    import oracle

    f64 = lambda t: t.detach().cpu().double().numpy()  # noqa: E731
    ws64, wt64 = f64(w_s), f64(w_t)
    lab = None if labels is None else labels.cpu().numpy()
    rows_done, elapsed = 0, 0.0
    r0 = 0
    while elapsed < budget_s and r0 < w.bt:
        r1 = min(w.bt, r0 + block)
        xs, xt = f64(x_s[r0:r1]), f64(x_t[r0:r1])
        lb = None if lab is None else lab[r0:r1]
        t0 = time.perf_counter()
        oracle.fljsd_ref(xs, ws64, xt, wt64, lb, beta=w.beta, temperature=w.temperature,
                         reduction=w.reduction)
        elapsed += time.perf_counter() - t0
        rows_done += r1 - r0
        r0 = r1
    del ws64, wt64
    cores = os.cpu_count()
    try:
        from threadpoolctl import threadpool_info

        cores = max((i.get("num_threads", 0) for i in threadpool_info()), default=cores) or cores
    except Exception:
        pass
    return {"value": rows_done / elapsed, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{rows_done} of {w.bt} rows of the {w.name} workload in blocks of {block} "
                      f"(full V={w.v}, H_s={w.h_s}, H_t={w.h_t}), float64 NumPy, "
                      f"{elapsed:.1f} s"}


# ---------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="headline")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--chunk-rows", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline field (0 disables)")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--ref-rows", type=int, default=16,
                    help="rows per step of the reference (oracle) arm")
    ap.add_argument("--ce-bt", type=int, default=8192,
                    help="rows of the cross-entropy path (--path flce)")
    ap.add_argument("--path", default="fljsd", choices=["fljsd", "jsd_logspace", "tvd", "flce"],
                    help="fljsd: the fused-linear JSD (the headline); the others measure the "
                         "distance kernels over given distributions")
    args = ap.parse_args()
    if args.path == "flce":
        return run_flce_bench(args)
    if args.path != "fljsd":
        return run_dist_bench(args)

    import torch

    import jsd_inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    w = jsd_inputs.WORKLOADS[args.workload]

    if args.impl == "reference":
        if rank != 0:
            return 0
        return run_reference(args, w, world)

    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)

    import lm_head_jsd_gb300 as fl
    from lm_head_jsd_gb300 import FusedLinearJSD

    x_s, w_s, x_t, w_t, labels = jsd_inputs.make_inputs(w, str(dev))
    run = FusedLinearJSD(w.bt, w.h_s, w.h_t, w.v, w.torch_dtype, beta=w.beta,
                         temperature=w.temperature, reduction=w.reduction,
                         chunk_rows=args.chunk_rows, device=dev)
    loss, gi, gw = run.alloc_outputs()
    one = torch.ones(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        run.forward(x_s, w_s, x_t, w_t, labels, out=(loss, gi, gw), stream=stream)
        run.backward(one, gi, gw, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)

    # ---- timed region ----
    clocks = ClockSampler(_gpu_index(torch, dev))
    fl.fljsd_trace_enable(args.steps * (5 * run.plan.num_chunks + 4) + 16)
    fl.fljsd_trace_reset()
    n_launch0 = fl.fljsd_launch_count()
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    clk = clocks.stop()
    launches = fl.fljsd_launch_count() - n_launch0
    peak_bytes = torch.cuda.max_memory_allocated(dev)
    ms_total = ev0.elapsed_time(ev1)
    kinds = {}
    for k in ("gemm_logits", "jsd_rows", "gemm_grad_input", "gemm_grad_weight", "small"):
        kinds[k] = fl.fljsd_trace_read(k)
    fl.fljsd_trace_enable(0)
    status = fl.fljsd_workspace_status(run.plan, run.workspace, stream)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    ms_total = reduce_max(ms_total, dist, dev)
    ms_step = ms_total / args.steps
    value = whole_job_tokens_per_s(world, w.bt, ms_step)

    # ---- roofline of the dominant kernel (the tensor-core GEMM) ----
    peaks = _peaks()
    gemm_ms = sum(kinds[k][0] for k in ("gemm_logits", "gemm_grad_input", "gemm_grad_weight"))
    gemm_n = sum(kinds[k][1] for k in ("gemm_logits", "gemm_grad_input", "gemm_grad_weight"))
    flop_step = w.flops()
    steps_traced = gemm_n / (4 * run.plan.num_chunks) if gemm_n else 0
    gemm_flop_per_launch = flop_step / (4 * run.plan.num_chunks)
    gemm_avg_ms = gemm_ms / gemm_n if gemm_n else float("nan")
    achieved = gemm_flop_per_launch / (gemm_avg_ms / 1e3) / 1e12
    # each GEMM launch lasts a few ms inside a step of tens of ms: the burst
    # peak is the denominator (the sustained one is given beside it)
    peak_tc = peaks["bf16_tflops"]
    peak_sus = peaks["bf16_tflops_sustained"]
    s = 2 if w.dtype == "bf16" else 4
    jsd_ms, jsd_n = kinds["jsd_rows"]
    jsd_bytes = 3 * w.bt * w.v * s / run.plan.num_chunks  # read Z_s, Z_t once; write dZ once
    jsd_gbs = jsd_bytes / (jsd_ms / jsd_n / 1e3) / 1e9 if jsd_n else float("nan")
    step_roof_ms = max(flop_step / (peak_tc * 1e12), 11 * w.bt * w.v * s / (peaks["hbm_gbs"] * 1e9)) * 1e3

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": round(value / (w.bt / (PAGES_MS_ONE_CHUNK / 1e3)), 3)
        if w.name == "headline" else None,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{w.name}: BT={w.bt} H_s={w.h_s} H_t={w.h_t} V={w.v} {w.dtype} "
                               f"beta={w.beta} T={w.temperature} {w.reduction}",
                   "global_batch": w.bt * world, "seq_len": None,
                   "parallelism": f"replicas{world}" if world > 1 else "single",
                   "chunk_rows": int(run.plan.chunk_rows), "num_chunks": int(run.plan.num_chunks),
                   "l2": "inputs larger than L2 (W_s, W_t 1 GB each; logits buffers "
                         f"{run.plan.logits_bytes / 1e9:.1f} GB)"},
        "roofline": {"bound": "tensor", "kernel": "k_gemm_tc (4 launches per chunk)",
                     "achieved": round(achieved, 1), "peak": peak_tc, "unit": "TFLOP/s",
                     "frac": round(achieved / peak_tc, 4),
                     "traffic": _profiled_traffic("k_gemm_tc", GEMM_SOURCES, w.name),
                     "peak_kind": f"bf16 burst ({peaks['source']})",
                     "frac_of_sustained": round(achieved / peak_sus, 4)},
        "roofline_step": {"flop": flop_step, "roofline_ms": round(step_roof_ms, 3),
                          "frac": round(step_roof_ms / ms_step, 4),
                          "peak": f"bf16 burst {peak_tc} TFLOP/s ({peaks['source']})",
                          "frac_of_sustained": round(
                              step_roof_ms * peak_tc / peak_sus / ms_step, 4)},
        "roofline_jsd": {"bound": "hbm", "achieved": round(jsd_gbs, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(jsd_gbs / peaks["hbm_gbs"], 4),
                         "algorithmic_bytes": "3*C*V*s per launch",
                         "traffic": _profiled_traffic("k_jsd_rows", ROWS_SOURCES, w.name)},
        "kernel_ms_per_step": {k: round(v[0] / max(steps_traced, 1), 4) for k, v in kinds.items()},
        "gpu_launches": launches,
        "clocks": clk,
        "peak_device_memory": {
            "bytes": int(peak_bytes), "gb": round(peak_bytes / 1e9, 3),
            "what": "torch allocator peak through the timed region: inputs, outputs and the "
                    "planned workspace (the library itself allocates nothing)"},
    }
    if args.e2e_steps > 0:
        out["e2e"] = run_e2e(torch, run, w, x_s, w_s, x_t, w_t, labels, args.e2e_steps, dist,
                             world, dev)
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        out["cpu_baseline"] = cpu_baseline(w, x_s, w_s, x_t, w_t, labels, args.cpu_budget)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def run_e2e(torch, run, w, x_s, w_s, x_t, w_t, labels, steps, dist, world, dev):
    """The same step through the public API with the per-step inputs (hidden
    states and labels) in pinned host memory, as a training loop runs it: the
    inputs of step i + 1 are copied host -> device on a second stream into the
    other of two device buffers while step i computes, and the loss of every
    step is copied back and read on the host (one step behind the launches).
    The timed region spans every copy and ends when the last loss is on the
    host. The lm_head weights stay resident (they are parameters, not per-step
    inputs)."""
    hx_s = x_s.cpu().pin_memory()
    hx_t = x_t.cpu().pin_memory()
    hlab = None if labels is None else labels.cpu().pin_memory()
    nloss = run.alloc_outputs()[0].numel()
    host_loss = [torch.empty(nloss, dtype=torch.float32).pin_memory() for _ in range(2)]
    dx_s = [torch.empty_like(x_s) for _ in range(2)]
    dx_t = [torch.empty_like(x_t) for _ in range(2)]
    dlab = [None if labels is None else torch.empty_like(labels) for _ in range(2)]
    loss, gi, gw = run.alloc_outputs()
    one = torch.ones(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event() for _ in range(2)]   # inputs of buffer b are on the device
    consumed = [torch.cuda.Event() for _ in range(2)]  # the step reading buffer b is done
    landed = [torch.cuda.Event() for _ in range(2)]   # the loss of the step is on the host
    seen = []

    def copy_in(b):
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(consumed[b])
            dx_s[b].copy_(hx_s, non_blocking=True)
            dx_t[b].copy_(hx_t, non_blocking=True)
            if hlab is not None:
                dlab[b].copy_(hlab, non_blocking=True)
            copied[b].record(copy_stream)

    def compute(b):
        stream.wait_event(copied[b])
        run.forward(dx_s[b], w_s, dx_t[b], w_t, dlab[b], out=(loss, gi, gw), stream=stream)
        run.backward(one, gi, gw, stream=stream)
        consumed[b].record(stream)
        host_loss[b].copy_(loss.view(-1), non_blocking=True)
        landed[b].record(stream)

    def loop(n):
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in((i + 1) % 2)
            compute(i % 2)
            if i >= 1:  # the previous step's loss, read on the host
                landed[(i - 1) % 2].synchronize()
                seen.append(float(host_loss[(i - 1) % 2][0]))
        landed[(n - 1) % 2].synchronize()
        seen.append(float(host_loss[(n - 1) % 2][0]))

    for b in range(2):  # the first wait on a never-recorded event is a no-op
        consumed[b].record(stream)
    loop(2)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    seen.clear()
    t0 = time.perf_counter()
    loop(steps)
    ms = reduce_max((time.perf_counter() - t0) * 1e3 / steps, dist, dev)
    if len(seen) != steps or not all(v == v for v in seen):
        raise RuntimeError("e2e: a step's loss did not come back")
    h2d = hx_s.numel() * hx_s.element_size() + hx_t.numel() * hx_t.element_size() + (
        0 if hlab is None else hlab.numel() * 8)
    return {"value": round(whole_job_tokens_per_s(world, w.bt, ms), 1), "unit": "tokens/s",
            "ms_per_step": round(ms, 4), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": nloss * 4,
            "what": "pinned-host X_s, X_t, labels -> device every step on a copy stream, "
                    "double-buffered so that step i+1's copy overlaps step i; fljsd_forward + "
                    "fljsd_backward; every step's loss -> host and read there (one step behind); "
                    "grad_input and grad_weight stay on the device (training continues there); "
                    "the lm_head weights are resident parameters; wall clock from the first "
                    "copy to the last loss on the host"}


def run_dist_bench(args):
    """Time one distance kernel (log-space JSD or TVD) on a [rows x V] bf16
    problem larger than L2; HBM roofline on 3 * rows * V * 2 bytes (read two
    tensors, write the gradient)."""
    import torch

    import jsd_inputs
    from lm_head_jsd_gb300 import _lib

    # TVD: the shape the tie-fix page timed (4096 x 32000 bf16); log-space JSD:
    # the fused path's BT x V.
    rows, v = (4096, 32000) if args.path == "tvd" else (8192, 128256)
    dev = torch.device("cuda", 0)
    a, b, _ = jsd_inputs.make_distributions(rows, v, "bf16", 100, logspace=args.path != "tvd",
                                            device=str(dev))
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    grad = torch.empty_like(a)
    ws = torch.empty(_lib.fljsd_rows_workspace_bytes(rows), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        if args.path == "tvd":
            _lib.fljsd_tvd(rows, v, "bf16", "batchmean", -100, a, b, None, loss, grad, ws,
                           stream=stream)
        else:
            _lib.fljsd_jsd_logspace(rows, v, "bf16", 0.5, "batchmean", -100, a, b, None, loss,
                                    grad, ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        call()
    torch.cuda.synchronize(dev)
    _lib.fljsd_trace_enable(4 * args.steps + 8)
    _lib.fljsd_trace_reset()
    n0 = _lib.fljsd_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        call()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / args.steps
    k_ms, k_n = _lib.fljsd_trace_read("jsd_rows")
    _lib.fljsd_trace_enable(0)
    peaks = _peaks()
    bytes_ = 3 * rows * v * 2
    kern_ms = k_ms / max(k_n, 1)
    gbs = bytes_ / (kern_ms / 1e3) / 1e9
    name = "TVD fwd+bwd" if args.path == "tvd" else "log-space JSD fwd+bwd"
    print(json.dumps({
        "metric": f"{name} rows/s at ({rows}, {v}) bf16", "value": round(rows / (ms / 1e3), 1),
        "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.path}: rows={rows} V={v} bf16 batchmean",
                   "l2": "inputs larger than L2"},
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": None,
                     "algorithmic_bytes": "3*rows*V*2 per call"},
        "gpu_launches": _lib.fljsd_launch_count() - n0}), flush=True)
    return 0


def run_flce_bench(args):
    """Fused linear cross-entropy fwd+bwd at BT=8192, H=4096, V=128256 bf16,
    reduction mean -- the shape of the grad_weight page's FLCE table (its H100
    figure, 37.34 ms, is context on another machine). Tensor-core roofline on
    6 * BT * V * H FLOPs."""
    import torch

    import jsd_inputs
    import lm_head_jsd_gb300 as fl
    from lm_head_jsd_gb300 import FusedLinearCrossEntropy

    bt, h, v = args.ce_bt, 4096, 128256
    dev = torch.device("cuda", 0)
    x, w, labels = jsd_inputs.make_ce_inputs(bt, h, v, "bf16", 200, device=str(dev))
    run = FusedLinearCrossEntropy(bt, h, v, torch.bfloat16, chunk_rows=args.chunk_rows,
                                  device=dev)
    loss, gi, gw = run.alloc_outputs()
    one = torch.ones(1, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        run.forward(x, w, labels, out=(loss, gi, gw), stream=stream)
        fl.fljsd_scale("bf16", gi, gi.numel(), one, stream=stream)
        fl.fljsd_scale("bf16", gw, gw.numel(), one, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    fl.fljsd_trace_enable(args.steps * (4 * run.plan.num_chunks + 4) + 16)
    fl.fljsd_trace_reset()
    n0 = fl.fljsd_launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    ms = ev0.elapsed_time(ev1) / args.steps
    kinds = {k: fl.fljsd_trace_read(k) for k in
             ("gemm_logits", "jsd_rows", "gemm_grad_input", "gemm_grad_weight", "small")}
    fl.fljsd_trace_enable(0)
    peaks = _peaks()
    flop = 6.0 * bt * v * h
    g_ms = sum(kinds[k][0] for k in ("gemm_logits", "gemm_grad_input", "gemm_grad_weight"))
    g_n = sum(kinds[k][1] for k in ("gemm_logits", "gemm_grad_input", "gemm_grad_weight"))
    achieved = (flop / 3) / (g_ms / g_n / 1e3) / 1e12 if g_n else float("nan")
    # GEMM launches of a few ms inside the step: the burst peak is the
    # denominator, the sustained one is given beside it
    peak = peaks["bf16_tflops"]
    peak_sus = peaks["bf16_tflops_sustained"]
    # the row kernel reads the logits once and writes dlogits over them (the
    # GEMM epilogue's per-128-column partials, 8 bytes each, come on top)
    r_ms, r_n = kinds["jsd_rows"]
    rows_bytes = (2 * bt * v * 2 + bt * ((v + 127) // 128) * 8) / run.plan.num_chunks
    rows_gbs = rows_bytes / (r_ms / r_n / 1e3) / 1e9 if r_n else float("nan")
    peak_bytes = torch.cuda.max_memory_allocated(dev)
    print(json.dumps({
        "metric": "fused-linear cross-entropy fwd+bwd tokens/s at H=4096,V=128256 bf16",
        "value": round(bt / (ms / 1e3), 1), "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"flce: BT={bt} H={h} V={v} bf16 mean",
                   "chunk_rows": int(run.plan.chunk_rows)},
        "roofline": {"bound": "tensor", "kernel": "k_gemm_tc (3 launches per chunk)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "peak_kind": f"bf16 burst ({peaks['source']})",
                     "frac_of_sustained": round(achieved / peak_sus, 4)},
        "roofline_step": {"flop": flop, "frac": round(flop / (peak * 1e12) * 1e3 / ms, 4),
                          "peak": f"bf16 burst {peak} TFLOP/s ({peaks['source']})"},
        "roofline_rows": {"bound": "hbm", "kernel": "k_ce_rows", "achieved": round(rows_gbs, 1),
                          "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": round(rows_gbs / peaks["hbm_gbs"], 4),
                          "algorithmic_bytes": "2*C*V*s (logits read, dlogits written) "
                                               "+ 8 bytes per row per 128 columns"},
        "kernel_ms_per_step": {k: round(t / args.steps, 4) for k, (t, _) in kinds.items()},
        "gpu_launches": fl.fljsd_launch_count() - n0,
        "peak_device_memory": {"bytes": int(peak_bytes), "gb": round(peak_bytes / 1e9, 3)}}),
        flush=True)
    return 0


def run_reference(args, w, world):
    """The reference arm: the float64 CPU oracle, as it stands, on the host cores,
    each step a bounded sample of `--ref-rows` rows of the same workload."""
    import numpy as np

    import jsd_inputs
    import oracle

    import torch

    # the same draw as the native arm (a CUDA generator when a GPU is present)
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    x_s, w_s, x_t, w_t, labels = (None if t is None else t.cpu()
                                  for t in jsd_inputs.make_inputs(w, gen_dev))
    f64 = lambda t: t.detach().double().numpy()  # noqa: E731
    ws64, wt64 = f64(w_s), f64(w_t)
    lab = None if labels is None else labels.numpy()
    rows = args.ref_rows

    def step(i):
        r0 = (i * rows) % max(1, x_s.shape[0] - rows + 1)
        oracle.fljsd_ref(f64(x_s[r0:r0 + rows]), ws64, f64(x_t[r0:r0 + rows]), wt64,
                         None if lab is None else lab[r0:r0 + rows], beta=w.beta,
                         temperature=w.temperature, reduction=w.reduction)

    for i in range(max(args.warmup, 1)):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    sec = time.perf_counter() - t0
    ms = sec * 1e3 / args.steps
    value = rows / (ms / 1e3)
    cores = os.cpu_count()
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
           "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 1),
           "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": f"{w.name}: BT={w.bt} H_s={w.h_s} H_t={w.h_t} V={w.v} {w.dtype} "
                                  f"beta={w.beta} T={w.temperature} {w.reduction}",
                      "rows_per_step": rows},
           "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                            "kind": "oracle",
                            "sample": f"{rows} rows per step of the {w.name} workload "
                                      f"(full V and H), float64 NumPy"},
           "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
