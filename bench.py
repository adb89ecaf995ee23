#!/usr/bin/env python
"""Benchmark of the dynamic short convolution on GB300.

Metric: fwd+bwd tokens/s and achieved HBM GB/s (fraction of the measured HBM
roofline).  One step = one forward (dsc_fwd) and one backward (dsc_bwd) pass
over one batch of the head-wise bf16 workload (B=8, T=2048, D=2048, W=4,
H=16: Q/K/V-sized activations at about 2B-model width, the shape on which the
pages quote their head-wise kernel) with inputs resident in HBM.  L2 is
flushed (512 MiB write) between timed steps, outside the timed events.

Prints ONE JSON line on rank 0.  Multi-GPU (torchrun) runs one independent
replica per GPU ("weak" scaling; the path shards by batch with no exchange).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this method
has) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dyn-conv fwd+bwd tokens/s and achieved HBM GB/s (% of GB300 roofline)"
UNIT = "tokens/s"
MAIN_WORKLOAD = "headwise_bf16"
FLUSH_BYTES = 512 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=MAIN_WORKLOAD)
    ap.add_argument("--no-rows", action="store_true", help="skip the per-workload table")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    return ap.parse_args()


# ----------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "dynamic_short_convolution_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


DENSE_BWD_SRC = ["dsc_dense_bwd.cu", "dsc_dense_common.cuh", "dsc_device.cuh"]
DENSE_FWD_SRC = ["dsc_dense_fwd.cu", "dsc_dense_common.cuh", "dsc_device.cuh"]


def measured_traffic(kernel, workload, digest):
    """DRAM bytes per launch from the committed ncu summary, if the kernel is unchanged since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
            return int(parts[3]) if parts[2] == digest else None
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while a region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        return self

    def summary(self, t0, t1):
        if self.proc is None:
            return None
        rows = []
        for ts, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((ts, float(f[1]), float(f[2]), f))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [r for r in rows if t0 <= r[0] <= t1] or rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for n, v in zip(names, r[3][5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside),
                "samples_in_timed_region": sum(1 for r in rows if t0 <= r[0] <= t1)}


# ----------------------------------------------------------------- workloads on the GPU

class DenseProblem:
    def __init__(self, wl, dev):
        import torch

        from dynamic_short_convolution_gb300 import inputs

        self.wl = wl
        d = inputs.make(wl)
        self.host = d
        g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
        self.x, self.w, self.dy, self.cu = g["x"], g["w"], g["dy"], g["cu_seqlens"]
        self.y = torch.empty_like(self.x)
        self.dx = torch.empty_like(self.x)
        self.dw = torch.empty_like(self.w)
        es = self.x.element_size()
        xb, wb = self.x.numel() * es, self.w.numel() * es
        cb = 0 if self.cu is None else self.cu.numel() * 4
        self.bytes_fwd = 2 * xb + wb + cb
        self.bytes_bwd = 3 * xb + 2 * wb + cb
        self.flops_fwd = self.flops_bwd = 0

    def fwd(self):
        import dynamic_short_convolution_gb300 as dsc

        dsc.dsc_fwd(self.x, self.w, self.y, cu_seqlens=self.cu)

    def bwd(self):
        import dynamic_short_convolution_gb300 as dsc

        dsc.dsc_bwd(self.x, self.w, self.dy, self.dx, self.dw, cu_seqlens=self.cu)


class LowrankProblem:
    def __init__(self, wl, dev):
        import torch

        from dynamic_short_convolution_gb300 import inputs

        self.wl = wl
        d = inputs.make(wl)
        self.host = d
        g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
        self.x, self.z, self.U, self.b, self.dy, self.cu = g["x"], g["z"], g["U"], g["bias"], g["dy"], g["cu_seqlens"]
        self.y = torch.empty_like(self.x)
        self.dx = torch.empty_like(self.x)
        self.dz = torch.empty_like(self.z)
        self.dU = torch.empty(self.U.shape, dtype=torch.float32, device=dev)
        self.db = torch.empty(self.b.shape, dtype=torch.float32, device=dev)
        import dynamic_short_convolution_gb300 as dsc

        nb = dsc.dsc_lowrank_bwd_workspace_bytes(wl.B, wl.T, wl.D, wl.W, wl.R)
        self.ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
        es = 2
        xb, zb, ub = self.x.numel() * es, self.z.numel() * es, self.U.numel() * es
        nw = wl.D * wl.W
        self.bytes_fwd = 2 * xb + zb + ub + 4 * nw
        self.bytes_bwd = 3 * xb + 2 * zb + ub + 4 * nw + 4 * wl.R * nw + 4 * nw
        m = wl.B * wl.T
        self.flops_fwd = 2 * m * nw * wl.R
        self.flops_bwd = 3 * 2 * m * nw * wl.R  # filter recompute + dz + dU

    def fwd(self):
        import dynamic_short_convolution_gb300 as dsc

        dsc.dsc_lowrank_fwd(self.x, self.z, self.U, self.b, self.y, cu_seqlens=self.cu)

    def bwd(self):
        import dynamic_short_convolution_gb300 as dsc

        dsc.dsc_lowrank_bwd(self.x, self.z, self.U, self.b, self.dy, self.dx, self.dz, self.dU, self.db, self.ws,
                            cu_seqlens=self.cu)


def make_problem(wl, dev):
    return LowrankProblem(wl, dev) if wl.kind == "lowrank" else DenseProblem(wl, dev)


def time_steps(prob, flush, steps):
    """Per-step device times (ms) of fwd, bwd and both, each step after an L2 flush."""
    import torch

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1, e2 in ev:
        flush.zero_()
        e0.record()
        prob.fwd()
        e1.record()
        prob.bwd()
        e2.record()
    torch.cuda.synchronize()
    f = [a.elapsed_time(b) for a, b, _ in ev]
    b = [b_.elapsed_time(c) for _, b_, c in ev]
    return f, b


# ----------------------------------------------------------------- CPU oracle arm

def oracle_tokens_per_s(wl, budget_s, min_tokens=64):
    """fp64 oracle fwd+bwd on a token range of the workload, grown until it takes about budget_s."""
    import oracle
    from dynamic_short_convolution_gb300 import inputs

    d = inputs.make(wl)
    oracle.build()
    BT = wl.B * wl.T
    n = min_tokens
    spent, done = 0.0, 0
    # calibrate on a short range, then run one range sized for the budget
    t0 = time.perf_counter()
    _oracle_step(oracle, wl, d, 0, n)
    dt = time.perf_counter() - t0
    per_tok = dt / n
    n2 = int(max(min_tokens, min(BT, (budget_s - dt) / max(per_tok, 1e-9))))
    t1 = time.perf_counter()
    _oracle_step(oracle, wl, d, 0, n2)
    spent = time.perf_counter() - t1
    done = n2
    return done / spent, done, spent


def _oracle_step(oracle, wl, d, r0, r1):
    if wl.kind == "lowrank":
        oracle.lowrank_fwd(d["x"], d["z"], d["U"], d["bias"], wl.W, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        oracle.lowrank_bwd(d["x"], d["z"], d["U"], d["bias"], d["dy"], wl.W, cu_seqlens=d["cu_seqlens"],
                           rows=(r0, r1), want=("dx", "dz"))
    else:
        oracle.fwd(d["x"], d["w"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        oracle.bwd(d["x"], d["w"], d["dy"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, wl, rank, world):
    if rank != 0:
        return 0
    import oracle
    from dynamic_short_convolution_gb300 import inputs

    d = inputs.make(wl)
    oracle.build()
    BT = wl.B * wl.T
    # size each step's sample so warm-up + steps take about two minutes
    t0 = time.perf_counter()
    _oracle_step(oracle, wl, d, 0, 64)
    per_tok = (time.perf_counter() - t0) / 64
    budget = 120.0 / max(args.steps + args.warmup, 1)
    n = int(max(16, min(BT, budget / max(per_tok, 1e-9))))
    for i in range(args.warmup):
        r0 = (i * n) % max(BT - n, 1)
        _oracle_step(oracle, wl, d, r0, r0 + n)
    times = []
    for i in range(args.steps):
        r0 = (i * 7919 * n) % max(BT - n, 1)
        t = time.perf_counter()
        _oracle_step(oracle, wl, d, r0, r0 + n)
        times.append(time.perf_counter() - t)
    total = sum(times)
    value = n * args.steps / total
    cores = host_cores()
    sample = f"{n} consecutive tokens (all {wl.D} channels) of {wl.name} per step, fwd + bwd"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, world):
    shape = f"B={wl.B} T={wl.T} D={wl.D} W={wl.W}" + (f" R={wl.R}" if wl.kind == "lowrank" else f" H={wl.H}")
    return {"workload": f"{wl.name}: {shape}" + (" packed documents" if wl.packed else ""),
            "global_batch": wl.B * world, "seq_len": wl.T, "parallelism": "replicas (one independent batch per GPU)",
            "l2": "flushed between timed steps (512 MiB write, outside the timed events)"}


# ----------------------------------------------------------------- main arm

def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from dynamic_short_convolution_gb300 import inputs

    wl = inputs.by_name(args.workload)
    if args.impl == "reference":
        return run_reference(args, wl, rank, world)

    # the CPU baseline first, before any GPU work (rank 0, single GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, n, spent = oracle_tokens_per_s(wl, budget_s=12.0)
        cpu = {"value": v, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{n} consecutive tokens (all {wl.D} channels) of {wl.name}, fwd + bwd, {spent:.1f} s"}

    import torch
    import torch.distributed as dist

    import dynamic_short_convolution_gb300 as dsc

    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    dsc.lib()

    def barrier():
        if world > 1:
            dist.barrier()

    hbm_peak, tc_peak, tc_sust, peak_src = peaks()
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    prob = make_problem(wl, dev)

    for _ in range(args.warmup):
        flush.zero_()
        prob.fwd()
        prob.bwd()
    torch.cuda.synchronize()
    if dsc.dsc_sync_status() != 0:
        raise RuntimeError("device status word set during warm-up")

    sampler = ClockSampler(dev.index) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier()
    torch.cuda.synchronize()
    launches0 = dsc.dsc_launch_count()
    t_wall0 = time.perf_counter()
    f_ms, b_ms = time_steps(prob, flush, args.steps)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.perf_counter()
    launches = dsc.dsc_launch_count() - launches0
    if sampler:
        sampler.stop()
    if dsc.dsc_sync_status() != 0:
        raise RuntimeError("device status word set during the timed region")

    step_ms = [a + b for a, b in zip(f_ms, b_ms)]
    total_ms = sum(step_ms)
    if world > 1:
        t = torch.tensor([total_ms], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    tokens = wl.B * wl.T
    value = world * tokens * args.steps / (total_ms / 1e3)
    mean_f, mean_b = statistics.fmean(f_ms), statistics.fmean(b_ms)
    step_bytes = prob.bytes_fwd + prob.bytes_bwd
    step_gbs = step_bytes / (total_ms / args.steps / 1e3) / 1e9

    # roofline of the dominant kernel
    if mean_b >= mean_f:
        kname, kbytes, kms, ksrc = "dense_bwd_tma", prob.bytes_bwd, mean_b, DENSE_BWD_SRC
    else:
        kname, kbytes, kms, ksrc = "dense_fwd_tma", prob.bytes_fwd, mean_f, DENSE_FWD_SRC
    achieved = kbytes / (kms / 1e3) / 1e9
    traffic = measured_traffic(kname, wl.name, kernel_source_digest(ksrc))
    roof = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": traffic, "algorithmic_bytes": kbytes,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src}

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(prob, flush, max(10, min(args.steps // 10, 200)), dev, world)

    rows = None
    if rank == 0 and world == 1 and not args.no_rows:
        rows = measure_rows(dev, flush, hbm_peak, tc_peak)

    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": workload_config(wl, world),
            "hbm_gbs": step_gbs, "hbm_frac": step_gbs / hbm_peak,
            "fwd_us": 1e3 * mean_f, "bwd_us": 1e3 * mean_b,
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
            "rows": rows,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def measure_e2e(prob, flush, steps, dev, world):
    """The same metric through the public API with pinned host buffers: every step copies the inputs
    host->device, runs fwd+bwd, and copies the results device->host, all inside the timed events."""
    import torch

    import torch.distributed as dist

    wl = prob.wl
    names_in = ["x", "w", "dy"] if wl.kind != "lowrank" else ["x", "z", "U", "bias", "dy"]
    names_out = ["y", "dx", "dw"] if wl.kind != "lowrank" else ["y", "dx", "dz", "dU", "db"]
    h_in = {n: prob.host[n].pin_memory() for n in names_in}
    h_out = {n: torch.empty(getattr(prob, n).shape, dtype=getattr(prob, n).dtype, pin_memory=True)
             for n in names_out}
    dev_in = {"x": prob.x, "dy": prob.dy}
    if wl.kind == "lowrank":
        dev_in.update({"z": prob.z, "U": prob.U, "bias": prob.b})
    else:
        dev_in["w"] = prob.w
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    times = []
    for i in range(steps + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for n in names_in:
            dev_in[n].copy_(h_in[n], non_blocking=True)
        prob.fwd()
        prob.bwd()
        for n in names_out:
            h_out[n].copy_(getattr(prob, n), non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        if i >= 3:
            times.append(e0.elapsed_time(e1))
    total = sum(times)
    if world > 1:
        t = torch.tensor([total], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total = float(t.item())
    value = world * wl.B * wl.T * steps / (total / 1e3)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": total / steps, "steps": steps,
            "api": "dynamic_short_convolution_gb300.dsc_fwd / dsc_bwd (or dsc_lowrank_*) on pinned host copies"}


def measure_rows(dev, flush, hbm_peak, tc_peak):
    """Every workload, timed the same way (fewer steps): fwd / bwd device time and roofline fractions."""
    import torch

    import dynamic_short_convolution_gb300 as dsc
    from dynamic_short_convolution_gb300 import inputs

    out = {}
    for wid, wl in inputs.WORKLOADS.items():
        try:
            prob = make_problem(wl, dev)
            for _ in range(3):
                flush.zero_()
                prob.fwd()
                prob.bwd()
            torch.cuda.synchronize()
            f, b = time_steps(prob, flush, 50)
        except dsc.DscError as e:
            out[wl.name] = {"status": str(e)}
            continue
        mf, mb = statistics.median(f), statistics.median(b)
        r = {"fwd_us": 1e3 * mf, "bwd_us": 1e3 * mb, "tokens_per_s": wl.B * wl.T / ((mf + mb) / 1e3),
             "fwd_gbs": prob.bytes_fwd / mf / 1e6, "bwd_gbs": prob.bytes_bwd / mb / 1e6,
             "fwd_bytes": prob.bytes_fwd, "bwd_bytes": prob.bytes_bwd}
        r["fwd_hbm_frac"] = r["fwd_gbs"] / hbm_peak
        r["bwd_hbm_frac"] = r["bwd_gbs"] / hbm_peak
        r["fwdbwd_hbm_frac"] = (prob.bytes_fwd + prob.bytes_bwd) / ((mf + mb) / 1e3) / 1e9 / hbm_peak
        if prob.flops_fwd:
            r["fwd_tflops"] = prob.flops_fwd / mf / 1e9
            r["bwd_tflops"] = prob.flops_bwd / mb / 1e9
            # bound: the slower of the HBM and tensor-core times for the algorithmic bytes and flops
            tb = (prob.bytes_fwd + prob.bytes_bwd) / (hbm_peak * 1e9)
            tt = (prob.flops_fwd + prob.flops_bwd) / (tc_peak * 1e12)
            r["bound_us"] = 1e6 * max(tb, tt)
            r["roofline_frac"] = r["bound_us"] / (1e3 * (mf + mb))
        else:
            r["bound_us"] = 1e6 * (prob.bytes_fwd + prob.bytes_bwd) / (hbm_peak * 1e9)
            r["roofline_frac"] = r["fwdbwd_hbm_frac"]
        out[wl.name] = r
        del prob
        torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    sys.exit(main())
