#!/usr/bin/env python
"""Benchmark of the dynamic short convolution on GB300.

Metric: fwd+bwd tokens/s and achieved HBM GB/s (fraction of the measured HBM
roofline).  One step = one forward (dsc_fwd) and one backward (dsc_bwd) pass
over one batch of the largest single-GPU workload, the Q/K/V placement over
packed documents (B=4, T=8192, D=3072 = Q, K and V of a 2048-wide model side by
side, W=4, head size H=16, document lengths ~U{128..4096}), with inputs
resident in HBM.  Steps run back to back and rotate over independent copies
of the workload's tensors (at least 600 MB together, several times the 129 MB
L2), so every step reads inputs that are not in L2 and each kernel pays for
its own write-backs.  Every other workload (head-wise, materialised,
low-rank, static, decode) is timed the same way in the ``rows`` table, each
with its own roofline fraction and its own CPU-oracle baseline.

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
MAIN_WORKLOAD = "qkv_packed_bf16"
ROTATE_BYTES = 600 << 20  # minimum bytes across the rotating copies


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
    ap.add_argument("--row", default=None, help="only measure this one row of the per-workload table and print it")
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
LOWRANK_BWD_SRC = ["dsc_lowrank_bwd.cu", "dsc_lowrank_bwd_du.cu", "dsc_lowrank_common.cuh", "dsc_tcgen05.cuh",
                   "dsc_device.cuh"]
LOWRANK_FWD_SRC = ["dsc_lowrank_fwd.cu", "dsc_lowrank_epi.cuh", "dsc_lowrank_common.cuh", "dsc_tcgen05.cuh", "dsc_device.cuh"]
STATIC_SRC = ["dsc_static.cu", "dsc_dense_common.cuh", "dsc_device.cuh"]
# (kernel name in the ncu launch list, source files) per workload kind and direction
KERNELS = {("dense", "bwd"): ("dense_bwd_tma", DENSE_BWD_SRC), ("dense", "fwd"): ("dense_fwd_tma", DENSE_FWD_SRC),
           ("lowrank", "bwd"): ("lowrank_bwd_dxdz+lowrank_bwd_dudb", LOWRANK_BWD_SRC),
           ("lowrank", "fwd"): ("lowrank_fwd_tc", LOWRANK_FWD_SRC),
           ("static", "bwd"): ("static_bwd_tma", STATIC_SRC), ("static", "fwd"): ("static_fwd_tma", STATIC_SRC)}


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

class _Sets:
    """Independent copies of one workload's device tensors; step i uses copy i % n."""

    def __init__(self, tensors: dict, per_copy_bytes: int, min_copies: int = 2):
        import torch

        n = max(min_copies, -(-ROTATE_BYTES // max(per_copy_bytes, 1)))
        self.n = n
        self.sets = [tensors] + [{k: (v.clone() if isinstance(v, torch.Tensor) else v) for k, v in tensors.items()}
                                 for _ in range(n - 1)]
        self.i = 0

    def next(self):
        s = self.sets[self.i % self.n]
        self.i += 1
        return s


class DenseProblem:
    def __init__(self, wl, dev):
        import torch

        from dynamic_short_convolution_gb300 import inputs

        self.wl = wl
        d = inputs.make(wl)
        self.host = d
        g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
        t = {"x": g["x"], "w": g["w"], "dy": g["dy"], "cu": g["cu_seqlens"], "y": torch.empty_like(g["x"]),
             "dx": torch.empty_like(g["x"]), "dw": torch.empty_like(g["w"])}
        es = g["x"].element_size()
        xb, wb = g["x"].numel() * es, g["w"].numel() * es
        cb = 0 if g["cu_seqlens"] is None else g["cu_seqlens"].numel() * 4
        self.bytes_fwd = 2 * xb + wb + cb
        self.bytes_bwd = 3 * xb + 2 * wb + cb
        self.flops_fwd = self.flops_bwd = 0
        self.rot = _Sets(t, 4 * xb + 2 * wb)
        self.cur = t

    def __getattr__(self, name):  # the current copy's tensors (x, w, dy, y, dx, dw)
        cur = self.__dict__.get("cur")
        if cur is not None and name in cur:
            return cur[name]
        raise AttributeError(name)

    def advance(self):
        self.cur = self.rot.next()

    def fwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_fwd(c["x"], c["w"], c["y"], cu_seqlens=c["cu"])

    def bwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_bwd(c["x"], c["w"], c["dy"], c["dx"], c["dw"], cu_seqlens=c["cu"])


class LowrankProblem:
    def __init__(self, wl, dev):
        import torch

        import dynamic_short_convolution_gb300 as dsc
        from dynamic_short_convolution_gb300 import inputs

        self.wl = wl
        d = inputs.make(wl)
        self.host = d
        g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
        nb = dsc.dsc_lowrank_bwd_workspace_bytes(wl.B, wl.T, wl.D, wl.W, wl.R)
        t = {"x": g["x"], "z": g["z"], "U": g["U"], "bias": g["bias"], "dy": g["dy"], "cu": g["cu_seqlens"],
             "y": torch.empty_like(g["x"]), "dx": torch.empty_like(g["x"]), "dz": torch.empty_like(g["z"]),
             "dU": torch.empty(g["U"].shape, dtype=torch.float32, device=dev),
             "db": torch.empty(g["bias"].shape, dtype=torch.float32, device=dev),
             "ws": torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)}
        es = 2
        xb, zb, ub = g["x"].numel() * es, g["z"].numel() * es, g["U"].numel() * es
        nw = wl.D * wl.W
        self.bytes_fwd = 2 * xb + zb + ub + 4 * nw
        self.bytes_bwd = 3 * xb + 2 * zb + ub + 4 * nw + 4 * wl.R * nw + 4 * nw
        m = wl.B * wl.T
        self.flops_fwd = 2 * m * nw * wl.R
        self.flops_bwd = 3 * 2 * m * nw * wl.R  # filter recompute + dz + dU
        self.rot = _Sets(t, 4 * xb + 3 * zb)
        self.cur = t

    def __getattr__(self, name):
        cur = self.__dict__.get("cur")
        if cur is not None and name in cur:
            return cur[name]
        raise AttributeError(name)

    def advance(self):
        self.cur = self.rot.next()

    def fwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_lowrank_fwd(c["x"], c["z"], c["U"], c["bias"], c["y"], cu_seqlens=c["cu"])

    def bwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_lowrank_bwd(c["x"], c["z"], c["U"], c["bias"], c["dy"], c["dx"], c["dz"], c["dU"], c["db"],
                            c["ws"], cu_seqlens=c["cu"])


class StaticProblem:
    """The static short convolution: one filter w [D, W] for every token; dw fp32 [D, W]."""

    def __init__(self, wl, dev):
        import torch

        from dynamic_short_convolution_gb300 import inputs

        self.wl = wl
        d = inputs.make(wl)
        self.host = d
        g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
        t = {"x": g["x"], "w": g["w"], "dy": g["dy"], "cu": g["cu_seqlens"], "y": torch.empty_like(g["x"]),
             "dx": torch.empty_like(g["x"]), "dw": torch.empty((wl.D, wl.W), dtype=torch.float32, device=dev)}
        xb = g["x"].numel() * g["x"].element_size()
        wb = g["w"].numel() * g["w"].element_size()
        cb = 0 if g["cu_seqlens"] is None else g["cu_seqlens"].numel() * 4
        self.bytes_fwd = 2 * xb + wb + cb
        self.bytes_bwd = 3 * xb + wb + 4 * wl.D * wl.W + cb
        self.flops_fwd = self.flops_bwd = 0
        self.rot = _Sets(t, 4 * xb)
        self.cur = t

    def __getattr__(self, name):
        cur = self.__dict__.get("cur")
        if cur is not None and name in cur:
            return cur[name]
        raise AttributeError(name)

    def advance(self):
        self.cur = self.rot.next()

    def fwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_static_fwd(c["x"], c["w"], c["y"], cu_seqlens=c["cu"])

    def bwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_static_bwd(c["x"], c["w"], c["dy"], c["dx"], c["dw"], cu_seqlens=c["cu"])


class DecodeProblem:
    """One decode step of B sequences (inference: no backward).  The algorithmic bytes count x, w, the
    history rows each token's document actually has (min(pos, W-1) of them), y, and the one ring slot
    written."""

    def __init__(self, wl, dev):
        import torch

        from dynamic_short_convolution_gb300 import inputs

        self.wl = wl
        d = inputs.make(wl)
        self.host = d
        g = {k: v.to(dev) for k, v in d.items()}
        t = {"x": g["x"], "w": g["w"], "hist": g["hist"], "pos": g["pos"], "y": torch.empty_like(g["x"])}
        es = g["x"].element_size()
        row = wl.D * es
        hist_rows = int(torch.clamp(d["pos"].long(), max=wl.W - 1).sum())
        self.bytes_fwd = (2 * wl.B * row + g["w"].numel() * es + hist_rows * row + (wl.B * row if wl.W > 1 else 0)
                          + wl.B * 4)
        self.bytes_bwd = 0
        self.flops_fwd = self.flops_bwd = 0
        self.rot = _Sets(t, 2 * wl.B * row + g["hist"].numel() * es)
        self.cur = t

    def __getattr__(self, name):
        cur = self.__dict__.get("cur")
        if cur is not None and name in cur:
            return cur[name]
        raise AttributeError(name)

    def advance(self):
        self.cur = self.rot.next()

    def fwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_decode_step(c["x"], c["w"], c["hist"], c["pos"], c["y"])

    def bwd(self):
        pass


class ProjProblem:
    """The projection with the convolution in its epilogue (forward only): h [B,T,Dm] and the weights in,
    y out.  Algorithmic bytes: h read once, the weights once, y written once; flops: 2 B T Dm (D + (D/H) W).
    ``unfused`` runs the same computation as a caller without the fused kernel would: cuBLAS GEMMs that
    store x and w (bf16; the generator bias added in the GEMM), then dsc_fwd."""

    def __init__(self, wl, dev):
        import torch

        from dynamic_short_convolution_gb300 import inputs

        self.wl = wl
        d = inputs.make(wl)
        self.host = d
        g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
        Dm = g["h"].shape[-1]
        NG = g["Wg"].shape[0]
        BT = wl.B * wl.T
        t = {"h": g["h"], "Wx": g["Wx"], "Wg": g["Wg"], "bg": g["bg"], "cu": g["cu_seqlens"],
             "y": torch.empty(wl.B, wl.T, wl.D, dtype=torch.bfloat16, device=dev),
             "x": torch.empty(wl.B, wl.T, wl.D, dtype=torch.bfloat16, device=dev),
             "w": torch.empty(wl.B, wl.T, wl.D // wl.H, wl.W, dtype=torch.bfloat16, device=dev)}
        self.bg16 = g["bg"].to(torch.bfloat16)
        hb = g["h"].numel() * 2
        self.bytes_fwd = hb + (g["Wx"].numel() + g["Wg"].numel()) * 2 + 4 * NG + BT * wl.D * 2
        self.bytes_bwd = 0
        self.flops_fwd = 2 * BT * Dm * (wl.D + NG)
        self.flops_bwd = 0
        self.Dm = Dm
        self.rot = _Sets({"h": t["h"]}, hb)  # only h is large; the weights stay in L2 as they would in a model
        self.t = t
        self.cur = t

    def advance(self):
        self.cur = dict(self.t, h=self.rot.next()["h"])

    def fwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_proj_fwd(c["h"], c["Wx"], c["Wg"], c["bg"], c["y"], W=self.wl.W, cu_seqlens=c["cu"])

    def unfused(self, ev=None):
        import torch

        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        h2 = c["h"].view(-1, self.Dm)
        torch.matmul(h2, c["Wx"].t(), out=c["x"].view(-1, self.wl.D))
        if ev:
            ev[0].record()
        torch.addmm(self.bg16, h2, c["Wg"].t(), out=c["w"].view(h2.shape[0], -1))
        if ev:
            ev[1].record()
        dsc.dsc_fwd(c["x"], c["w"], c["y"], cu_seqlens=c["cu"])

    def bwd(self):
        pass


class ZprojProblem:
    """The low-rank forward with the generator's first projection on chip (forward only): x, the layer input
    h and the weights in, y out.  Algorithmic bytes: x, h, W1, U and the bias read once, y written once;
    flops: the two projections, 2 B T R (Dm + D W).  ``unfused`` is the caller's path without the fused kernel:
    z = h W1^T + b1 by cuBLAS, stored bf16, then dsc_lowrank_fwd."""

    def __init__(self, wl, dev):
        import torch

        from dynamic_short_convolution_gb300 import inputs

        self.wl = wl
        d = inputs.make(wl)
        g = {k: (v.to(dev) if v is not None else None) for k, v in d.items()}
        BT = wl.B * wl.T
        Dm = g["h"].shape[-1]
        self.Dm = Dm
        t = {"x": g["x"], "h": g["h"], "W1": g["W1"], "b1": g["b1"], "U": g["U"], "bias": g["bias"], "cu": g["cu_seqlens"],
             "y": torch.empty(wl.B, wl.T, wl.D, dtype=torch.bfloat16, device=dev),
             "z": torch.empty(wl.B, wl.T, wl.R, dtype=torch.bfloat16, device=dev)}
        per = (g["x"].numel() + g["h"].numel()) * 2
        self.bytes_fwd = (per + (g["W1"].numel() + g["U"].numel()) * 2 + 4 * (g["bias"].numel() + g["b1"].numel())
                          + BT * wl.D * 2)
        self.bytes_bwd = 0
        self.flops_fwd = 2 * BT * wl.R * (Dm + wl.D * wl.W)
        self.flops_bwd = 0
        self.b1_16 = g["b1"].to(torch.bfloat16)
        self.rot = _Sets({"x": t["x"], "h": t["h"]}, per)
        self.t = t
        self.cur = t

    def advance(self):
        self.cur = dict(self.t, **self.rot.next())

    def fwd(self):
        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        dsc.dsc_lowrank_zproj_fwd(c["x"], c["h"], c["W1"], c["U"], c["bias"], c["y"], b1=c["b1"], cu_seqlens=c["cu"])

    def unfused(self, ev=None):
        import torch

        import dynamic_short_convolution_gb300 as dsc

        c = self.cur
        torch.addmm(self.b1_16, c["h"].view(-1, self.Dm), c["W1"].t(), out=c["z"].view(-1, self.wl.R))
        if ev:
            ev[0].record()
        dsc.dsc_lowrank_fwd(c["x"], c["z"], c["U"], c["bias"], c["y"], cu_seqlens=c["cu"])

    def bwd(self):
        pass


def make_problem(wl, dev):
    return {"lowrank": LowrankProblem, "static": StaticProblem, "decode": DecodeProblem,
            "proj": ProjProblem, "zproj": ZprojProblem}.get(wl.kind, DenseProblem)(wl, dev)


def time_graph_replay(prob, steps):
    """Device time per forward call (ms) when `steps` calls (over the rotating copies) are recorded in one
    CUDA graph and replayed, as a serving loop runs them."""
    import torch

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(steps):
            prob.advance()
            prob.fwd()
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_steps_back_to_back(prob, steps):
    """Device time per fwd + bwd step (ms) for steps shorter than the host's launch path: every step is
    queued behind a GPU sleep first, then they run back to back between two events."""
    import torch

    torch.cuda._sleep(int(2e6) + steps * 120000)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        prob.advance()
        prob.fwd()
        prob.bwd()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_back_to_back(prob, steps):
    """Device time per forward call (ms) for a kernel shorter than the host's launch path: a GPU sleep
    lets the host queue every call first, then they run back to back between two events."""
    import torch

    torch.cuda._sleep(int(2e6) + steps * 60000)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        prob.advance()
        prob.fwd()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_steps(prob, steps):
    """Per-step device times (ms) of fwd and bwd; steps back to back on rotating input copies."""
    import torch

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps + 1)]
    ev[0].record()
    for i in range(steps):
        prob.advance()
        prob.fwd()
        ev[2 * i + 1].record()
        prob.bwd()
        ev[2 * i + 2].record()
    torch.cuda.synchronize()
    f = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)]
    b = [ev[2 * i + 1].elapsed_time(ev[2 * i + 2]) for i in range(steps)]
    return f, b


# ----------------------------------------------------------------- CPU oracle arm

def oracle_tokens_per_s(wl, budget_s, min_tokens=64):
    """fp64 oracle fwd+bwd over consecutive token ranges of the workload (wrapping around), until about
    budget_s of CPU time has been spent; returns (tokens/s, tokens, seconds)."""
    import oracle
    from dynamic_short_convolution_gb300 import inputs

    d = inputs.make(wl)
    oracle.build()
    BT = wl.B * wl.T
    t0 = time.perf_counter()
    _oracle_step(oracle, wl, d, 0, min_tokens)
    per_tok = (time.perf_counter() - t0) / min_tokens
    chunk = int(max(min_tokens, min(BT, 0.25 * budget_s / max(per_tok, 1e-9))))
    done, pos = 0, 0
    t1 = time.perf_counter()
    while True:
        n = min(chunk, BT - pos)
        _oracle_step(oracle, wl, d, pos, pos + n)
        done += n
        pos = (pos + n) % BT
        spent = time.perf_counter() - t1
        if spent >= budget_s:
            break
    return done / spent, done, spent


def _oracle_step(oracle, wl, d, r0, r1):
    """One fwd + bwd sample of the oracle: every per-token output over tokens [r0, r1), and, for the
    low-rank form, its parameter gradients dU and db (sums over every token) over the same fraction of
    their filter columns, so each output's share of the work matches the sample's share of the tokens."""
    if wl.kind == "static":
        oracle.static_fwd(d["x"], d["w"], wl.W, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        oracle.static_bwd(d["x"], d["w"], d["dy"], wl.W, cu_seqlens=d["cu_seqlens"], rows=(r0, r1), want_dw=False)
    elif wl.kind == "lowrank":
        oracle.lowrank_fwd(d["x"], d["z"], d["U"], d["bias"], wl.W, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        oracle.lowrank_bwd(d["x"], d["z"], d["U"], d["bias"], d["dy"], wl.W, cu_seqlens=d["cu_seqlens"],
                           rows=(r0, r1), want=("dx", "dz"))
        nw, BT = wl.D * wl.W, wl.B * wl.T
        c0 = (r0 * nw) // BT
        c1 = max(c0 + 1, (r1 * nw) // BT)
        oracle.lowrank_bwd(d["x"], d["z"], d["U"], d["bias"], d["dy"], wl.W, cu_seqlens=d["cu_seqlens"],
                           cols=list(range(c0, min(c1, nw))), want=("dU", "db"))
    elif wl.kind == "proj":  # the fused projection + convolution: forward rows [r0, r1) (no backward)
        oracle.proj_fwd(d["h"], d["Wx"], d["Wg"], d["bg"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
    elif wl.kind == "zproj":  # the low-rank forward with z from the layer input: rows [r0, r1) (no backward)
        oracle.lowrank_zproj_fwd(d["x"], d["h"], d["W1"], d["U"], d["bias"], wl.W, cu_seqlens=d["cu_seqlens"],
                                 rows=(r0, r1), b1=d["b1"])
    elif wl.kind == "decode":  # one decode step of sequences [r0, r1) (no backward: inference)
        oracle.decode_step(d["x"][r0:r1], d["w"][r0:r1], d["hist"][r0:r1], d["pos"][r0:r1], wl.W, wl.H)
    else:
        oracle.fwd(d["x"], d["w"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))
        oracle.bwd(d["x"], d["w"], d["dy"], wl.W, wl.H, cu_seqlens=d["cu_seqlens"], rows=(r0, r1))


def _omp_threads(n):
    """Set the OpenMP thread count of the oracle's parallel loops (the calling thread's setting)."""
    import ctypes

    try:
        ctypes.CDLL("libgomp.so.1").omp_set_num_threads(int(n))
        return True
    except OSError:
        return False


def cpu_rows(budget_s=2.5):
    """The oracle, as it stands, on a bounded sample of every workload (tokens/s on the host cores), and
    the tiny fp32 workload also on one thread.  Run before any GPU work."""
    from dynamic_short_convolution_gb300 import inputs

    out = {}
    cores = host_cores()
    for wl in inputs.WORKLOADS.values():
        v, n, spent = oracle_tokens_per_s(wl, budget_s=budget_s)
        r = {"cpu_tokens_per_s": v, "cpu_cores": cores,
             "cpu_sample": f"{n} tokens of {wl.name} in {spent:.1f} s" + ("" if wl.kind in ("decode", "proj", "zproj") else ", fwd + bwd")}
        if wl.wid == 1 and _omp_threads(1):
            v1, n1, s1 = oracle_tokens_per_s(wl, budget_s=budget_s)
            _omp_threads(cores)
            r.update({"cpu_tokens_per_s_1thread": v1, "cpu_sample_1thread": f"{n1} tokens in {s1:.1f} s on one thread"})
        out[wl.name] = r
    return out


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


def max_over_ranks(local_ms, world, device):
    """The job's time: the largest of the ranks' times (replicas run in lockstep, the slowest one decides)."""
    if world <= 1:
        return local_ms
    import torch
    import torch.distributed as dist

    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tokens_per_s(world, tokens_per_replica, steps, total_ms):
    """Tokens processed by all replicas together per second of the job's time (weak scaling)."""
    return world * tokens_per_replica * steps / (total_ms / 1e3)


def workload_config(wl, world):
    shape = f"B={wl.B} T={wl.T} D={wl.D} W={wl.W}" + (f" R={wl.R}" if wl.kind == "lowrank" else f" H={wl.H}")
    return {"workload": f"{wl.name}: {shape}" + (" packed documents" if wl.packed else ""),
            "global_batch": wl.B * world, "seq_len": wl.T, "parallelism": "replicas (one independent batch per GPU)",
            "l2": "inputs larger than L2: steps back to back over rotating copies of the tensors (>= 600 MB)"}


# ----------------------------------------------------------------- main arm

def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from dynamic_short_convolution_gb300 import inputs

    if args.row is not None:  # one row of the table alone (for profiling one workload's kernels)
        import torch

        inputs.by_name(args.row)
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        hbm_peak, tc_peak, _, _ = peaks()
        print(json.dumps({"rows": measure_rows(dev, hbm_peak, tc_peak, only=args.row)}), flush=True)
        return 0
    wl = inputs.by_name(args.workload)
    if wl.kind == "decode":
        raise SystemExit("the decode step has no backward pass: it is measured in the rows table only")
    if args.impl == "reference":
        return run_reference(args, wl, rank, world)

    # the CPU baseline first, before any GPU work (rank 0, single GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, n, spent = oracle_tokens_per_s(wl, budget_s=12.0)
        cpu = {"value": v, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{n} tokens (all {wl.D} channels; consecutive ranges of {wl.name}, wrapping) fwd + bwd "
                         f"in {spent:.1f} s"}
    crows = cpu_rows() if rank == 0 and world == 1 and not args.no_cpu and not args.no_rows else None

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
    prob = make_problem(wl, dev)

    for _ in range(args.warmup):
        prob.advance()
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
    f_ms, b_ms = time_steps(prob, args.steps)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.perf_counter()
    launches = dsc.dsc_launch_count() - launches0
    if sampler:
        sampler.stop()
    if dsc.dsc_sync_status() != 0:
        raise RuntimeError("device status word set during the timed region")

    step_ms = [a + b for a, b in zip(f_ms, b_ms)]
    total_ms = max_over_ranks(sum(step_ms), world, dev)
    value = whole_job_tokens_per_s(world, wl.B * wl.T, args.steps, total_ms)
    mean_f, mean_b = statistics.fmean(f_ms), statistics.fmean(b_ms)
    step_bytes = prob.bytes_fwd + prob.bytes_bwd
    step_gbs = step_bytes / (total_ms / args.steps / 1e3) / 1e9

    # roofline of the dominant kernel: HBM bytes, or tensor-core flops where those take longer at peak
    direction = "bwd" if mean_b >= mean_f else "fwd"
    kname, ksrc = KERNELS[(wl.kind if wl.kind in ("lowrank", "static") else "dense", direction)]
    kms = mean_b if direction == "bwd" else mean_f
    kbytes = prob.bytes_bwd if direction == "bwd" else prob.bytes_fwd
    kflops = prob.flops_bwd if direction == "bwd" else prob.flops_fwd
    traffic = measured_traffic(kname, wl.name, kernel_source_digest(ksrc))
    if kflops and kflops / (tc_peak * 1e12) > kbytes / (hbm_peak * 1e9):
        achieved = kflops / (kms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": kname, "achieved": achieved, "peak": tc_peak, "unit": "TFLOP/s",
                "frac": achieved / tc_peak, "traffic": traffic, "algorithmic_flops": kflops,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16_tflops)" if peak_src == "measured" else peak_src}
    else:
        achieved = kbytes / (kms / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": kname, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic, "algorithmic_bytes": kbytes,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else peak_src}

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(prob, max(10, min(args.steps // 10, 200)), dev, world)

    rows = None
    if rank == 0 and world == 1 and not args.no_rows:
        rows = measure_rows(dev, hbm_peak, tc_peak)
        for name, r in (crows or {}).items():
            if name in rows:
                rows[name].update(r)

    clocks = sampler.summary(t_wall0, t_wall1) if sampler else None
    if clocks is not None and clocks.get("samples_in_timed_region", 0) < 3:
        # the timed region was shorter than a few sampling periods: run the same steps again, untimed, for
        # about a second, and report the clocks seen there beside it
        chk = ClockSampler(dev.index)
        chk.start()
        c0 = time.perf_counter()
        while time.perf_counter() - c0 < 1.2:
            time_steps(prob, max(1, min(args.steps, 200)))
        torch.cuda.synchronize()
        c1 = time.perf_counter()
        chk.stop()
        clocks["same_steps_for_1s_after"] = chk.summary(c0, c1)
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


def measure_e2e(prob, steps, dev, world):
    """The same metric through the public API with pinned host buffers: every step copies its inputs
    host->device, runs fwd+bwd, and copies all of its results device->host, all inside the timed region.
    Steps are pipelined over the rotating device copies on three streams (inputs in, compute, results
    out), so step i's compute overlaps step i+1's input copies and step i-1's result copies."""
    import torch

    wl = prob.wl
    names_in = ["x", "w", "dy"] if wl.kind != "lowrank" else ["x", "z", "U", "bias", "dy"]
    names_out = ["y", "dx", "dw"] if wl.kind != "lowrank" else ["y", "dx", "dz", "dU", "db"]
    h_in = {n: prob.host[n].pin_memory() for n in names_in}
    h_out = {n: torch.empty(getattr(prob, n).shape, dtype=getattr(prob, n).dtype, pin_memory=True)
             for n in names_out}
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    s_comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nsets = prob.rot.n
    ev = lambda: torch.cuda.Event()  # noqa: E731
    comp_done = [None] * nsets  # compute of the last step that used copy k (its inputs are free after it)
    out_done = [None] * nsets   # result copies of the last step that used copy k (its outputs are free after)

    def step():
        k = prob.rot.i % prob.rot.n
        prob.advance()
        with torch.cuda.stream(s_in):
            if comp_done[k] is not None:
                s_in.wait_event(comp_done[k])
            for n in names_in:
                getattr(prob, n).copy_(h_in[n], non_blocking=True)
            in_ready = ev()
            in_ready.record(s_in)
        s_comp.wait_event(in_ready)
        if out_done[k] is not None:
            s_comp.wait_event(out_done[k])
        prob.fwd()
        prob.bwd()
        comp_done[k] = ev()
        comp_done[k].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[k])
            for n in names_out:
                h_out[n].copy_(getattr(prob, n), non_blocking=True)
            out_done[k] = ev()
            out_done[k].record(s_out)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(steps):
        step()
    s_in.wait_stream(s_out)
    e1.record(s_in)
    torch.cuda.synchronize(dev)
    total = max_over_ranks(e0.elapsed_time(e1), world, dev)
    value = whole_job_tokens_per_s(world, wl.B * wl.T, steps, total)
    return {"value": value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": total / steps, "steps": steps, "copy_sets": nsets,
            "api": "dynamic_short_convolution_gb300.dsc_fwd / dsc_bwd (or dsc_lowrank_*) on pinned host copies, "
                   "steps pipelined on three streams"}


def measure_proj_row(prob, hbm_peak, tc_peak, reps=30):
    """The fused projection + convolution against the unfused path, per call (CUDA events, medians)."""
    import torch

    wl = prob.wl
    for _ in range(3):
        prob.advance()
        prob.fwd()
        prob.unfused()
    torch.cuda.synchronize()
    fused, unf, gx, gw = [], [], [], []
    for _ in range(reps):
        prob.advance()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record()
        prob.fwd()
        e[1].record()
        u = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        prob.advance()
        u[0].record()
        prob.unfused(ev=u[1:3])
        u[3].record()
        torch.cuda.synchronize()
        fused.append(e[0].elapsed_time(e[1]))
        unf.append(u[0].elapsed_time(u[3]))
        gx.append(u[0].elapsed_time(u[1]))
        gw.append(u[1].elapsed_time(u[2]))
    mf, mu = statistics.median(fused), statistics.median(unf)
    tf = prob.flops_fwd / (mf / 1e3) / 1e12
    return {"fwd_us": 1e3 * mf, "tokens_per_s": wl.B * wl.T / (mf / 1e3), "fwd_tflops": tf,
            "tensor_frac": tf / tc_peak, "fwd_bytes": prob.bytes_fwd, "fwd_flops": prob.flops_fwd,
            "bound_us": 1e6 * max(prob.flops_fwd / (tc_peak * 1e12), prob.bytes_fwd / (hbm_peak * 1e9)),
            "roofline_frac": 1e6 * prob.flops_fwd / (tc_peak * 1e12) / (1e3 * mf),
            "unfused_us": 1e3 * mu, "unfused_gemm_x_us": 1e3 * statistics.median(gx),
            "unfused_gemm_w_us": 1e3 * statistics.median(gw),
            "unfused_conv_us": 1e3 * (mu - statistics.median(gx) - statistics.median(gw)),
            "speedup_vs_unfused": mu / mf,
            "unfused_path": "torch.matmul (cuBLAS) for x, torch.addmm for w with its bias, both stored bf16, then "
                            "dsc_fwd",
            "timing": f"median of {reps} calls, CUDA events, h rotated over copies larger than L2"}


def measure_zproj_row(prob, hbm_peak, tc_peak, reps=30):
    """The fused-code low-rank forward against the unfused path, per call (CUDA events, medians)."""
    import torch

    wl = prob.wl
    for _ in range(3):
        prob.advance()
        prob.fwd()
        prob.unfused()
    torch.cuda.synchronize()
    fused, unf, gz = [], [], []
    for _ in range(reps):
        prob.advance()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e[0].record()
        prob.fwd()
        e[1].record()
        u = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        prob.advance()
        u[0].record()
        prob.unfused(ev=u[1:2])
        u[2].record()
        torch.cuda.synchronize()
        fused.append(e[0].elapsed_time(e[1]))
        unf.append(u[0].elapsed_time(u[2]))
        gz.append(u[0].elapsed_time(u[1]))
    mf, mu = statistics.median(fused), statistics.median(unf)
    bound = max(prob.flops_fwd / (tc_peak * 1e12), prob.bytes_fwd / (hbm_peak * 1e9))
    return {"fwd_us": 1e3 * mf, "tokens_per_s": wl.B * wl.T / (mf / 1e3), "fwd_bytes": prob.bytes_fwd,
            "fwd_flops": prob.flops_fwd, "fwd_gbs": prob.bytes_fwd / mf / 1e6,
            "fwd_hbm_frac": prob.bytes_fwd / mf / 1e6 / hbm_peak, "bound_us": 1e6 * bound,
            "roofline_frac": 1e6 * bound / (1e3 * mf), "unfused_us": 1e3 * mu,
            "unfused_gemm_z_us": 1e3 * statistics.median(gz),
            "unfused_conv_us": 1e3 * (mu - statistics.median(gz)), "speedup_vs_unfused": mu / mf,
            "unfused_path": "torch.addmm (cuBLAS) for z = h W1^T + b1 stored bf16, then dsc_lowrank_fwd",
            "timing": f"median of {reps} calls, CUDA events, x and h rotated over copies larger than L2"}


def measure_rows(dev, hbm_peak, tc_peak, only=None):
    """Every workload (or the one named `only`), timed the same way (fewer steps): fwd / bwd device time and
    roofline fractions."""
    import torch

    import dynamic_short_convolution_gb300 as dsc
    from dynamic_short_convolution_gb300 import inputs

    out = {}
    for wid, wl in inputs.WORKLOADS.items():
        if only is not None and wl.name != only:
            continue
        try:
            prob = make_problem(wl, dev)
            for _ in range(3):
                prob.advance()
                prob.fwd()
                prob.bwd()
            torch.cuda.synchronize()
            if wl.kind in ("proj", "zproj"):
                out[wl.name] = (measure_proj_row if wl.kind == "proj" else measure_zproj_row)(prob, hbm_peak, tc_peak)
                del prob
                torch.cuda.empty_cache()
                continue
            if wl.kind == "decode":
                ms = time_back_to_back(prob, 200)
                gms = time_graph_replay(prob, 200)
                gbs = prob.bytes_fwd / ms / 1e6
                out[wl.name] = {"step_us": 1e3 * ms, "tokens_per_s": wl.B / (ms / 1e3), "fwd_bytes": prob.bytes_fwd,
                                "fwd_gbs": gbs, "fwd_hbm_frac": gbs / hbm_peak,
                                "bound_us": 1e6 * prob.bytes_fwd / (hbm_peak * 1e9), "roofline_frac": gbs / hbm_peak,
                                "timing": "200 steps queued behind a GPU sleep, back to back between two events",
                                "graph_step_us": 1e3 * gms, "graph_hbm_frac": prob.bytes_fwd / gms / 1e6 / hbm_peak,
                                "graph_timing": "the same 200 steps recorded in one CUDA graph, one replay timed"}
                del prob
                torch.cuda.empty_cache()
                continue
            f, b = time_steps(prob, 100)
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
        if (mf + mb) * 1e3 < 60.0:  # a step this short is host-bound between events: its device time too
            ms = time_steps_back_to_back(prob, 100)
            r["step_us_back_to_back"] = 1e3 * ms
            r["tokens_per_s_back_to_back"] = wl.B * wl.T / (ms / 1e3)
        out[wl.name] = r
        del prob
        torch.cuda.empty_cache()
    return out


if __name__ == "__main__":
    sys.exit(main())
