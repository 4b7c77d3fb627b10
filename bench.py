#!/usr/bin/env python
"""Benchmark of the mixed-precision cast-and-scale path on GB300.

One step = one pass of every row of the hot path over one batch of
synthetic inputs resident in HBM:
  * gs_unscale_check_update over the Llama-3-8B-shaped FP16 gradient list
    (290 tensors, 8,030,257,152 elements; a NaN planted on every 4th step),
  * fp8_quant_block E4M3 1x128 of a bf16 [16384, 8192] activation with
    outlier channels, then fp8_dequant of it back to bf16,
  * fp8_quant_block E4M3 128x128 of a bf16 8192x28672 weight,
  * fp8_quant_tensor E5M2 of a bf16 8192x28672 gradient.
value = algorithmic HBM bytes of the step / device time (GB/s).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--sweep] [--no-e2e] [--no-extra] [--only KERNEL]
Under torchrun (N > 1) every rank runs its own replica of the step on its
own GPU (no data-path collective); rank 0 prints one JSON line.
At N = 1 the line also carries, timed after the step and outside `value`:
`sweep` (the unscale and 1x128 quantiser at 1 MiB, 128 MiB, 2 GiB and
8 GiB) and `kernels_extra` (MXFP8 quantise / dequantise, delayed E5M2, the
norm form of the unscale, the master update, and the FP8 GEMM in TFLOP/s
against the FP8 tensor peak).
--impl reference times the CPU oracle on the host threads (the pages ship no
implementation); --sweep runs every point of the 1 MiB .. 8 GiB bandwidth
sweep; --only times one kernel alone.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "HBM GB/s (and % of GB300 peak) for grad unscale/inf-check and FP8 block quantise"
UNIT = "GB/s"
WORKLOAD = ("Llama-3-8B fp16 grad list unscale+check+update (290 tensors, 8.03e9 elems) + "
            "E4M3 1x128 quant/dequant of bf16 [16384,8192] activations + E4M3 128x128 quant of "
            "bf16 8192x28672 weights + E5M2 per-tensor quant of a bf16 8192x28672 gradient")
FALLBACK_HBM_GBS = 6800.0
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "unscale_check_update": ["unscale_check.cu", "gs_device.cuh", "gs_layout.h"],
    "quant_1x128": ["fp8_quant.cu", "gs_device.cuh", "gs_quant.cuh"],
    "dequant_1x128_bf16": ["fp8_dequant.cu", "gs_device.cuh"],
    "quant_128x128": ["fp8_quant.cu", "gs_device.cuh", "gs_quant.cuh"],
    "quant_tensor_e5m2": ["fp8_quant.cu", "gs_device.cuh", "gs_quant.cuh"],
}


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--sweep", action="store_true", help="bandwidth sweep 1 MiB..8 GiB (config 5)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--only", choices=ONLY_CASES,
                   help="time one kernel alone on a small case (for ncu captures)")
    p.add_argument("--no-extra", action="store_true",
                   help="skip the sweep points and the rows beyond the step after the step")
    return p.parse_args(argv)


# ---- multi-process plumbing ---------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_init(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend, init_method="env://")
    return dist if world > 1 else None


def aggregate(elapsed_s: float, units: float, dist=None, device=None) -> tuple[float, float]:
    """Max elapsed time over ranks and total units over ranks."""
    if dist is None:
        return elapsed_s, units
    import torch
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def host_memory_available(meminfo: str = None, cgroup: tuple = None):
    """Bytes of host memory still available to this process: MemAvailable
    from /proc/meminfo, capped by what the cgroup's memory limit leaves (v2
    or v1). None when neither can be read."""
    avail = None
    try:
        if meminfo is None:
            with open("/proc/meminfo") as f:
                meminfo = f.read()
        for line in meminfo.splitlines():
            if line.startswith("MemAvailable:"):
                avail = int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    pairs = [cgroup] if cgroup else [("/sys/fs/cgroup/memory.max", "/sys/fs/cgroup/memory.current"),
                                     ("/sys/fs/cgroup/memory/memory.limit_in_bytes",
                                      "/sys/fs/cgroup/memory/memory.usage_in_bytes")]
    for lim_f, cur_f in pairs:
        try:
            with open(lim_f) as f:
                lim = f.read().strip()
            with open(cur_f) as f:
                cur = int(f.read().strip())
        except (OSError, ValueError):
            continue
        if lim != "max" and int(lim) < (1 << 60):
            room = max(int(lim) - cur, 0)
            avail = room if avail is None else min(avail, room)
        break
    return avail


def e2e_fits(pinned_bytes: int, local_ranks: int, available) -> bool:
    """True when the pinned host buffers of every rank on this node take at
    most 60% of the host memory available (or when it cannot be read)."""
    return available is None or pinned_bytes * local_ranks <= 0.6 * available


def throughput(total_bytes: float, elapsed_s: float) -> float:
    return total_bytes / elapsed_s / 1e9


def link_ceiling(step_bytes: float, h2d_bytes: float, d2h_bytes: float, h2d_gbs: float,
                 d2h_gbs: float, both_gbs: float) -> float:
    """Best end-to-end rate the host link allows, in the metric's unit
    (algorithmic bytes of one step / the shortest time its copies can take):
    both directions share the link (each at half the measured concurrent
    total) until the smaller transfer is done, then the rest of the larger
    one runs alone at its own one-way rate."""
    each = both_gbs / 2.0
    common = min(h2d_bytes, d2h_bytes)
    rest, rest_gbs = (d2h_bytes - common, d2h_gbs) if d2h_bytes >= h2d_bytes else \
        (h2d_bytes - common, h2d_gbs)
    t = common / (each * 1e9) + rest / (rest_gbs * 1e9)
    return step_bytes / t / 1e9 if t > 0 else 0.0


def measure_link(torch, nbytes: int = 1 << 30, reps: int = 3) -> dict:
    """Pinned host <-> device copy rates on this machine (best of `reps`): one
    way each, and both at once on two streams."""
    d1 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d2 = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    h1 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h2 = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def best(fn, moved):
        ms = []
        for _ in range(reps):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            ms.append(time.perf_counter() - t0)
        return moved / min(ms) / 1e9

    def both():
        with torch.cuda.stream(s1):
            d1.copy_(h1, non_blocking=True)
        with torch.cuda.stream(s2):
            h2.copy_(d2, non_blocking=True)

    r = {"h2d_gbs": round(best(lambda: d1.copy_(h1, non_blocking=True), nbytes), 1),
         "d2h_gbs": round(best(lambda: h2.copy_(d2, non_blocking=True), nbytes), 1),
         "both_gbs": round(best(both, 2 * nbytes), 1)}
    del d1, d2, h1, h2
    return r


# ---- peaks, traffic, clocks --------------------------------------------------------

def fp8_peak(sustained: bool) -> tuple[float, str]:
    """Dense FP8 tensor peak: a measured bf16 GEMM rate x 2 (the nominal
    FP8 / bf16 ratio of the part) -- the sustained (power-capped) rate for a
    loop that runs for half a second or more, else the burst rate."""
    try:
        with open(PEAKS_FILE) as f:
            pk = json.load(f)
        key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
        return 2.0 * float(pk[key]), f"measured {key} x 2"
    except Exception:
        return 2.0 * (1700.0 if sustained else 1900.0), "fallback bf16 x 2"


def hbm_peak() -> tuple[float, str]:
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def sources_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "mixed_precision_numerics_gradscaler_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, or None if the
    kernel's sources changed since those counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)[kernel]
        return rec["dram_bytes_per_launch"] if rec["sources_sha"] == sources_sha(kernel) else None
    except Exception:
        return None


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        rows = []
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
            if len(parts) != 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), parts[3:]))
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r[2] > 300.0] or rows   # samples taken under load
        reasons = sorted({self.NAMES[i] for r in busy for i, v in enumerate(r[3]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy),
                "sm_max_mhz": max(r[1] for r in rows), "reasons": reasons,
                "samples": len(busy), "power_w_max": max(r[2] for r in rows)}


# ---- the step -------------------------------------------------------------------

class Workload:
    """Every buffer of one step, resident on the current GPU."""

    def __init__(self, gs, torch, small: bool = False):
        import datagen as dg
        from datagen import workloads as wl
        self.gs, self.torch, self.dg = gs, torch, dg
        dev = torch.device("cuda", torch.cuda.current_device())
        st = torch.cuda.current_stream().cuda_stream
        self.cfg2 = wl.cfg2_grads()
        f16, f32, bf16, u8 = torch.float16, torch.float32, torch.bfloat16, torch.uint8
        # the gradient list and its outputs as views into two flat buffers (one
        # host<->device copy each in the end-to-end loop)
        self.g_flat = torch.empty(self.cfg2.total, dtype=f16, device=dev)
        self.o_flat = torch.empty(self.cfg2.total, dtype=f32, device=dev)
        self.grads, self.outs = self._views(self.g_flat, self.o_flat)
        for t, (g, n) in enumerate(zip(self.grads, self.cfg2.numels)):
            dg.fill_device(self.cfg2.spec(t, 0), 0, n, g.data_ptr(), st)
        self.tl = gs.gs_tensor_list_create(self.grads, self.outs)
        self.scale = torch.tensor([self.cfg2.init_scale], dtype=f32, device=dev)
        self.tracker = torch.zeros(1, dtype=torch.int32, device=dev)
        self.found = torch.zeros(1, dtype=torch.int32, device=dev)
        self.skipped = torch.zeros(1, dtype=torch.int64, device=dev)
        a, w, g = wl.cfg3_act(), wl.cfg4_weight(), wl.cfg4_grad()
        self.x3 = torch.empty(a.rows, a.cols, dtype=bf16, device=dev)
        dg.fill_device(a.spec, 0, a.numel, self.x3.data_ptr(), st)
        self.q3 = torch.empty(a.rows, a.cols, dtype=u8, device=dev)
        self.s3 = torch.empty(a.rows, a.cols // 128, dtype=f32, device=dev)
        self.y3 = torch.empty(a.rows, a.cols, dtype=bf16, device=dev)
        self.x4 = torch.empty(w.rows, w.cols, dtype=bf16, device=dev)
        dg.fill_device(w.spec, 0, w.numel, self.x4.data_ptr(), st)
        self.q4 = torch.empty(w.rows, w.cols, dtype=u8, device=dev)
        self.s4 = torch.empty(w.rows // 128, w.cols // 128, dtype=f32, device=dev)
        self.x5 = torch.empty(g.numel, dtype=bf16, device=dev)
        dg.fill_device(g.spec, 0, g.numel, self.x5.data_ptr(), st)
        self.q5 = torch.empty(g.numel, dtype=u8, device=dev)
        self.s5 = torch.empty(1, dtype=f32, device=dev)
        self.ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=dev)
        # NaN planted on every 4th step at a seeded (tensor, index)
        t, i = self.cfg2.plant(4)
        self.plant_t, self.plant_i = t, i
        self.plant_ptr = self.grads[t].data_ptr() + 2 * i
        self.plant_orig = int(dg.fill_host_idx(self.cfg2.spec(t, 0), __import__("numpy").array([i]))[0])
        n2, n3, n4, n5 = self.cfg2.total, a.numel, w.numel, g.numel
        self.bytes = {
            "unscale_check_update": 6 * n2,
            "quant_1x128": 3 * n3 + 4 * (n3 // 128),
            "dequant_1x128_bf16": 3 * n3 + 4 * (n3 // 128),
            "quant_128x128": 3 * n4 + 4 * (n4 // 16384),
            "quant_tensor_e5m2": 5 * n5 + 4,
        }
        self.launches = {"unscale_check_update": 1, "quant_1x128": 1, "dequant_1x128_bf16": 1,
                         "quant_128x128": 1, "quant_tensor_e5m2": 2}
        torch.cuda.synchronize()

    def _views(self, g_flat, o_flat):
        """Per-tensor views of the flat gradient and output buffers (every
        tensor starts at a multiple of 4096 elements)."""
        grads, outs, off = [], [], 0
        for n in self.cfg2.numels:
            grads.append(g_flat[off:off + n])
            outs.append(o_flat[off:off + n])
            off += n
        return grads, outs

    @property
    def bytes_per_step(self) -> int:
        return sum(self.bytes.values())

    @property
    def launches_per_step(self) -> int:
        return sum(self.launches.values())

    def step(self, k: int, events=None):
        gs, torch = self.gs, self.torch
        st = torch.cuda.current_stream().cuda_stream
        nan_step = (k % 4) == 3

        def mark(name, fn):
            if events is None:
                fn()
                return
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            events.append((name, e0, e1))

        if nan_step:
            self.dg.plant_device(self.plant_ptr, 0x7E00, st)
        mark("unscale_check_update", lambda: gs.gs_unscale_check_update(
            self.tl, self.scale, self.tracker, self.found, self.skipped, 2.0, 0.5, 2000))
        if nan_step:
            self.dg.plant_device(self.plant_ptr, self.plant_orig, st)
        mark("quant_1x128", lambda: gs.fp8_quant_block(self.x3, 1, 128, "e4m3", self.q3, self.s3))
        mark("dequant_1x128_bf16", lambda: gs.fp8_dequant(self.q3, self.s3, 1, 128, "e4m3", self.y3))
        mark("quant_128x128", lambda: gs.fp8_quant_block(self.x4, 128, 128, "e4m3", self.q4, self.s4))
        mark("quant_tensor_e5m2", lambda: gs.fp8_quant_tensor(self.x5, "e5m2", self.q5, self.s5, self.ws))

    # -- end to end: host (pinned) buffers, copies inside the timed region ----
    # Steps are pipelined the way a training loop would run them: step k+1's
    # inputs go up (copy-in stream) while step k computes and step k-1's
    # results come down (copy-out stream).  Two device buffer sets (two
    # gradient lists) alternate; events keep every buffer from being
    # overwritten while a copy or a kernel still uses it.  Each gradient list
    # and its outputs live in one flat buffer, so a step is 4 copies up and
    # 11 down.
    def e2e_host_bytes(self) -> int:
        """Pinned host bytes e2e_setup allocates: the step's inputs and all its
        results (and the scaler state), one copy each."""
        ins = [self.g_flat, self.x3, self.x4, self.x5]
        res = [self.o_flat, self.q3, self.s3, self.y3, self.q4, self.s4, self.q5, self.s5,
               self.scale, self.tracker, self.found]
        return sum(t.numel() * t.element_size() for t in ins + res)

    def e2e_setup(self):
        torch, gs = self.torch, self.gs
        pin = dict(pin_memory=True)
        dev = self.grads[0].device
        self.sets = []
        for k in range(2):
            if k == 0:
                d = dict(g_flat=self.g_flat, o_flat=self.o_flat, grads=self.grads, outs=self.outs,
                         x3=self.x3, q3=self.q3, s3=self.s3, y3=self.y3, x4=self.x4, q4=self.q4,
                         s4=self.s4, x5=self.x5, q5=self.q5, s5=self.s5, tl=self.tl)
            else:
                d = dict(g_flat=torch.empty_like(self.g_flat), o_flat=torch.empty_like(self.o_flat),
                         x3=torch.empty_like(self.x3), q3=torch.empty_like(self.q3),
                         s3=torch.empty_like(self.s3), y3=torch.empty_like(self.y3),
                         x4=torch.empty_like(self.x4), q4=torch.empty_like(self.q4),
                         s4=torch.empty_like(self.s4), x5=torch.empty_like(self.x5),
                         q5=torch.empty_like(self.q5), s5=torch.empty_like(self.s5))
                d["grads"], d["outs"] = self._views(d["g_flat"], d["o_flat"])
                d["tl"] = gs.gs_tensor_list_create(d["grads"], d["outs"])
            d["ins"] = [d["g_flat"], d["x3"], d["x4"], d["x5"]]
            d["res"] = [d["o_flat"], d["q3"], d["s3"], d["y3"], d["q4"], d["s4"], d["q5"], d["s5"]]
            self.sets.append(d)
        self.h_in = [torch.empty(t.shape, dtype=t.dtype, **pin) for t in self.sets[0]["ins"]]
        for h, t in zip(self.h_in, self.sets[0]["ins"]):
            h.copy_(t)
        state = [self.scale, self.tracker, self.found]
        self.h_out = [torch.empty(t.shape, dtype=t.dtype, **pin)
                      for t in self.sets[0]["res"] + state]
        self.s_in = torch.cuda.Stream(dev)
        self.s_out = torch.cuda.Stream(dev)
        self.ev_in = [torch.cuda.Event() for _ in range(2)]       # inputs of set k uploaded
        self.ev_done = [torch.cuda.Event() for _ in range(2)]     # step on set k finished
        self.ev_out = [torch.cuda.Event() for _ in range(2)]      # results of set k downloaded
        for e in self.ev_done + self.ev_out:
            e.record()
        torch.cuda.synchronize()
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.h_in)
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in self.h_out)

    def release(self):
        """Frees every device and pinned host buffer of the step."""
        for d in getattr(self, "sets", []):
            if d["tl"] is not self.tl:
                d["tl"].close()
        self.tl.close()
        self.sets = []
        self.h_in = self.h_out = None
        self.grads = self.outs = self.g_flat = self.o_flat = None
        self.x3 = self.q3 = self.s3 = self.y3 = self.x4 = self.q4 = self.s4 = None
        self.x5 = self.q5 = self.s5 = self.ws = None

    def _step_on(self, d, k):
        gs = self.gs
        st = self.torch.cuda.current_stream().cuda_stream
        nan_step = (k % 4) == 3
        if nan_step:
            self.dg.plant_device(d["grads"][self.plant_t].data_ptr() + 2 * self.plant_i, 0x7E00, st)
        gs.gs_unscale_check_update(d["tl"], self.scale, self.tracker, self.found, self.skipped,
                                   2.0, 0.5, 2000)
        gs.fp8_quant_block(d["x3"], 1, 128, "e4m3", d["q3"], d["s3"])
        gs.fp8_dequant(d["q3"], d["s3"], 1, 128, "e4m3", d["y3"])
        gs.fp8_quant_block(d["x4"], 128, 128, "e4m3", d["q4"], d["s4"])
        gs.fp8_quant_tensor(d["x5"], "e5m2", d["q5"], d["s5"], self.ws)

    def e2e_step(self, k):
        torch = self.torch
        b = k % 2
        d = self.sets[b]
        comp = torch.cuda.current_stream()
        with torch.cuda.stream(self.s_in):                 # upload step k's inputs
            self.s_in.wait_event(self.ev_done[b])          # set b no longer read by step k-2
            for h, t in zip(self.h_in, d["ins"]):
                t.copy_(h, non_blocking=True)
            self.ev_in[b].record()
        comp.wait_event(self.ev_in[b])
        comp.wait_event(self.ev_out[b])                    # step k-2's results are down
        self._step_on(d, k)
        self.ev_done[b].record()
        with torch.cuda.stream(self.s_out):                # download step k's results
            self.s_out.wait_event(self.ev_done[b])
            for h, t in zip(self.h_out, d["res"] + [self.scale, self.tracker, self.found]):
                h.copy_(t, non_blocking=True)
            self.ev_out[b].record()


# ---- CPU oracle baseline ---------------------------------------------------------

class OracleSample:
    """A bounded sample of the same step, run by the CPU oracle: the first
    elements of the gradient list, whole rows of the activation, whole
    128-row block-rows of the weight, a slice of the gradient, in roughly
    the step's byte proportions (fraction `frac` of the full step)."""

    def __init__(self, frac: float = 1.0 / 1000):
        import numpy as np
        import datagen as dg
        from datagen import workloads as wl
        self.np = np
        cfg2 = wl.cfg2_grads()
        self.n_u = max(8, int(cfg2.total * frac))
        self.g_bits = dg.fill_host(cfg2.spec(0, 0), 0, self.n_u)
        a = wl.cfg3_act()
        self.rows3 = max(1, int(a.rows * frac))
        self.x3 = dg.fill_host(a.spec, 0, self.rows3 * a.cols).reshape(self.rows3, a.cols)
        w = wl.cfg4_weight()
        self.blocks4 = max(1, int(round(w.numel * frac / 16384)))
        cols4 = 128 * self.blocks4
        self.x4 = np.stack([dg.fill_host(w.spec, r * w.cols, cols4) for r in range(128)])
        g = wl.cfg4_grad()
        self.n5 = max(1, int(g.numel * frac))
        self.x5 = dg.fill_host(g.spec, 0, self.n5)
        n3, n4 = self.x3.size, self.x4.size
        self.bytes = (6 * self.n_u + 2 * (3 * n3 + 4 * (n3 // 128)) + 3 * n4 + 4 * (n4 // 16384)
                      + 5 * self.n5)
        self.desc = (f"oracle on {self.n_u} grad elems + {self.rows3}x{a.cols} act (1x128 quant + "
                     f"bf16 dequant) + 128x{cols4} weight (128x128) + {self.n5} grad elems "
                     f"(E5M2 per-tensor): {frac:.4g} of one step")

    def run(self):
        import oracle as orc
        orc.unscale_check(self.g_bits, 65536.0)
        q, s = orc.quant_block(self.x3, 1, 128, orc.E4M3, dtype=orc.BF16)
        orc.dequant(q, s, 1, 128, orc.E4M3, out_dtype=orc.BF16)
        orc.quant_block(self.x4, 128, 128, orc.E4M3, dtype=orc.BF16)
        orc.quant_tensor(self.x5, orc.E5M2, dtype=orc.BF16)


def _oracle_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except Exception:
        return max(1, os.cpu_count() or 1)


_ARM_PARTS = {0xd0c: "Arm Neoverse-N1", 0xd40: "Arm Neoverse-V1", 0xd49: "Arm Neoverse-N2",
              0xd4f: "Arm Neoverse-V2"}


def cpu_model(cpuinfo: str = None) -> str:
    """The host CPU's name from /proc/cpuinfo: "model name" on x86; on Arm,
    which lists only implementer and part numbers, the Arm part's name."""
    if cpuinfo is None:
        try:
            with open("/proc/cpuinfo") as f:
                cpuinfo = f.read()
        except OSError:
            return "unknown"
    impl = part = None
    for line in cpuinfo.splitlines():
        key, _, val = line.partition(":")
        key, val = key.strip().lower(), val.strip()
        if key == "model name" and val:
            return val
        if key == "cpu implementer" and impl is None:
            impl = val
        if key == "cpu part" and part is None:
            part = val
    if impl and part:
        try:
            if int(impl, 16) == 0x41 and int(part, 16) in _ARM_PARTS:
                return _ARM_PARTS[int(part, 16)]
        except ValueError:
            pass
        return f"implementer {impl} part {part}"
    return "unknown"


def oracle_parallel(sample, threads: int, seconds: float = None, reps: int = None):
    """Runs sample.run() on `threads` host threads (the oracle is plain C
    behind ctypes, which releases the GIL; the inputs are shared read-only)
    until `seconds` have passed or `reps` runs are done. Returns (runs,
    elapsed seconds)."""
    import threading
    from concurrent.futures import ThreadPoolExecutor
    lock = threading.Lock()
    state = {"left": reps, "done": 0}
    t0 = time.perf_counter()

    def worker():
        while True:
            with lock:
                if reps is not None:
                    if state["left"] <= 0:
                        return
                    state["left"] -= 1
                elif time.perf_counter() - t0 >= seconds:
                    return
            sample.run()
            with lock:
                state["done"] += 1

    with ThreadPoolExecutor(max_workers=threads) as ex:
        for f in [ex.submit(worker) for _ in range(threads)]:
            f.result()
    return state["done"], time.perf_counter() - t0


def cpu_baseline(seconds: float) -> dict:
    """The oracle on a bounded sample of the step: single-threaded for half
    the budget, then on every host core for the other half (reported)."""
    sample = OracleSample()
    sample.run()  # warm (and loads the oracle library before any thread starts)
    reps1, el1 = oracle_parallel(sample, 1, seconds=seconds / 2)
    n = _oracle_threads()
    repsn, eln = oracle_parallel(sample, n, seconds=seconds / 2)
    single = throughput(sample.bytes * reps1, el1)
    return {"value": throughput(sample.bytes * repsn, eln), "unit": UNIT, "cores": n,
            "kind": "oracle", "single_thread_value": single, "cpu_model": cpu_model(),
            "sample": f"{sample.desc}; {repsn} runs in {eln:.1f} s on {n} host threads "
                      f"({reps1} runs in {el1:.1f} s on one thread: {single:.3f} {UNIT})"}


# ---- arms -----------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    sample = OracleSample()
    sample.run()  # loads the oracle library before any thread starts
    n = _oracle_threads()
    # one step = one sample on every host thread, so each step uses all n
    oracle_parallel(sample, n, reps=args.warmup * n)
    runs, el = oracle_parallel(sample, n, reps=args.steps * n)
    value = throughput(sample.bytes * runs, el)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * el / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": WORKLOAD, "reference": "CPU oracle (plain C, scalar), the "
                       "pages ship no implementation; each step runs the sample once on "
                       "every host thread", "sample_bytes_per_step": sample.bytes * n},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": n, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"{sample.desc}, once per thread on {n} threads per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def gpu_uuid(torch, dev_index: int) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev_index)


def run_ours(args):
    import torch
    import mixed_precision_numerics_gradscaler_gb300 as gs

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dist = dist_init(world, "nccl")
    dev = torch.device("cuda", local)
    w = Workload(gs, torch)

    for k in range(args.warmup):
        w.step(k)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    events = []
    with ClockSampler(gpu_uuid(torch, local)) as clocks:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_start.record()
        for k in range(args.steps):
            w.step(args.warmup + k, events)
        t_end.record()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
    elapsed = t_start.elapsed_time(t_end) / 1000.0
    max_el, total_bytes = aggregate(elapsed, float(w.bytes_per_step * args.steps), dist, dev)
    launches = w.launches_per_step * args.steps
    bytes_per_step = w.bytes_per_step
    value = throughput(total_bytes, max_el)

    per = {}
    for name, e0, e1 in events:
        per.setdefault(name, []).append(e0.elapsed_time(e1))
    peak, peak_src = hbm_peak()
    kernels = {}
    for name, ts in per.items():
        ms = sum(ts) / len(ts)
        gbs = w.bytes[name] / (ms / 1000.0) / 1e9
        kernels[name] = {"avg_ms": round(ms, 4), "bytes": w.bytes[name], "gbs": round(gbs, 1),
                         "frac": round(gbs / peak, 4), "launches_per_step": w.launches[name]}
    dom = max(kernels, key=lambda n: kernels[n]["avg_ms"])
    roofline = {"bound": "hbm", "achieved": kernels[dom]["gbs"], "peak": peak, "unit": UNIT,
                "frac": kernels[dom]["frac"], "traffic": measured_traffic(dom), "kernel": dom,
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_src})",
                "frac_of_8tbs_nominal": round(kernels[dom]["gbs"] / 8000.0, 4)}

    e2e = None
    if not args.no_e2e:
        # every rank pins its own copy of the step's inputs and results: run
        # e2e only if all of this node's ranks fit in the host's memory (the
        # decision is the same on every rank, or the collectives below hang)
        need = w.e2e_host_bytes()
        local_ranks = int(os.environ.get("LOCAL_WORLD_SIZE", world))
        avail = host_memory_available()
        ok = torch.tensor([1 if e2e_fits(need, local_ranks, avail) else 0], device=dev)
        if dist:
            dist.all_reduce(ok, op=dist.ReduceOp.MIN)
        if not int(ok.item()):
            e2e = {"value": None, "unit": UNIT,
                   "skipped": f"pinned host buffers of {need / 1e9:.1f} GB per rank x "
                              f"{local_ranks} ranks exceed 60% of the host memory available "
                              f"({(avail or 0) / 1e9:.0f} GB) on some node"}
    if not args.no_e2e and e2e is None:
        w.e2e_setup()
        for k in range(2):
            w.e2e_step(k)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t0 = time.perf_counter()
        for k in range(args.e2e_steps):
            w.e2e_step(k)
        torch.cuda.synchronize()
        el = time.perf_counter() - t0
        if dist:
            dist.barrier()
        max_e2e, tot = aggregate(el, float(w.bytes_per_step * args.e2e_steps), dist, dev)
        link = measure_link(torch)
        link["ceiling_gbs"] = round(link_ceiling(w.bytes_per_step, w.h2d_bytes, w.d2h_bytes,
                                                 link["h2d_gbs"], link["d2h_gbs"],
                                                 link["both_gbs"]), 1)
        e2e = {"value": throughput(tot, max_e2e), "unit": UNIT,
               "link": link,
               "h2d_bytes_per_step": w.h2d_bytes, "d2h_bytes_per_step": w.d2h_bytes,
               "steps": args.e2e_steps, "ms_per_step": 1000 * max_e2e / args.e2e_steps,
               "pipeline": "two device buffer sets; step k+1's upload and step k-1's download "
                           "overlap step k (copy-in, compute and copy-out streams)"}

    cpu = cpu_baseline(args.cpu_seconds) if (rank == 0 and world == 1) else None
    sweep = extra = None
    if world == 1 and not args.no_extra:
        scale_after, skipped_after = float(w.scale.item()), int(w.skipped.item())
        w.release()
        del w
        torch.cuda.empty_cache()
        sweep = sweep_points(torch, gs, SWEEP_BENCH_SIZES, args.warmup)
        extra = kernels_extra(torch, gs, args.warmup)
    else:
        scale_after, skipped_after = float(w.scale.item()), int(w.skipped.item())
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1000 * max_el / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded counter-based generator, inputs resident in HBM)",
                "config": {"workload": WORKLOAD, "bytes_per_step": bytes_per_step,
                           "l2": "no flush: every input (16 GB, 268 MB, 470 MB, 470 MB) is larger "
                                 "than the 129 MB L2", "parallelism": f"replicas x{world}"},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches,
                "clocks": clocks.summary(), "kernels": kernels,
                "state_after": {"scale": scale_after, "skipped": skipped_after},
                "sweep": sweep, "kernels_extra": extra}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


# ---- config 5: the bandwidth sweep ---------------------------------------------

SWEEP_BENCH_SIZES = [1 << 20, 1 << 27, 1 << 31, 1 << 33]   # the points in the default line


def sweep_points(torch, gs, sizes, warmup: int, reps: int = 10) -> list:
    """GB/s of unscale (one flat fp16 tensor, config 2's distribution) and of
    1x128 E4M3 quantisation (bf16 [bytes/16384, 8192], config 3's
    distribution) for inputs of the given byte sizes; L2 flushed (a 512 MiB
    buffer zeroed) before every timed launch; median of `reps` launches."""
    import datagen as dg
    from datagen import workloads as wl
    st = torch.cuda.current_stream().cuda_stream
    peak, _ = hbm_peak()
    flush = torch.empty(512 * 2 ** 20, dtype=torch.uint8, device="cuda")

    def timed(fn):
        ts = []
        for r in range(max(warmup, 3) + reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            if r >= max(warmup, 3):
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    points = []
    for nbytes in sizes:
        res = {"input_bytes": nbytes, "cache_resident": nbytes < 2 * 129 * 2 ** 20}
        n = nbytes // 2
        g = torch.empty(n, dtype=torch.float16, device="cuda")
        dg.fill_device(wl.cfg5_grad_spec(), 0, n, g.data_ptr(), st)
        o = torch.empty(n, dtype=torch.float32, device="cuda")
        tl = gs.gs_tensor_list_create([g], [o])
        sc = torch.tensor([65536.0], device="cuda")
        tr = torch.zeros(1, dtype=torch.int32, device="cuda")
        fi = torch.zeros(1, dtype=torch.int32, device="cuda")
        ms = timed(lambda: gs.gs_unscale_check_update(tl, sc, tr, fi, None, 2.0, 0.5, 2000))
        b = 6 * n
        res["unscale"] = {"ms": round(ms, 5), "gbs": round(b / ms / 1e6, 1),
                          "frac": round(b / ms / 1e6 / peak, 4)}
        tl.close()
        del g, o, tl
        torch.cuda.empty_cache()
        a = wl.cfg5_act(nbytes)
        x = torch.empty(a.rows, a.cols, dtype=torch.bfloat16, device="cuda")
        dg.fill_device(a.spec, 0, a.numel, x.data_ptr(), st)
        q = torch.empty(a.rows, a.cols, dtype=torch.uint8, device="cuda")
        s = torch.empty(a.rows, a.cols // 128, dtype=torch.float32, device="cuda")
        ms = timed(lambda: gs.fp8_quant_block(x, 1, 128, "e4m3", q, s))
        b = 3 * a.numel + 4 * (a.numel // 128)
        res["quant_1x128"] = {"ms": round(ms, 5), "gbs": round(b / ms / 1e6, 1),
                              "frac": round(b / ms / 1e6 / peak, 4)}
        del x, q, s
        torch.cuda.empty_cache()
        points.append(res)
    del flush
    torch.cuda.empty_cache()
    return points


def run_sweep(args):
    """Config 5: every size of the sweep, 1 MiB .. 8 GiB."""
    import torch
    from datagen import workloads as wl
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    peak, src = hbm_peak()
    points = sweep_points(torch, gs, wl.cfg5_sizes(), args.warmup)
    print(json.dumps({"metric": METRIC, "unit": UNIT, "peak": peak, "peak_source": src,
                      "l2": "512 MiB buffer zeroed before every timed launch", "sweep": points}))
    return 0


# ---- one kernel alone --------------------------------------------------------------

ONLY_CASES = ["unscale", "quant_1x128", "dequant", "quant_128x128", "quant_128x128_16b",
              "quant_tensor", "quant_mx", "dequant_mx", "quant_delayed", "unscale_norm",
              "master_update", "gemm"]
# the rows beyond the step, timed after it in the default run
EXTRA_CASES = ["quant_mx", "dequant_mx", "quant_delayed", "unscale_norm", "master_update", "gemm"]


def kernel_case(torch, gs, name: str) -> dict:
    """Buffers and the launch of one kernel on its own workload: the unscale
    forms and the master update on the first two layers of the Llama-3-8B
    list (18 tensors, 436 M elements); the quantisers on their configs
    (268-470 MB of input); the FP8 GEMM on activations [16384, 8192] times a
    weight [28672, 8192].  Returns {"fn", "bytes" (algorithmic, per launch)
    or "flops", "workload"}."""
    import datagen as dg
    from datagen import workloads as wl
    st = torch.cuda.current_stream().cuda_stream
    dev = "cuda"
    if name in ("unscale", "unscale_norm", "master_update"):
        cfg = wl.cfg2_grads()
        n_t = 18
        grads = [torch.empty(n, dtype=torch.float16, device=dev) for n in cfg.numels[:n_t]]
        outs = [torch.empty(n, dtype=torch.float32, device=dev) for n in cfg.numels[:n_t]]
        for t, g in enumerate(grads):
            dg.fill_device(cfg.spec(t, 0), 0, g.numel(), g.data_ptr(), st)
        tl = gs.gs_tensor_list_create(grads, outs)
        sc = torch.tensor([65536.0], device=dev)
        tr = torch.zeros(1, dtype=torch.int32, device=dev)
        fi = torch.zeros(1, dtype=torch.int32, device=dev)
        nrm = torch.empty(1, dtype=torch.float32, device=dev)
        n_par = sum(cfg.numels[:n_t])
        wk = "Llama-3-8B grads, first 2 layers (18 tensors, %d elems)" % n_par
        if name == "unscale":
            return {"fn": lambda: gs.gs_unscale_check_update(tl, sc, tr, fi, None, 2.0, 0.5, 2000),
                    "bytes": 6 * n_par, "workload": wk, "keep": (grads, outs, tl)}
        gs.gs_unscale_check_update_norm(tl, sc, tr, fi, nrm, None, 2.0, 0.5, 2000)
        if name == "unscale_norm":
            return {"fn": lambda: gs.gs_unscale_check_update_norm(tl, sc, tr, fi, nrm, None, 2.0,
                                                                  0.5, 2000),
                    "bytes": 6 * n_par, "workload": wk, "keep": (grads, outs, tl)}
        w32 = [torch.zeros(n, dtype=torch.float32, device=dev) for n in cfg.numels[:n_t]]
        wbf = [torch.zeros(n, dtype=torch.bfloat16, device=dev) for n in cfg.numels[:n_t]]
        pl = gs.gs_param_list_create(w32, outs, wbf)
        return {"fn": lambda: gs.gs_master_update_sgd(pl, 1e-4, 1.0, nrm, fi),
                "bytes": 14 * n_par, "workload": wk + ", SGD on fp32 masters + bf16 copies",
                "keep": (grads, outs, tl, w32, wbf, pl)}
    if name in ("quant_1x128", "dequant", "quant_mx", "dequant_mx"):
        a = wl.cfg3_act()
        x = torch.empty(a.rows, a.cols, dtype=torch.bfloat16, device=dev)
        dg.fill_device(a.spec, 0, a.numel, x.data_ptr(), st)
        q = torch.empty(a.rows, a.cols, dtype=torch.uint8, device=dev)
        y = torch.empty(a.rows, a.cols, dtype=torch.bfloat16, device=dev)
        wk = "bf16 activations [16384, 8192]"
        if name in ("quant_1x128", "dequant"):
            s = torch.empty(a.rows, a.cols // 128, dtype=torch.float32, device=dev)
            gs.fp8_quant_block(x, 1, 128, "e4m3", q, s)
            fn = (lambda: gs.fp8_quant_block(x, 1, 128, "e4m3", q, s)) if name == "quant_1x128" \
                else (lambda: gs.fp8_dequant(q, s, 1, 128, "e4m3", y))
            return {"fn": fn, "bytes": 3 * a.numel + 4 * (a.numel // 128),
                    "workload": wk + (", E4M3 1x128" if name == "quant_1x128" else
                                      ", E4M3 1x128 -> bf16"), "keep": (x, q, s, y)}
        s = torch.empty(a.rows, a.cols // 32, dtype=torch.uint8, device=dev)
        gs.fp8_quant_mx(x, "e4m3", q, s)
        fn = (lambda: gs.fp8_quant_mx(x, "e4m3", q, s)) if name == "quant_mx" \
            else (lambda: gs.fp8_dequant_mx(q, s, "e4m3", y))
        return {"fn": fn, "bytes": 3 * a.numel + a.numel // 32,
                "workload": wk + (", MXFP8 E4M3" if name == "quant_mx" else ", MXFP8 E4M3 -> bf16"),
                "keep": (x, q, s, y)}
    if name == "gemm":
        a = wl.cfg3_act()
        w = wl.cfg4_weight(rows=28672, cols=8192)
        x = torch.empty(a.rows, a.cols, dtype=torch.bfloat16, device=dev)
        dg.fill_device(a.spec, 0, a.numel, x.data_ptr(), st)
        wt = torch.empty(w.rows, w.cols, dtype=torch.bfloat16, device=dev)
        dg.fill_device(w.spec, 0, w.numel, wt.data_ptr(), st)
        qa = torch.empty(a.rows, a.cols, dtype=torch.uint8, device=dev)
        sa = torch.empty(a.rows, a.cols // 128, dtype=torch.float32, device=dev)
        qb = torch.empty(w.rows, w.cols, dtype=torch.uint8, device=dev)
        sb = torch.empty(w.rows // 128, w.cols // 128, dtype=torch.float32, device=dev)
        gs.fp8_quant_block(x, 1, 128, "e4m3", qa, sa)
        gs.fp8_quant_block(wt, 128, 128, "e4m3", qb, sb)
        del x, wt
        d = torch.empty(a.rows, w.rows, dtype=torch.bfloat16, device=dev)
        return {"fn": lambda: gs.fp8_gemm_block_scaled(qa, sa, qb, sb, "e4m3", d),
                "flops": 2 * a.rows * w.rows * a.cols,
                "workload": "E4M3 [16384, 8192] (1x128 scales) x [28672, 8192]^T (128x128 "
                            "scales) -> bf16", "keep": (qa, sa, qb, sb, d)}
    if name in ("quant_128x128", "quant_128x128_16b"):
        w = wl.cfg4_weight()
        # input 16-byte but not 32-byte aligned: the 16-byte-load kernel
        off = 8 if name == "quant_128x128_16b" else 0
        xbuf = torch.empty(w.numel + off, dtype=torch.bfloat16, device=dev)
        x = xbuf[off:].view(w.rows, w.cols)
        dg.fill_device(w.spec, 0, w.numel, x.data_ptr(), st)
        q = torch.empty(w.rows, w.cols, dtype=torch.uint8, device=dev)
        s = torch.empty(w.rows // 128, w.cols // 128, dtype=torch.float32, device=dev)
        return {"fn": lambda: gs.fp8_quant_block(x, 128, 128, "e4m3", q, s),
                "bytes": 3 * w.numel + 4 * (w.numel // 16384),
                "workload": "bf16 weight 8192x28672, E4M3 128x128" +
                            (" (input 16-byte aligned)" if off else ""), "keep": (xbuf, q, s)}
    g = wl.cfg4_grad()
    x = torch.empty(g.numel, dtype=torch.bfloat16, device=dev)
    dg.fill_device(g.spec, 0, g.numel, x.data_ptr(), st)
    q = torch.empty(g.numel, dtype=torch.uint8, device=dev)
    ws = torch.empty(gs.gs_ws_bytes() // 4, dtype=torch.int32, device=dev)
    if name == "quant_delayed":
        hist = torch.full((16,), 1e-2, dtype=torch.float32, device=dev)
        pos = torch.zeros(1, dtype=torch.int32, device=dev)
        used = torch.empty(1, dtype=torch.float32, device=dev)
        return {"fn": lambda: gs.fp8_quant_tensor_delayed(x, "e5m2", q, hist, pos, used, ws),
                "bytes": 3 * g.numel + 4,
                "workload": "bf16 gradient 8192x28672, E5M2 delayed (history of 16)",
                "keep": (x, q, ws, hist, pos, used)}
    s = torch.empty(1, dtype=torch.float32, device=dev)
    return {"fn": lambda: gs.fp8_quant_tensor(x, "e5m2", q, s, ws), "bytes": 5 * g.numel + 4,
            "workload": "bf16 gradient 8192x28672, E5M2 per-tensor (two passes)",
            "keep": (x, q, ws, s)}


def time_case(torch, case: dict, warmup: int, iters: int, reps: int = 10) -> dict:
    """Median per-launch time of `reps` back-to-back launches between two
    events (host launch latency stays outside the interval; every input
    exceeds L2), over `iters` iterations, with the SM clocks sampled."""
    fn = case["fn"]
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    with ClockSampler(gpu_uuid(torch, torch.cuda.current_device())) as clocks:
        for _ in range(iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            fn()
            e0.record()
            for _ in range(reps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / reps)
    ms = statistics.median(ts)
    out = {"workload": case["workload"], "median_ms": round(ms, 5), "iters": iters,
           "launches_timed": iters * reps, "timed_s": round(sum(ts) * reps / 1e3, 3),
           "clocks": clocks.summary()}
    if "flops" in case:
        peak_s, src_s = fp8_peak(sustained=True)
        peak_b, src_b = fp8_peak(sustained=False)
        tf = case["flops"] / ms / 1e9
        first = case["flops"] / ts[0] / 1e9
        out.update({"flops": case["flops"], "tflops": round(tf, 1), "peak_tflops": peak_s,
                    "frac": round(tf / peak_s, 4), "peak_source": src_s,
                    "tflops_first_iter": round(first, 1), "peak_burst_tflops": peak_b,
                    "frac_burst": round(first / peak_b, 4)})
    else:
        peak, src = hbm_peak()
        gbs = case["bytes"] / ms / 1e6
        out.update({"bytes": case["bytes"], "gbs": round(gbs, 1), "peak": peak,
                    "frac": round(gbs / peak, 4), "peak_source": src})
    return out


def kernels_extra(torch, gs, warmup: int) -> dict:
    """The rows beyond the step, each timed alone after it: MXFP8 quantise and
    dequantise, delayed E5M2, the norm form of the unscale, the master
    update, and the FP8 GEMM (timed for about a second, against the sustained
    FP8 peak)."""
    out = {}
    for name in EXTRA_CASES:
        case = kernel_case(torch, gs, name)
        out[name] = time_case(torch, case, max(warmup, 3), 40 if name == "gemm" else 10)
        del case
        torch.cuda.empty_cache()
    out["gpu_status"] = gs.gs_device_status()
    return out


def run_only(args):
    """One kernel alone, on a case small enough for a full ncu capture."""
    import torch
    import mixed_precision_numerics_gradscaler_gb300 as gs
    torch.cuda.set_device(0)
    case = kernel_case(torch, gs, args.only)
    r = time_case(torch, case, args.warmup, args.steps)
    r["only"] = args.only
    r["gpu_status"] = gs.gs_device_status()
    print(json.dumps(r), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.only:
        return run_only(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
