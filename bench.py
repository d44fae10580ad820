#!/usr/bin/env python
"""Throughput of one cached-attention denoising step of a LLaDA-8B attention layer.

One step (the timed unit) on the batch-32 workload: top-32 selection of the previous
step's most-attended positions and, in the same launch, the gather of those tokens'
hidden states from this step's hidden states of every position; the fused QKV
projection + rotary embedding + cache write of the 32-token active block of every
sequence together with the K/V of the 32 tracked tokens, whose cosine drift against
the cache the same kernel's epilogue sums (a small kernel after it writes the cosines
and the refresh flags); and bidirectional attention of the block over the 1024-slot
cache.  Inputs are seeded synthetic
arrays from ``workloads``; the cache (512 MiB), the weights and the layer's hidden
states (256 MiB) are resident in HBM.

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 oracle instead,
on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# Enough hardware work queues that the copy-in, compute and copy-out streams of the
# end-to-end loop do not serialise behind one another (process setting, read at CUDA
# initialisation).
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

METRIC = "layer-steps/s & fraction of roofline (TC % / HBM GB/s), LLaDA-8B layer, bs 1-32"
UNIT = "layer-steps/s"
L2_BYTES = 126 * 2 ** 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llada8b-b32-drift", choices=["llada8b-b1", "llada8b-b32-drift"],
                    help="the step's workload: the LLaDA-8B layer at batch 32 with drift tracking (default) or batch 1")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-unfused", action="store_true", help="skip the fused-vs-unfused comparison")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline sample")
    ap.add_argument("--no-elastic", action="store_true", help="skip the multi-layer refresh step")
    ap.add_argument("--elastic-layers", type=int, default=32)
    ap.add_argument("--probe", choices=["attend", "project"], default=None,
                    help="run only this kernel of --probe-workload (for one-kernel profiler captures) and exit")
    ap.add_argument("--probe-workload", default="llada8b-b8-refresh-fp8",
                    choices=["llada8b-b32-drift", "llada8b-b1", "llada8b-b16-verify", "llada8b-b8-refresh-fp8"])
    ap.add_argument("--probe-iters", type=int, default=5)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_traffic(kernel_key: str):
    """DRAM bytes per launch of a kernel from the committed ncu capture, or None when the
    kernel's sources have changed since that capture (hash recorded beside the figure)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic_llada8b_b32.json")
    files = {"project": ["proj_rope_store.cu", "ptx.cuh", "internal.h"],
             "attend": ["attn_cache.cu", "ptx.cuh", "internal.h"]}[kernel_key]
    try:
        with open(path) as f:
            rec = json.load(f)["kernels"][kernel_key]
        h = hashlib.sha256()
        for fn in files:
            with open(os.path.join(ROOT, "denoising_step_attention_qkv_b300", "csrc", fn), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != rec["sources_sha256_16"]:
            return None
        return rec["traffic_bytes"]
    except (OSError, KeyError, ValueError):
        return None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ----------------------------------------------------------------------------- clocks
class Clocks:
    """Samples the SM clock and the clock-event reasons of the GPU that runs the bench,
    every 5 ms on a background thread while the timed region runs.  It reads the
    driver's NVML library through ctypes (the device is found by its PCI bus id); when
    that library cannot be opened it falls back to ``nvidia-smi -lms 50``, keeping only
    samples stamped inside the timed window."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, torch_device):
        import ctypes
        import threading
        self.samples, self.reason_bits, self.max_mhz = [], 0, None
        self.stop_evt = threading.Event()
        self.thread = None
        self.proc = None
        self.t0 = time.time()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            props = __import__("torch").cuda.get_device_properties(torch_device)
            bus = f"{props.pci_domain_id:08X}:{props.pci_bus_id:02X}:{props.pci_device_id:02X}.0".encode()
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) != 0:
                raise OSError(f"no NVML device at {bus!r}")
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) != 0:
                raise OSError("nvmlDeviceGetMaxClockInfo failed")
            self.nv, self.h, self.max_mhz = nv, h, mx.value
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
        except Exception as exc:  # no NVML library: sample with nvidia-smi instead
            print(f"clock sampling: NVML unavailable ({exc!r}); using nvidia-smi", file=sys.stderr)
            self.nv = None
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={torch_device.index or 0}",
                     "--query-gpu=timestamp,clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
                time.sleep(0.5)
            except OSError:
                self.proc = None

    def start(self):
        self.t0 = time.time()

    def _poll(self):
        import ctypes
        nv, h = self.nv, self.h
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop_evt.is_set():
            if nv.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if nv.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                self.reason_bits |= int(rs.value)
            self.stop_evt.wait(0.005)

    def stop(self):
        t1 = time.time()
        if self.thread is not None:
            self.stop_evt.set()
            self.thread.join()
            reasons = sorted(v for k, v in self.REASONS.items() if self.reason_bits & k)
            if not self.samples:
                return None
            return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz, "reasons": reasons,
                    "samples": len(self.samples), "source": "NVML, 5 ms polling during the timed region"}
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        self.proc.wait()
        import datetime
        sm, bits, mx = [], 0, None
        for ln in open(self.f.name):
            r = [x.strip() for x in ln.split(",")]
            if len(r) != 4:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                if not (self.t0 <= ts <= t1):
                    continue
                sm.append(float(r[1]))
                mx = float(r[2])
                bits |= int(r[3], 16)
            except ValueError:
                continue
        os.unlink(self.f.name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(v for k, v in self.REASONS.items() if bits & k), "samples": len(sm),
                "source": "nvidia-smi -lms 50 inside the timed window"}


# ------------------------------------------------------------------- job throughput
def job_rate(local_ms: float, steps: int, world: int, device=None):
    """Whole-job throughput from each rank's timed total: the slowest rank's time
    (max over ranks) covers the steps of all ranks.  Returns (ms_per_step, steps/s)."""
    total_ms = float(local_ms)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms / steps, world * steps / (total_ms / 1e3)


# --------------------------------------------------------------------------- workload
def algorithmic(wl):
    """FLOPs and bytes of each kernel of the step, counting each tensor once."""
    s = wl.shape
    B, D, H, hd, S = s.batch, s.D, s.n_heads, s.head_dim, s.max_pos
    n_tok = wl.x.shape[1]
    k = wl.drift_k
    proj_flops = 2.0 * B * n_tok * 3 * D * D + 2.0 * B * k * 2 * D * D
    # W once, the block and tracked rows in, Q and the block's K/V out, and (the fused
    # drift test) the tracked tokens' cached K/V read
    proj_bytes = 3 * D * D * 2 + B * (n_tok + k) * D * 2 + B * n_tok * 3 * D * 2 + B * k * 2 * D * 2
    attn_bytes = B * H * S * hd * 2 * 2 + 2 * B * n_tok * D * 2
    attn_flops = 4.0 * B * H * n_tok * S * hd
    drift_bytes = B * k * 2 * D * 2 * 2  # the separate drift kernel: cache rows + probe rows
    gather_bytes = 2 * B * k * D * 2
    return dict(proj_flops=proj_flops, proj_bytes=proj_bytes, attn_bytes=attn_bytes, attn_flops=attn_flops,
                drift_bytes=drift_bytes, gather_bytes=gather_bytes)


def roofline_entry(name, us, flops, nbytes, pk, tc_peak=None):
    """One kernel against the slower of its two bounds: the ideal time is the larger of
    FLOPs at the tensor peak and bytes at the copy peak; frac = ideal / measured.  The
    achieved figure is reported in the bound's own unit."""
    tc = pk["bf16_tflops"] if tc_peak is None else tc_peak
    t_tc = flops / (tc * 1e12) if flops else 0.0
    t_hbm = nbytes / (pk["hbm_gbs"] * 1e9)
    tensor = t_tc >= t_hbm
    sec = us * 1e-6
    ach = (flops / sec / 1e12) if tensor else (nbytes / sec / 1e9)
    peak = tc if tensor else pk["hbm_gbs"]
    return {"kernel": name, "us": us, "bound": "tensor" if tensor else "hbm", "achieved": ach,
            "unit": "TFLOP/s" if tensor else "GB/s", "peak": peak, "frac": ach / peak,
            "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
            "other_bound_frac": (nbytes / sec / 1e9 / pk["hbm_gbs"]) if tensor else (flops / sec / 1e12 / tc)}


def elastic_leg(args, dev, B, S, D, H, hd, theta, beta, k, gamma, flush, kv_dtype=None):
    """One denoising step over L layers with the depth-wise drift refresh
    (dllm_elastic_step), LLaDA-8B layer shapes.  Inputs are drawn on the device from a
    seeded generator: per layer the hidden states the cache was built from, x_prev ~
    N(0, 1), and this step's x_all = x_prev + sigma[l][b] * N(0, 1) with
    sigma[l][b] = 0.6 * (l + 1) / L * s_b, s_b ~ U(0.3, 1.2): drift grows with depth and
    some sequences fail the test in deep layers.  The step is stationary (the failing
    layer keeps its cache, so every repetition refreshes the same sequence-layers).
    Also timed: gamma = -2 (never refresh) and gamma = 2 (every sequence recomputes
    layers 1..L-1), the two ends of the threshold.  kv_dtype: the cache's storage type
    (bf16 by default; e4m3 refreshes into the FP8 cache with its per-group scales)."""
    import torch
    from denoising_step_attention_qkv_b300 import capi
    if kv_dtype is None:
        kv_dtype = capi.DLLM_BF16
    L = args.elastic_layers
    g = torch.Generator(device=dev)
    g.manual_seed(2024)
    cache = capi.Cache(L, B, S, H, hd, kv_dtype, theta, 0, device=dev)
    all_pos = torch.arange(S, dtype=torch.int32, device=dev).repeat(B, 1)
    s_b = 0.3 + 0.9 * torch.rand(B, generator=g, device=dev)
    ws, xs = [], []
    for l in range(L):
        w = (torch.randn((3 * D, D), generator=g, device=dev) * 0.02).to(torch.bfloat16)
        x_prev = torch.randn((B, S, D), generator=g, device=dev)
        capi.dllm_cache_step(cache.handle, l, None, w, None, None, None, kv_x=x_prev.to(torch.bfloat16),
                             kv_positions=all_pos)
        sig = (0.6 * (l + 1) / L) * s_b
        x_prev += sig[:, None, None] * torch.randn((B, S, D), generator=g, device=dev)
        ws.append(w)
        xs.append(x_prev.to(torch.bfloat16))
        del x_prev
    mass = torch.distributions.Dirichlet(torch.full((S,), 0.1, device=dev)).sample((L, B)).float().contiguous()
    win_lo = (512 + beta * torch.randint(0, (S - 512) // beta, (B,), generator=g, device=dev)).to(torch.int32)
    out = torch.empty((L, B, beta, D), dtype=torch.bfloat16, device=dev)
    cos = torch.empty((L, B, k, 2), dtype=torch.float32, device=dev)
    flags = torch.empty((L, B), dtype=torch.int32, device=dev)
    work = torch.empty(capi.dllm_elastic_workspace_bytes(cache.handle, beta, k), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    n = max(3, min(args.steps, 10))

    def run(gm):
        step = lambda: capi.dllm_elastic_step(cache.handle, xs, ws, win_lo, beta, mass, k, gm, out, cos, flags, work,
                                              stream=stream)
        for _ in range(2):
            step()
        evs = []
        for _ in range(n):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            step()
            b_.record(stream)
            evs.append((a_, b_))
        torch.cuda.synchronize(dev)
        ms = statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)
        f = flags.cpu().numpy()
        failed = np.cumsum(f, axis=0) > 0  # failed at or above each layer
        refreshed = int(failed[:-1].sum())  # sequence-layers recomputed in the next layer down
        return {"gamma": gm, "ms_per_step": ms, "layer_steps_per_s": L * 1e3 / ms,
                "refreshed_sequence_layers": refreshed, "of": B * L,
                "first_failing_layer": [int(np.argmax(f[:, b])) if f[:, b].any() else None for b in range(B)]}

    res = {"layers": L, "batch": B, "window": beta, "tracked": k, "steps": n,
           "kv": "e4m3" if kv_dtype == capi.DLLM_E4M3 else "bf16", "runs": [run(gamma), run(-2.0), run(2.0)],
           "inputs": "device-generated, seeded: x_prev ~ N(0,1); x_all = x_prev + sigma[l][b] N(0,1), "
                     "sigma = 0.6 (l+1)/L s_b, s_b ~ U(0.3, 1.2); mass ~ Dirichlet(0.1); L2 flushed between steps"}
    rc, bits = cache.status()
    if rc != capi.DLLM_OK:
        raise RuntimeError(f"device status {bits:#x} in the multi-layer step")
    del cache, xs, ws
    torch.cuda.empty_cache()
    return res


OTHER_WORKLOADS = ("llada8b-b1", "llada8b-b16-verify", "llada8b-b8-refresh-fp8")


def workload_calls(dev, wl_name, stream):
    """A workload's cache (prefilled when the workload has a prefix) and its projection
    and attention calls on `stream`.  Returns (workload, cache, project, attend, x, kv_x,
    view)."""
    import torch
    import workloads as W
    from denoising_step_attention_qkv_b300 import capi
    kvt = {"bf16": capi.DLLM_BF16, "e4m3": capi.DLLM_E4M3}

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(dev)

    wl = W.make(wl_name)
    s = wl.shape
    cache = capi.Cache(1, s.batch, s.max_pos, s.n_heads, s.head_dim, kvt[s.kv], s.rope_theta, s.tail_slots,
                       device=dev)
    w = bf(wl.w)
    if wl.pre_x is not None:
        capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None, kv_x=bf(wl.pre_x),
                             kv_positions=torch.from_numpy(wl.pre_pos).to(dev))
    x = bf(wl.x)
    pos = torch.from_numpy(wl.positions).to(dev)
    view = torch.from_numpy(wl.view).to(dev) if wl.view is not None else None
    kv_x = bf(wl.kv_x) if wl.kv_x is not None else None
    kv_pos = torch.from_numpy(wl.kv_pos).to(dev) if wl.kv_pos is not None else None
    out = torch.empty_like(x)

    def project(st=stream):
        capi.dllm_cache_project(cache.handle, 0, x, w, pos, view, out, kv_x=kv_x, kv_positions=kv_pos, stream=st)

    def attend(st=stream):
        capi.dllm_cache_attend(cache.handle, 0, pos, view, out, stream=st)

    return wl, cache, project, attend, x, kv_x, view


def probe(args):
    """One kernel of one workload, alone: the projection once (the attention's queries),
    then `--probe-iters` calls of the probed kernel, and one JSON line with their median
    time.  For one-kernel profiler captures; no other work runs."""
    import torch
    from denoising_step_attention_qkv_b300 import capi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    wl, cache, project, attend, *_ = workload_calls(dev, args.probe_workload, stream)
    project()
    fn = attend if args.probe == "attend" else project
    evs = []
    for _ in range(args.probe_iters):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        fn()
        b_.record(stream)
        evs.append((a_, b_))
    torch.cuda.synchronize(dev)
    rc, bits = cache.status()
    if rc != capi.DLLM_OK:
        raise RuntimeError(f"device status {bits:#x}")
    print(json.dumps({"probe": args.probe, "workload": wl.name, "iters": args.probe_iters,
                      "median_us": statistics.median(a_.elapsed_time(b_) for a_, b_ in evs) * 1e3}), flush=True)


def other_configs(dev, flush, n_iter=30):
    """Projection and attention of the other workloads against their rooflines: the
    LLaDA-8B layer at batch 1 (eager and replayed as one CUDA graph, which shows the
    launch overhead), the batch-16 Flash-Verify step (48 rows per sequence, 16 tail
    slots) and the batch-8 full refresh into an e4m3 cache (every non-block position
    K/V, then the 32-row block).  Per-call CUDA events, L2 flushed before each call."""
    import torch
    from denoising_step_attention_qkv_b300 import capi
    pk = peaks()
    stream = torch.cuda.current_stream(dev)

    def timed(fn):
        for _ in range(3):
            fn()
        evs = []
        for _ in range(n_iter):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            fn()
            b_.record(stream)
            evs.append((a_, b_))
        torch.cuda.synchronize(dev)
        return statistics.median(a_.elapsed_time(b_) for a_, b_ in evs) * 1e3

    res = {}
    for wl_name in OTHER_WORKLOADS:
        wl, cache, project, attend, x, kv_x, view = workload_calls(dev, wl_name, stream)
        s = wl.shape
        B, D, H, hd, S, T = s.batch, s.D, s.n_heads, s.head_dim, s.max_pos, s.tail_slots
        n = x.shape[1]
        n_kv = 0 if kv_x is None else kv_x.shape[1]

        # attention alone, timed first (before the projection's long power-capped GEMM
        # loop): after one projection, each call attends with the previous call's output
        # as its queries (same work; the values stay finite)
        project()
        t_a = timed(attend)
        t_p = timed(project)
        flops = 2.0 * B * (n * 3 * D + n_kv * 2 * D) * D
        elt = 1 if s.kv == "e4m3" else 2
        slots = S + (T if view is not None else 0)
        a_bytes = B * slots * 2 * D * elt + (B * slots * 2 * H * 4 if s.kv == "e4m3" else 0) + 2 * B * n * D * 2
        a_flops = 4.0 * B * H * n * slots * hd
        # projection bytes: W once, the rows in, Q out, K/V (and e4m3 scales) to the cache
        kv_row = 2 * D * elt + (2 * H * 4 if s.kv == "e4m3" else 0)
        p_bytes = 3 * D * D * 2 + B * (n + n_kv) * D * 2 + B * n * D * 2 + B * (n + n_kv) * kv_row
        rp = roofline_entry("project", t_p, flops, p_bytes, pk)
        ra = roofline_entry("attend", t_a, a_flops, a_bytes, pk)
        r = {"workload": wl.name, "rows_per_seq": n, "refresh_rows_per_seq": n_kv, "kv": s.kv,
             "project_us": t_p, "project_bound": rp["bound"], "project_achieved": rp["achieved"],
             "project_unit": rp["unit"], "project_frac": rp["frac"],
             "attend_us": t_a, "attend_bound": ra["bound"], "attend_achieved": ra["achieved"],
             "attend_unit": ra["unit"], "attend_frac": ra["frac"],
             "algorithmic_flops": flops, "project_bytes": p_bytes, "attend_bytes": a_bytes,
             "frac_note": "each fraction against the slower of its two bounds (FLOPs at the bf16 peak, "
                          "algorithmic bytes at the copy peak)"}
        if wl_name == "llada8b-b1":  # the same two calls replayed from one CUDA graph: no launch cost
            g = torch.cuda.CUDAGraph()
            s_cap = torch.cuda.Stream(dev)
            s_cap.wait_stream(stream)
            with torch.cuda.stream(s_cap):
                for _ in range(2):
                    project(s_cap)
                    attend(s_cap)
                with torch.cuda.graph(g, stream=s_cap):
                    project(s_cap)
                    attend(s_cap)
            stream.wait_stream(s_cap)
            r["project_attend_graph_us"] = timed(g.replay)
            r["project_attend_eager_us"] = timed(lambda: (project(), attend()))
        rc, bits = cache.status()
        if rc != capi.DLLM_OK:
            raise RuntimeError(f"device status {bits:#x} in {wl.name}")
        res[wl.name] = r
        del cache
    return res


def run_ours(args, rank, world, local):
    import torch
    import workloads as W
    from denoising_step_attention_qkv_b300 import capi

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = _with_drift_inputs(W.make(args.workload))
    s = wl.shape
    B, D, S = s.batch, s.D, s.max_pos
    k = wl.drift_k

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).to(dev)

    cache = capi.Cache(1, B, S, s.n_heads, s.head_dim, capi.DLLM_BF16, s.rope_theta, 0, device=dev)
    w = bf(wl.w)
    capi.dllm_cache_step(cache.handle, 0, None, w, None, None, None, kv_x=bf(wl.pre_x),
                         kv_positions=torch.from_numpy(wl.pre_pos).to(dev))
    x = bf(wl.x)
    pos = torch.from_numpy(wl.positions).to(dev)
    out = torch.empty_like(x)
    mass = torch.from_numpy(wl.mass).to(dev)
    block_lo = torch.from_numpy(wl.block_lo).to(dev)
    idx = torch.empty((B, k), dtype=torch.int32, device=dev)
    probe = torch.empty((B, k, 2, D), dtype=torch.bfloat16, device=dev)
    cos = torch.empty((B, k, 2), dtype=torch.float32, device=dev)
    refresh = torch.empty(B, dtype=torch.int32, device=dev)
    # this step's hidden states of every position (resident, like the cache): the step
    # gathers the tracked tokens' rows from it on the device
    x_all = bf(wl.probe_rows(np.tile(np.arange(S, dtype=np.int32), (B, 1))))
    x_probe = torch.empty((B, k, D), dtype=torch.bfloat16, device=dev)  # the gathered rows
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    KERNELS = ("topk_gather", "project", "attend")

    def step_plain():
        capi.dllm_kv_topk_gather(cache.handle, mass, block_lo, wl.block_len, k, idx, x_all, x_probe, stream=stream)
        capi.dllm_cache_project_drift(cache.handle, 0, x, w, pos, None, out, x_probe, idx, wl.gamma, cos, refresh,
                                      stream=stream)
        capi.dllm_cache_attend(cache.handle, 0, pos, None, out, stream=stream)

    def step():
        capi.dllm_kv_topk_gather(cache.handle, mass, block_lo, wl.block_len, k, idx, x_all, x_probe, stream=stream)
        ev[1].record(stream)
        capi.dllm_cache_project_drift(cache.handle, 0, x, w, pos, None, out, x_probe, idx, wl.gamma, cos, refresh,
                                      stream=stream)
        ev[2].record(stream)
        capi.dllm_cache_attend(cache.handle, 0, pos, None, out, stream=stream)

    ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)]
    for _ in range(max(args.warmup, 3)):
        ev[0].record(stream)
        step()
        ev[-1].record(stream)
    torch.cuda.synchronize(dev)
    rc, bits = cache.status()
    if rc != capi.DLLM_OK:
        raise RuntimeError(f"device status {bits:#x} after warm-up")

    # ---- timed region: K steps, L2 flushed between steps (outside the events).  Events
    # only at step boundaries, so that each kernel's prologue overlaps the end of the one
    # before it (programmatic dependent launch), as in a real step.
    per = {"step": [], **{kname: [] for kname in KERNELS}}
    clocks = Clocks(dev) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    if clocks:
        clocks.start()
    evs = []
    t_wall = time.perf_counter()
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step_plain()
        e1.record(stream)
        evs.append((e0, e1))
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop() if clocks else None
    per["step"] = [e0.elapsed_time(e1) for e0, e1 in evs]
    ms_per_step, value = job_rate(sum(per["step"]), args.steps, world, dev)

    # ---- per-kernel times (the roofline's durations): a second timed pass of the same
    # step with an event between every two kernels (which stops their overlap, so these
    # intervals are each kernel's own duration plus its launch)
    n_bd = min(args.steps, 300)
    evs = []
    for _ in range(n_bd):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)]
        ev[0].record(stream)
        step()
        ev[-1].record(stream)
        evs.append(ev)
    torch.cuda.synchronize(dev)
    for ev in evs:
        for i, kname in enumerate(KERNELS):
            per[kname].append(ev[i].elapsed_time(ev[i + 1]))

    def timed_us(fn, n):
        """Mean device time of fn in microseconds over n calls, L2 flushed before each."""
        for _ in range(3):
            fn()
        evs2 = []
        for _ in range(n):
            flush.zero_()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            fn()
            b_.record(stream)
            evs2.append((a_, b_))
        torch.cuda.synchronize(dev)
        return statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs2) * 1e3

    # ---- end to end through the C ABI with host buffers (copies inside the timed region).
    # Every step copies its inputs from pinned host memory and reads its results back.
    # Steady state is one CUDA graph per step with three independent branches: the
    # copy-in of step i+1, the kernels of step i and the read-back of step i-1, on
    # double-buffered device tensors, so a step costs the slowest branch.  The timed
    # region is the copy-in of step 0, K graph launches and the read-back of step K-1
    # (the graphs also copy in one step too many and read back one too many: counted).
    # No L2 flush here: every step streams the whole cache, which is larger than L2.
    e2e = None
    if not args.no_e2e:
        # host buffers: page-locked blocks from the library's allocator; the inputs are
        # written into them with its streaming-store copy, as a serving loop stages them
        h_in = [capi.dllm_host_stage(capi.host_empty(t.shape, t.dtype), t.cpu())
                for t in (x, pos, mass, block_lo)]
        d_in = [[x, pos, mass, block_lo], [t.clone() for t in (x, pos, mass, block_lo)]]
        d_xtrk = [x_probe, torch.empty_like(x_probe)]
        d_out = [[out, cos, refresh], [torch.empty_like(t) for t in (out, cos, refresh)]]
        h_out = [[capi.host_empty(t.shape, t.dtype) for t in (out, cos, refresh)] for _ in range(2)]
        d_idx = [idx, torch.empty_like(idx)]
        h2d = sum(t.numel() * t.element_size() for t in h_in)
        d2h = sum(t.numel() * t.element_size() for t in h_out[0])
        s_cp_in, s_cp_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def copy_in(j):
            for d_, h_ in zip(d_in[j], h_in):
                d_.copy_(h_, non_blocking=True)

        def compute(j):
            xi, posi, massi, loi = d_in[j]
            outi, cosi, refi = d_out[j]
            capi.dllm_kv_topk_gather(cache.handle, massi, loi, wl.block_len, k, d_idx[j], x_all, d_xtrk[j])
            capi.dllm_cache_project_drift(cache.handle, 0, xi, w, posi, None, outi, d_xtrk[j], d_idx[j], wl.gamma,
                                          cosi, refi)
            capi.dllm_cache_attend(cache.handle, 0, posi, None, outi)

        def copy_out(j):
            for h_, d_ in zip(h_out[j], d_out[j]):
                h_.copy_(d_, non_blocking=True)

        def capture(j):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                cap = torch.cuda.current_stream()
                s_cp_in.wait_stream(cap)
                s_cp_out.wait_stream(cap)
                with torch.cuda.stream(s_cp_in):
                    copy_in(j ^ 1)  # the next step's inputs
                with torch.cuda.stream(s_cp_out):
                    copy_out(j ^ 1)  # the previous step's results
                compute(j)
                cap.wait_stream(s_cp_in)
                cap.wait_stream(s_cp_out)
            return g

        graphs = [capture(0), capture(1)]
        # warm-up: two steps through the graphs
        copy_in(0)
        for i in range(4):
            graphs[i & 1].replay()
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        copy_in(0)
        for i in range(args.steps):
            graphs[i & 1].replay()
        copy_out((args.steps - 1) & 1)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        step_us = e0.elapsed_time(e1) * 1e3 / args.steps
        _, e2e_value = job_rate(e0.elapsed_time(e1), args.steps, world, dev)

        # the copies alone (no kernels), each direction and both at once, on the same
        # buffers and streams: the floor of a step that moves these bytes
        def copies_us(do_in, do_out, n=20):
            cur = torch.cuda.current_stream()
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(cur)
            s_cp_in.wait_stream(cur)
            s_cp_out.wait_stream(cur)
            for i in range(n):
                if do_in:
                    with torch.cuda.stream(s_cp_in):
                        copy_in(i & 1)
                if do_out:
                    with torch.cuda.stream(s_cp_out):
                        copy_out(i & 1)
            cur.wait_stream(s_cp_in)
            cur.wait_stream(s_cp_out)
            b_.record(cur)
            torch.cuda.synchronize(dev)
            return a_.elapsed_time(b_) * 1e3 / n

        t_in, t_out, t_both = copies_us(True, False), copies_us(False, True), copies_us(True, True)
        e2e = {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "graphs": "one CUDA graph per step: copy-in(i+1) | step(i) | read-back(i-1)",
               "host_buffers": "page-locked dllm_host_alloc blocks; the inputs written into them once, before the "
                               "timed region, with dllm_host_stage (streaming stores)",
               "inputs": "copied in every step: the block's hidden states, positions, previous-step mass and block "
                         "offsets; resident: cache, weights and the layer's hidden states of every position (the "
                         "tracked rows are gathered from them on the device)",
               "us_per_step": step_us,
               "copies_only": {"h2d_us": t_in, "h2d_gbs": h2d / t_in / 1e3, "d2h_us": t_out,
                               "d2h_gbs": d2h / t_out / 1e3, "both_us": t_both,
                               "frac": t_both / step_us,
                               "note": "the step's copies without its kernels, on the same page-locked buffers; "
                                       "frac = both_us / us_per_step"}}
        np.testing.assert_array_equal(h_out[(args.steps - 1) & 1][2].numpy(), refresh.cpu().numpy())

    # ---- fused vs the conventional four-kernel pipeline (projection GEMM, rotary, cache
    # write, attention as separate kernels with intermediates in HBM), same inputs and
    # L2 flush; the projection part of the unfused step is its total minus the attention
    fvu = None
    if not args.no_unfused:
        ws = torch.empty(capi.dllm_unfused_workspace_bytes(cache.handle, wl.x.shape[1], k), dtype=torch.uint8,
                         device=dev)
        n_cmp = min(args.steps, 200)

        def fused_pair():
            capi.dllm_cache_project_drift(cache.handle, 0, x, w, pos, None, out, x_probe, idx, wl.gamma, cos,
                                          refresh, stream=stream)
            capi.dllm_cache_attend(cache.handle, 0, pos, None, out, stream=stream)

        def unfused():
            capi.dllm_cache_step_unfused(cache.handle, 0, x, w, pos, None, out, ws, kv_x=x_probe,
                                         kv_positions=idx, probe_kv=probe, stream=stream)
            capi.dllm_kv_drift(cache.handle, 0, idx, probe, wl.gamma, cos, refresh, stream=stream)

        def separate_drift():  # the fused kernels with the drift test as its own launch
            capi.dllm_cache_project(cache.handle, 0, x, w, pos, None, out, kv_x=x_probe, kv_positions=idx,
                                    probe_kv=probe, stream=stream)
            capi.dllm_cache_attend(cache.handle, 0, pos, None, out, stream=stream)
            capi.dllm_kv_drift(cache.handle, 0, idx, probe, wl.gamma, cos, refresh, stream=stream)

        def timed(fn):
            return timed_us(fn, n_cmp)

        t_fused, t_unfused, t_sep = timed(fused_pair), timed(unfused), timed(separate_drift)
        # the per-position attention mass that the next step's top-k reads (optional
        # output; the workload's mass input stands in for it in the timed step)
        mass_out = torch.empty((B, S), dtype=torch.float32, device=dev)

        def with_mass():
            capi.dllm_cache_project_drift(cache.handle, 0, x, w, pos, None, out, x_probe, idx, wl.gamma, cos,
                                          refresh, stream=stream)
            capi.dllm_attention_mass(cache.handle, 0, pos, None, out, mass_out, stream=stream)
            capi.dllm_cache_attend(cache.handle, 0, pos, None, out, stream=stream)

        t_mass = timed(with_mass) - t_fused
        attend_us = statistics.mean(per["attend"]) * 1e3
        fvu = {"steps": n_cmp, "fused_project_attend_us": t_fused, "unfused_us": t_unfused,
               "ratio": t_unfused / t_fused,
               "projection_part": {"fused_us": statistics.mean(per["project"]) * 1e3,
                                   "unfused_us": t_unfused - attend_us,
                                   "ratio": (t_unfused - attend_us) / (statistics.mean(per["project"]) * 1e3)},
               "drift_as_own_launch_us": t_sep,
               "note": "fused = projection with the drift test in its epilogue, then attention; unfused = "
                       "projection GEMM to a bf16 workspace, rotary kernel, cache-write kernel (probes to a "
                       "buffer), attention, drift kernel; drift_as_own_launch = the fused projection storing the "
                       "probes, attention, drift kernel.  The pages quote 1.37x for their fused kernel alone "
                       "on an RTX 3090",
               "attention_mass_us": t_mass}

    # ---- ragged batches and partial softmax states over slot ranges, on this step's
    # rotated queries: ragged attention with seeded per-sequence key lengths, a partial
    # state over the last quarter of the slots, and the merge of two states.  Bytes are
    # algorithmic (keys and values read once, queries read, outputs written).
    nxt = None
    if not args.no_unfused:
        n_nx = min(args.steps, 200)
        n_tok = wl.x.shape[1]
        H, hd = s.n_heads, s.head_dim
        q_rows = torch.empty_like(out)
        capi.dllm_cache_project(cache.handle, 0, x, w, pos, None, q_rows, stream=stream)
        scratch = q_rows.clone()  # holds queries on entry; each call overwrites it with its output
        lens = np.random.default_rng(1234).integers(128, S + 1, size=B).astype(np.int32)
        key_len = torch.from_numpy(lens).to(dev)
        t_rag = timed_us(lambda: capi.dllm_cache_attend_ragged(cache.handle, 0, pos, key_len, scratch, stream=stream),
                         n_nx)
        rag_bytes = float(lens.sum()) * H * hd * 2 * 2 + 2 * B * n_tok * D * 2
        st_shape = (B, n_tok, H, hd + 2)
        st_a = torch.empty(st_shape, dtype=torch.float32, device=dev)
        st_b = torch.empty_like(st_a)
        lo = S - S // 4
        t_part = timed_us(lambda: capi.dllm_cache_attend_partial(cache.handle, 0, pos, q_rows, lo, S, st_a,
                                                                 stream=stream), n_nx)
        part_bytes = float(B) * (S - lo) * H * hd * 2 * 2 + B * n_tok * D * 2 + st_a.numel() * 4
        capi.dllm_cache_attend_partial(cache.handle, 0, pos, q_rows, 0, lo, st_b, stream=stream)
        t_merge = timed_us(lambda: capi.dllm_attend_merge(st_a, st_b, out=scratch, stream=stream), n_nx)
        merge_bytes = 2.0 * st_a.numel() * 4 + B * n_tok * D * 2
        # FACache reuse as one call: attention over the last quarter (the slots a step
        # rewrote) merged with the cached state of the rest, against one pass over all
        t_reuse = timed_us(lambda: capi.dllm_cache_attend_with_state(cache.handle, 0, pos, q_rows, lo, S, st_b, scratch,
                                                                     stream=stream), n_nx)
        reuse_bytes = float(B) * (S - lo) * H * hd * 2 * 2 + B * n_tok * D * 2 * 2 + st_b.numel() * 4
        t_onepass = timed_us(lambda: capi.dllm_cache_attend(cache.handle, 0, pos, None, scratch, stream=stream), n_nx)
        hbm = peaks()["hbm_gbs"]

        def row(us, nbytes, **kw):
            gbs = nbytes / (us * 1e-6) / 1e9
            return dict(us=us, algorithmic_bytes=nbytes, achieved_gbs=gbs, frac=gbs / hbm, **kw)

        nxt = {"steps": n_nx,
               "ragged": row(t_rag, rag_bytes, key_len="seeded uniform [128, %d], mean %.0f" % (S, lens.mean())),
               "partial_state": row(t_part, part_bytes, slots=[lo, S]),
               "merge": row(t_merge, merge_bytes),
               "facache_reuse": row(t_reuse, reuse_bytes, slots=[lo, S], one_pass_us=t_onepass,
                                    saving=t_onepass / t_reuse,
                                    note="attention over the rewritten slots merged in-kernel with the cached state "
                                         "of the others (dllm_cache_attend_with_state), against one pass over "
                                         "every slot")}

    others = None
    if not args.no_unfused and not args.no_elastic and rank == 0:
        others = other_configs(dev, flush)

    if nxt is not None and not args.no_elastic:
        nxt["elastic"] = elastic_leg(args, dev, B, S, D, s.n_heads, s.head_dim, s.rope_theta, wl.block_len, k,
                                     wl.gamma, flush)
        nxt["elastic_fp8"] = elastic_leg(args, dev, B, S, D, s.n_heads, s.head_dim, s.rope_theta, wl.block_len, k,
                                         wl.gamma, flush, kv_dtype=capi.DLLM_E4M3)

    rc, bits = cache.status()
    if rc != capi.DLLM_OK:
        raise RuntimeError(f"device status {bits:#x}")

    alg = algorithmic(wl)
    pk = peaks()
    cache_bytes = B * S * 2 * D * 2  # the layer's K and V
    mean = {kname: statistics.mean(v) for kname, v in per.items()}
    # every kernel against the slower of its two bounds (FLOPs at the bf16 burst peak,
    # algorithmic bytes at the copy peak)
    kernels = {
        "project": roofline_entry("project", mean["project"] * 1e3, alg["proj_flops"], alg["proj_bytes"], pk),
        "attend": roofline_entry("attend", mean["attend"] * 1e3, alg["attn_flops"], alg["attn_bytes"], pk),
        "topk_gather": {"kernel": "topk_gather", "us": mean["topk_gather"] * 1e3, "bound": "latency",
                        "algorithmic_bytes": alg["gather_bytes"],
                        "note": "top-32 of the previous step's mass and the copy of those tokens' hidden states, "
                                "one launch (one block per sequence)"},
    }
    for kname in ("project", "attend"):
        kernels[kname]["traffic"] = measured_traffic(kname)
    dom = "project" if mean["project"] >= mean["attend"] else "attend"
    kd = kernels[dom]
    # the contract's object describes the dominant kernel; per_kernel carries both graded
    # kernels (projection and attention) in the same form
    graded = []
    for kname in ("project", "attend"):
        e = kernels[kname]
        graded.append({"kernel": kname, "bound": e["bound"], "achieved": e["achieved"], "peak": e["peak"],
                       "unit": e["unit"], "frac": e["frac"], "traffic": e["traffic"], "us": e["us"]})
    roofline = {"kernel": dom, "bound": kd["bound"], "achieved": kd["achieved"], "peak": kd["peak"],
                "unit": kd["unit"], "frac": kd["frac"], "traffic": kd["traffic"],
                "peak_source": pk["source"] + (" burst" if kd["bound"] == "tensor" else ""),
                "per_kernel": graded}
    # top-k, gather, projection with the drift test, attention (+ the split-KV merge when
    # units < SMs)
    # top-k with the gather, projection, the drift test's finalize, attention (+ the split
    # merge when the units are fewer than the SMs)
    n_launch_per_step = 4 + (1 if B * s.n_heads < torch.cuda.get_device_properties(dev).multi_processor_count else 0)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": B, "d_model": D, "n_heads": s.n_heads, "head_dim": s.head_dim,
                   "cache_positions": S, "block": wl.block_len, "tracked_topk": k, "rope_theta": s.rope_theta,
                   "l2": "value: flushed between steps (256 MiB write); e2e: no flush, every step streams the "
                         + ("%.0f MiB cache (larger than L2)" % (cache_bytes / 2**20) if cache_bytes > L2_BYTES
                            else "%.1f MiB cache, which fits in L2 (e2e steps run L2-warm)" % (cache_bytes / 2**20)),
                   "timing": "value: K steps with events at step boundaries only; kernels: a second pass of "
                             "min(K, 300) steps with an event between every two kernels",
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": value * B * wl.block_len,
        "roofline": roofline, "kernels": kernels, "fused_vs_unfused": fvu, "next_rows": nxt, "other_configs": others,
        "e2e": e2e, "clocks": clk,
        "gpu_launches": n_launch_per_step * args.steps, "wall_s_timed": t_wall,
    }
    if world > 1:
        torch.distributed.destroy_process_group()
    return line, wl


# --------------------------------------------------------------------- CPU (oracle)
class OracleSample:
    """The fp64 oracle on sequence 0 of the workload: the cache of that sequence is
    filled once (untimed state before the step); ``rep()`` runs and times the whole
    step for it (top-k, probe projection, block projection + attention, drift)."""

    def __init__(self, wl):
        import oracle as O
        self.O, self.wl = O, wl
        s = wl.shape
        self.one = lambda a: None if a is None else a[0:1]  # noqa: E731
        self.cache = O.OracleCache(1, s.max_pos, 0, s.n_heads, s.head_dim)
        O.write_rows(self.cache, wl.w, self.one(wl.pre_x), self.one(wl.pre_pos), s.rope_theta)
        try:
            from threadpoolctl import threadpool_info
            self.cores = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
        except Exception:
            self.cores = os.cpu_count()
        self.threads = (f"up to {self.cores}: numpy's BLAS pool for the matrix products; "
                        "the oracle's loops and einsum contractions run on one thread")

    def rep(self) -> float:
        O, wl, one, s = self.O, self.wl, self.one, self.wl.shape
        t0 = time.perf_counter()
        idx = O.kv_topk(one(wl.mass), one(wl.block_lo), wl.block_len, wl.drift_k)
        xp = wl.probe_rows(idx)
        _, probe = O.step(self.cache, wl.w, s.rope_theta, one(wl.x)[:, :0], one(wl.positions)[:, :0], kv_x=xp,
                          kv_pos=idx, probe=True)
        O.step(self.cache, wl.w, s.rope_theta, one(wl.x), one(wl.positions))
        cos = O.kv_drift(self.cache, idx, probe)
        _ = cos.min() < wl.gamma
        return time.perf_counter() - t0


def _with_drift_inputs(wl):
    if wl.mass is None:  # batch-1 shape: track 32 positions under a uniform mass
        wl.mass = np.full((wl.shape.batch, wl.shape.max_pos), 1.0 / wl.shape.max_pos, np.float32)
        wl.drift_k = 32
    return wl


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.probe is not None:
        if rank == 0:
            probe(args)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        import workloads as W
        wl = _with_drift_inputs(W.make(args.workload))
        sample = OracleSample(wl)
        for _ in range(args.warmup):
            sample.rep()
        per_seq = [sample.rep() for _ in range(args.steps)]
        B = wl.shape.batch
        timed_s = sum(per_seq)
        # each timed step is one sequence of the B a layer-step covers: the layer-step rate
        # is steps / (B x timed seconds); ms_per_step is the measured time of one such step
        value = args.steps / (B * timed_s)
        sample_desc = ("each timed step: the whole step for sequence 0 of the batch (top-k, probe and block "
                       "projection, attention, drift), i.e. 1/%d of a layer-step" % B)
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * timed_s / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": wl.name, "batch": B},
                "layer_steps_per_timed_step": 1.0 / B, "timed_s": timed_s,
                "cpu_baseline": {"value": value, "unit": UNIT, "cores": sample.cores, "kind": "oracle",
                                 "threads": sample.threads, "sample": sample_desc,
                                 "ms_per_sequence": 1e3 * timed_s / args.steps, "sequences_per_layer_step": B},
                "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    line, wl = run_ours(args, rank, world, local)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample(wl)
        reps = []
        while sum(reps) < args.cpu_seconds or len(reps) < 2:
            reps.append(sample.rep())
        per_seq = statistics.mean(reps)
        line["cpu_baseline"] = {"value": 1.0 / (per_seq * wl.shape.batch), "unit": UNIT, "cores": sample.cores,
                                "kind": "oracle", "threads": sample.threads,
                                "sample": f"{len(reps)} repetitions of the whole step for sequence 0 of "
                                          f"{wl.shape.batch} (top-k, probe and block projection, attention, "
                                          f"drift); a layer-step covers all {wl.shape.batch} sequences",
                                "ms_per_sequence": 1e3 * per_seq, "sequences_per_layer_step": wl.shape.batch}
    if rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
