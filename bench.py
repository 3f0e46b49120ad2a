"""Benchmark of the routed MoE FFN layer on GB300.

One step = one pass of the whole layer (router, descriptors, fused gate+up
SwiGLU, down projection, combine with the shared expert) over one batch of
synthetic tokens, through the C ABI (moe_layer_forward), replayed as a CUDA
graph.  The headline workload is single-token decode (T = 1, d 4096, 256
experts, top-10, FFN 1024 + shared 1024, int4 g128); the same JSON line also
carries, under "secondary", the 32-token decode batch, the T = 2048
chunked-prefill pass and the T = 8192 skewed-routing pass (the latter also
with the grouped kernel's CTA scheduling switched off, MOE_FLAG_NO_SCHED).

Timing: the --steps steps of a config are one window, bracketed by a
synchronize (and a barrier across ranks) and timed with CUDA events on the
launching stream; windows are repeated (at least 5, and for at least a
second so that the clock sampler sees the load) and the median window is
reported.

Inputs larger than L2: each step reads a different copy of the packed
weights (NCOPY copies, each 1.67 GB) and a different activation batch, so
no step finds its weights in the 129 MB L2.

--impl reference times the CPU oracle (the plain C definition of the layer)
on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

HEADLINE = "decode1"
SECONDARY = "decode32,prefill2048,skew8192"
# secondary configs also timed with the W8A8 experts (fp8 weights and activations)
W8A8_CONFIGS = ("prefill2048", "skew8192")
FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)
# steps per timed window of each secondary config (about 0.1-0.5 s each)
SECONDARY_STEPS = {"decode1": 4000, "decode32": 1000, "prefill2048": 300, "skew8192": 60,
                   "tiny": 4000}
MIN_WINDOWS = 5
MIN_TIMED_S = 1.0  # default of --min-time
METRIC = "MoE-layer tokens/s at T=1 and T=2048; % of HBM / BF16 tensor-core roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

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
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------- GPU arm

def kernels_per_step(cfg, flags=0, fmt="w4"):
    """Kernels libmoe.so launches for one moe_layer_forward (memset nodes excluded)."""
    if fmt == "w8":  # router (2), descriptors (4), x quantiser, GEMM, H quantiser, GEMM, combine
        return 2 + 4 + 1 + 1 + 1 + 1 + 1
    gemv = (flags & 0x1) or (cfg.T <= 2 and not flags & 0x2)
    if gemv and cfg.T == 1 and flags & 0x8:
        return 1  # the cooperative single-launch step
    if gemv and cfg.T <= 64:
        return 3  # fused router + descriptors, gate+up GEMV, down GEMV + combine
    if gemv:
        return 2 + 4 + 2  # router (2), descriptors (4), the two GEMVs (combine fused)
    return 2 + 4 + 1 + 2 + 1  # router, descriptors, row gather, two grouped GEMMs, combine


class GpuBench:
    def __init__(self, cfg, device, ncopy: int, nbatch: int, flags: int = 0, fmt: str = "w4"):
        import torch

        import moe_expert_layer_sigmoid_gb300 as moe
        from workloads.device import upload

        self.torch, self.moe = torch, moe
        self.cfg = cfg
        self.device = device
        self.fmt = fmt
        self.layer = upload(cfg, device=device, extra_batches=nbatch - 1, fmt=fmt)
        L = self.layer
        self.xs = [L.x] + list(L.x_batches)
        # weight copies: copy 0 is the uploaded one; every copy has its own router
        # weights too, as every layer of a model does, so none stays in L2
        wrap = moe.w8 if fmt == "w8" else moe.w4
        self.copies = [L.w8s() if fmt == "w8" else L.w4s()]
        self.routers = [(L.W_r, L.bias)]
        self._keep = []
        for _ in range(ncopy - 1):
            ts = [t.clone() for t in (L.gu_q, L.gu_s, L.dn_q, L.dn_s, L.sgu_q, L.sgu_s, L.sdn_q,
                                      L.sdn_s, L.W_r, L.bias)]
            self._keep.append(ts)
            self.copies.append((wrap(ts[0], ts[1]), wrap(ts[2], ts[3]), wrap(ts[4], ts[5]),
                                wrap(ts[6], ts[7])))
            self.routers.append((ts[8], ts[9]))
        self.dims = L.dims()
        self.dims.flags = flags
        self.ws_bytes = (moe.moe_layer_workspace_bytes_w8a8 if fmt == "w8" else
                         moe.moe_layer_workspace_bytes)
        self.ws = moe.workspace(self.ws_bytes(self.dims), device)
        self.out = torch.empty((cfg.T, cfg.d), dtype=torch.int16, device=device)
        self.stream = torch.cuda.Stream(device)
        self.nslots = max(len(self.copies), len(self.xs))
        # the copies were made on the current stream; the steps run on self.stream, which
        # does not wait for it
        torch.cuda.synchronize(device)

    def step(self, i, stream=None):
        c = self.copies[i % len(self.copies)]
        wr, bias = self.routers[i % len(self.routers)]
        x = self.xs[i % len(self.xs)]
        fwd = self.moe.moe_layer_forward_w8a8 if self.fmt == "w8" else self.moe.moe_layer_forward
        fwd(x, wr, bias, self.dims, *c, self.out, self.ws, stream=stream)

    def capture(self):
        """One graph per slot, and one graph of all slots in a row (so that a
        replay is launched per nslots steps, not per step)."""
        torch = self.torch
        self.graphs = []
        with torch.cuda.stream(self.stream):
            for i in range(self.nslots):  # warm every slot once outside capture
                self.step(i, self.stream)
        self.stream.synchronize()
        for i in range(self.nslots):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                self.step(i, self.stream)
            self.graphs.append(g)
        self.round = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.round, stream=self.stream):
            for i in range(self.nslots):
                self.step(i, self.stream)
        torch.cuda.synchronize(self.device)

    def replay_steps(self, steps: int):
        """Enqueue exactly `steps` layer steps, rotating the slots."""
        full, rest = divmod(steps, self.nslots)
        for _ in range(full):
            self.round.replay()
        for i in range(rest):
            self.graphs[i].replay()

    def run(self, warmup: int, steps: int, clocks=None, min_time: float = MIN_TIMED_S):
        """Median ms per step over repeated windows of exactly `steps` steps (at least
        MIN_WINDOWS windows and MIN_TIMED_S seconds); the clock sampler runs across all
        windows.  Returns (median, per-window list)."""
        torch = self.torch
        with torch.cuda.stream(self.stream):
            self.replay_steps(warmup)
        torch.cuda.synchronize(self.device)
        if clocks is not None:
            clocks.start()
        per = []

        def window():
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(self.device)
            barrier()
            with torch.cuda.stream(self.stream):
                start.record(self.stream)
                self.replay_steps(steps)
                end.record(self.stream)
            end.synchronize()
            barrier()
            per.append(start.elapsed_time(end) / steps)

        window()
        # the same number of windows on every rank (each window is a barrier pair)
        n = max(MIN_WINDOWS, int(np.ceil(min_time / max(per[0] * steps * 1e-3, 1e-6))))
        n = int(max_over_ranks(float(min(n, 100000)), self.device))
        while len(per) < n:
            window()
        clk = clocks.stop() if clocks is not None else None
        return float(np.median(per)), per, clk

    def windows(self, enqueue, units: int, min_windows: int = MIN_WINDOWS):
        """Median ms per unit over at least min_windows CUDA-event windows, each running
        enqueue() (which issues `units` units of work) on the bench stream."""
        torch = self.torch
        per = []
        for _ in range(min_windows):
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize(self.device)
            with torch.cuda.stream(self.stream):
                start.record(self.stream)
                enqueue()
                end.record(self.stream)
            end.synchronize()
            per.append(start.elapsed_time(end) / units)
        return float(np.median(per))

    def descriptors(self, i):
        """Per-slot counts (read back outside any timed region)."""
        moe, torch = self.moe, self.torch
        T, k, E = self.cfg.T, self.cfg.k, self.cfg.E
        dims = self.dims
        ws = moe.workspace(self.ws_bytes(dims), self.device)
        i32 = dict(dtype=torch.int32, device=self.device)
        idx = torch.empty((T, k), **i32)
        w = torch.empty((T, k), dtype=torch.float32, device=self.device)
        counts, offsets = torch.empty(E, **i32), torch.empty(E + 1, **i32)
        perm, pos, sched = torch.empty(T * k, **i32), torch.empty(T * k, **i32), torch.empty(E, **i32)
        moe.moe_router_topk(self.xs[i % len(self.xs)], self.layer.W_r, self.layer.bias, dims, idx, w,
                            None, ws)
        moe.moe_build_descriptors(idx, dims, counts, offsets, perm, pos, sched, ws)
        torch.cuda.synchronize(self.device)
        return dict(idx=idx, w=w, counts=counts, offsets=offsets, perm=perm, pos=pos, sched=sched,
                    ws=ws)

    def time_gateup(self, warmup: int, steps: int):
        """Average duration of a standalone gate+up launch (moe_gateup_swiglu_w4a16 on
        precomputed descriptors, no prefetch from a router), CUDA events on its own
        stream, rotating weight copies and batches, replayed from a graph."""
        moe, torch = self.moe, self.torch
        descs = [self.descriptors(i) for i in range(self.nslots)]
        Fmax = max(self.cfg.F, self.cfg.Fs)
        H = torch.empty((self.cfg.rows, Fmax), dtype=torch.int16, device=self.device)

        def launch(i):
            dsc = descs[i % self.nslots]
            c = self.copies[i % len(self.copies)]
            if self.fmt == "w8":
                moe.moe_gateup_swiglu_w8a8(self.xs[i % len(self.xs)], self.dims, dsc["perm"],
                                           c[0], c[2], H, dsc["ws"], stream=self.stream)
            else:
                moe.moe_gateup_swiglu_w4a16(self.xs[i % len(self.xs)], self.dims, dsc["offsets"],
                                            dsc["perm"], dsc["sched"], c[0], c[2], H, dsc["ws"],
                                            stream=self.stream)

        with torch.cuda.stream(self.stream):
            for i in range(self.nslots):
                launch(i)
        self.stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=self.stream):
            for i in range(self.nslots):
                launch(i)
        reps_w = max(1, warmup // self.nslots)
        reps = max(1, steps // self.nslots)
        with torch.cuda.stream(self.stream):
            for _ in range(reps_w):
                g.replay()
        self.stream.synchronize()

        def enqueue():
            for _ in range(reps):
                g.replay()

        ms = self.windows(enqueue, reps * self.nslots)
        active = [int((d["counts"] > 0).sum().item()) for d in descs]
        return ms, active

    def e2e(self, warmup: int, steps: int):
        """moe_layer_forward_host: pinned host x in, pinned host out, captured as a graph."""
        moe, torch = self.moe, self.torch
        T, d = self.cfg.T, self.cfg.d
        xh = [torch.empty((T, d), dtype=torch.int16, pin_memory=True) for _ in self.xs]
        for a, b in zip(xh, self.xs):
            a.copy_(b.cpu())
        oh = torch.empty((T, d), dtype=torch.int16, pin_memory=True)
        def fwd(i):
            c = self.copies[i % len(self.copies)]
            wr, bias = self.routers[i % len(self.routers)]
            moe.moe_layer_forward_host(xh[i % len(xh)], wr, bias, self.dims, *c, oh, self.ws,
                                       stream=self.stream)

        graphs = []
        for i in range(self.nslots):
            with torch.cuda.stream(self.stream):
                fwd(i)
            self.stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                fwd(i)
            graphs.append(g)
        whole = torch.cuda.CUDAGraph()
        with torch.cuda.graph(whole, stream=self.stream):
            for i in range(self.nslots):
                fwd(i)

        def replay(n):
            full, rest = divmod(n, self.nslots)
            for _ in range(full):
                whole.replay()
            for i in range(rest):
                graphs[i].replay()

        with torch.cuda.stream(self.stream):
            replay(warmup)
        torch.cuda.synchronize(self.device)
        ms = self.windows(lambda: replay(steps), steps)
        return ms, 2 * T * d, 2 * T * d

    def free(self):
        self.graphs = []
        self.round = None
        self._keep = []
        self.copies = []
        self.layer = None
        self.torch.cuda.empty_cache()


# DRAM bytes (read + write) per step of the decode chain at decode1, summed over
# router_decode_kernel, gateup_gemv_kernel and down_gemv_kernel of one step, from
# one `ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum` capture of this
# code (cold caches, --ncopy 1 --nbatch 1, one step of three launches).
DECODE1_TRAFFIC = 4_269_312 + 48_596_992 + 23_854_848


def gpu_roofline_decode(cfg, ms, active, pk, pk_kind, gu_ms, flags=0):
    """The decode step against HBM.  Algorithmic bytes = packed int4 weights + fp16 scales
    of the active routed experts and of the shared expert (gate+up and down), per step.
    The step is three launches (fused router, gate+up GEMV, down GEMV + combine) and the
    router's L2 prefetch moves expert bytes across their boundaries, so the unit is the
    step (one graph node sequence), timed with CUDA events on its stream."""
    nbytes = float(np.mean([(a + 1) * cfg.packed_expert_bytes() for a in active]))
    achieved = nbytes / (ms * 1e-3) / 1e9
    peak = pk["hbm_gbs"]
    router_bytes = cfg.E * cfg.d * 4
    kernel_of_step = kernels_per_step(cfg, flags)
    kernel = ("decode step: router_decode_kernel + gateup_gemv_kernel + down_gemv_kernel"
              if kernel_of_step == 3 else
              "layer step on the grouped path (router, descriptors, gather, grouped GEMMs, combine)")
    return {"kernel": kernel,
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": (DECODE1_TRAFFIC if cfg.name == "decode1" and kernel_of_step == 3
                        else None),
            "bytes_per_step": int(nbytes),
            "router_weight_bytes_not_counted": router_bytes,
            "step_us": round(ms * 1e3, 3),
            "standalone_gateup_us": round(gu_ms * 1e3, 3),
            "peak_source": f"{pk_kind} hbm_gbs"}


# DRAM bytes (read + write) of one gate+up launch at prefill2048 from one
# `ncu --set full` capture of grouped_w4a16_kernel on this code (cold caches).
PREFILL2048_GATEUP_TRAFFIC = 356_328_704 + 47_281_664


def gpu_roofline_prefill(cfg, gu_ms, pk, pk_kind):
    """Gate+up kernel at prefill: algorithmic flops = 2 * (2F) * d per routed slot and per
    shared row."""
    flops = 2.0 * 2 * cfg.d * (cfg.F * cfg.slots + cfg.Fs * cfg.T)
    achieved = flops / (gu_ms * 1e-3) / 1e12
    peak = pk["bf16_tflops"]
    return {"kernel": "gateup", "bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
            "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "traffic": PREFILL2048_GATEUP_TRAFFIC if cfg.name == "prefill2048" else None,
            "flops_per_launch": flops, "launch_us": round(gu_ms * 1e3, 2),
            "peak_source": f"{pk_kind} bf16_tflops"}


def measure_config(name, device, warmup, steps, ncopy, nbatch, pk, pk_kind, gpu_index, flags=0,
                   ab_flags=None, min_time=MIN_TIMED_S, fmt="w4"):
    """Layer step (median of windows, clocks sampled across them), the standalone gate+up
    launch, and the end-to-end host call, on one config.  With ab_flags, the layer step
    and the gate+up launch are timed again with those flags (same inputs)."""
    cfg = workloads.CONFIGS[name]
    b = GpuBench(cfg, device, ncopy=ncopy, nbatch=nbatch, flags=flags, fmt=fmt)
    b.capture()
    ms, per, clk = b.run(warmup, steps, ClockSampler(gpu_index), min_time)
    gu_ms, active = b.time_gateup(warmup, steps)
    # the host-buffer entry point is the W4A16 layer's
    e2e_ms, h2d, d2h = b.e2e(warmup, steps) if fmt == "w4" else (None, 0, 0)
    layer_bytes = float(np.mean([(a + 1) * cfg.packed_expert_bytes() for a in active]))
    res = dict(cfg=cfg, ms=ms, windows=per, clocks=clk, gu_ms=gu_ms, active=active,
               e2e_ms=e2e_ms, h2d=h2d, d2h=d2h, layer_bytes=layer_bytes,
               packed_copies=len(b.copies), batches=len(b.xs), steps=steps, flags=flags)
    if ab_flags is not None:
        b.dims.flags = ab_flags
        b.capture()
        ms_ab, per_ab, clk_ab = b.run(warmup, steps, ClockSampler(gpu_index), min_time)
        gu_ab, _ = b.time_gateup(warmup, steps)
        res["ab"] = dict(flags=ab_flags, ms=ms_ab, windows=per_ab, clocks=clk_ab, gu_ms=gu_ab)
    b.free()
    return res


# ---------------------------------------------------------------- CPU oracle

def oracle_sample(cfg, budget_s: float, max_tokens: int):
    """Time the oracle (router + experts + combine) on tokens of the workload until about
    budget_s of CPU work; experts are quantised beforehand (load time, untimed).
    Returns (tokens, seconds)."""
    import oracle
    done, spent, batch = 0, 0.0, 0
    wr, bias = workloads.gen_router(cfg)
    cache = {}

    def packed(e):
        if e not in cache:
            cache[e] = (oracle.pack_w4(workloads.gen_gateup(cfg, e), cfg.group),
                        oracle.pack_w4(workloads.gen_down(cfg, e), cfg.group))
        return cache[e]

    sq_gu, sq_dn = packed(-1)
    while spent < budget_s and done < max_tokens:
        x = workloads.gen_x(cfg, batch)[:1]
        idx, w, _, _ = oracle.router(x, wr, bias, cfg.k)
        sel = idx[0]
        for e in sel:
            packed(int(e))
        # a compact expert stack holding only the selected experts (relabelled 0..k-1)
        W = oracle.PackedLayer(
            np.stack([cache[int(e)][0][0] for e in sel]), np.stack([cache[int(e)][0][1] for e in sel]),
            np.stack([cache[int(e)][1][0] for e in sel]), np.stack([cache[int(e)][1][1] for e in sel]),
            sq_gu[0], sq_gu[1], sq_dn[0], sq_dn[1], cfg.group)
        local_idx = np.arange(cfg.k, dtype=np.int32)[None, :]
        t0 = time.perf_counter()
        oracle.router(x, wr, bias, cfg.k)
        oracle.layer_tokens(x, W, local_idx, w, np.array([0]))
        spent += time.perf_counter() - t0
        done += 1
        batch += 1
    return done, spent


# ---------------------------------------------------------------- main

def barrier():
    """A barrier across ranks when a process group is up."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(x: float, device="cpu") -> float:
    """The largest of a per-rank value over the process group (the slowest rank's step time
    sets the job's throughput); the value itself when no group is initialised."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def config_dict(cfg, ncopy: int, nbatch: int) -> dict:
    """The workload, worded identically in both arms."""
    return {
        "workload": f"{cfg.name}: T={cfg.T}, d={cfg.d}, E={cfg.E}, top-{cfg.k}, F={cfg.F}, "
                    f"shared F={cfg.Fs}, int4 g{cfg.group}, seed {cfg.seed}",
        "l2": f"inputs larger than L2: {ncopy} copies of the expert and router weights x "
              f"{nbatch} activation batches, rotated per step",
    }


def timing_dict(res) -> dict:
    w = res["windows"]
    return {"method": "CUDA graph replay of moe_layer_forward; CUDA events on the launching "
                      "stream around each window of --steps steps; median window reported",
            "windows": len(w), "steps_per_window": res["steps"],
            "ms_per_step_min": round(min(w), 5), "ms_per_step_max": round(max(w), 5)}


def e2e_dict(res) -> dict:
    cfg = res["cfg"]
    return {"value": round(cfg.T / (res["e2e_ms"] * 1e-3), 2), "unit": "tokens/s",
            "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
            "ms_per_step": round(res["e2e_ms"], 5),
            "mode": "graph replay of moe_layer_forward_host (pinned host x and out), "
                    "median of 5 windows"}


def roofline_of(res, ms, pk, pk_kind) -> dict:
    cfg = res["cfg"]
    if cfg.T <= 64:  # decode: weight streaming against HBM, per step
        return gpu_roofline_decode(cfg, ms, res["active"], pk, pk_kind, res["gu_ms"],
                                   res["flags"])
    # prefill: the gate+up grouped kernel against the dense bf16 peak
    roof = gpu_roofline_prefill(cfg, res["gu_ms"], pk, pk_kind)
    roof["layer_tflops"] = round(cfg.flops() / (ms * 1e-3) / 1e12, 2)
    roof["layer_frac_of_bf16_peak"] = round(roof["layer_tflops"] / pk["bf16_tflops"], 4)
    return roof


def w8a8_entry(res, base, pk, pk_kind) -> dict:
    """The W8A8 layer on the same workload, against the fp8 peak (the measured bf16
    peak times the nominal fp8 / bf16 ratio) and against the W4A16 layer (base)."""
    cfg = res["cfg"]
    flops = 2.0 * 2 * cfg.d * (cfg.F * cfg.slots + cfg.Fs * cfg.T)
    tf = flops / (res["gu_ms"] * 1e-3) / 1e12
    peak = pk["bf16_tflops"] * FP8_OVER_BF16
    layer_tf = cfg.flops() / (res["ms"] * 1e-3) / 1e12
    return {
        "experts": "W8A8: E4M3 weights (one scale per row) x E4M3 activations (one scale per "
                   "row), tcgen05 kind::f8f6f4",
        "value": round(cfg.T / (res["ms"] * 1e-3), 1), "unit": "tokens/s",
        "us_per_layer": round(res["ms"] * 1e3, 2),
        "layer_tflops": round(layer_tf, 2),
        "timing": timing_dict(res),
        "roofline": {"kernel": "gateup (grouped_w8a8_kernel)", "bound": "tensor",
                     "achieved": round(tf, 2), "peak": round(peak, 1), "unit": "TFLOP/s",
                     "frac": round(tf / peak, 4), "traffic": None, "flops_per_launch": flops,
                     "launch_us": round(res["gu_ms"] * 1e3, 2),
                     "peak_source": f"{pk_kind} bf16_tflops x {FP8_OVER_BF16} (nominal fp8/bf16)"},
        "speedup_vs_w4a16_layer": round(base["ms"] / res["ms"], 3),
        "speedup_vs_w4a16_gateup": round(base["gu_ms"] / res["gu_ms"], 3),
        "clocks": res["clocks"],
    }


def secondary_entry(res, pk, pk_kind) -> dict:
    cfg = res["cfg"]
    ms = res["ms"]
    tf = cfg.flops() / (ms * 1e-3) / 1e12
    ent = {
        "workload": config_dict(cfg, res["packed_copies"], res["batches"])["workload"],
        "value": round(cfg.T / (ms * 1e-3), 1), "unit": "tokens/s",
        "us_per_layer": round(ms * 1e3, 2),
        "layer_tflops": round(tf, 2),
        "layer_frac_of_bf16_peak": round(tf / pk["bf16_tflops"], 4),
        "active_experts_mean": float(np.mean(res["active"])),
        "kernels_per_step": kernels_per_step(cfg, res["flags"]),
        "timing": timing_dict(res),
        "roofline": roofline_of(res, ms, pk, pk_kind),
        "clocks": res["clocks"],
        "e2e": e2e_dict(res),
    }
    if "w8" in res:
        ent["w8a8"] = w8a8_entry(res["w8"], res, pk, pk_kind)
    if "ab" in res:
        ab = res["ab"]
        ent["no_sched"] = {
            "flags": "MOE_FLAG_NO_SCHED (expert-id tile order, no N-banding)",
            "us_per_layer": round(ab["ms"] * 1e3, 2),
            "gateup_us": round(ab["gu_ms"] * 1e3, 2),
            "windows": len(ab["windows"]), "clocks": ab["clocks"],
            "sched_speedup_layer": round(ab["ms"] / ms, 4),
            "sched_speedup_gateup": round(ab["gu_ms"] / res["gu_ms"], 4),
        }
    return ent


SWEEP_T = (1, 2, 3, 4, 6, 8, 16, 32, 64, 128, 256)


def run_sweep(args, device, gpu_index):
    """Layer time per step against T on each forced expert path (and the tensor-core
    single-token step at T = 1), on one uploaded layer of the decode shapes: the
    weights of decode1's seed, x the first T rows of each 256-token batch."""
    import dataclasses

    import torch
    base = workloads.CONFIGS[args.config]
    tmax = max(SWEEP_T)
    cfg = dataclasses.replace(base, name=f"{base.name}_sweep", T=tmax)
    b = GpuBench(cfg, device, ncopy=args.ncopy, nbatch=args.nbatch)
    moe = b.moe
    full_x, full_out = list(b.xs), b.out
    paths = [("gemv", 0x1), ("grouped", 0x2)]
    rows = []
    for T in SWEEP_T:
        for name, flags in paths + ([("mma_step", 0x9)] if T == 1 else []):
            dims = b.layer.dims(flags, T=T)
            if moe.moe_layer_workspace_bytes(dims) > b.ws.numel():
                continue
            b.dims = dims
            b.xs = [x[:T] for x in full_x]
            b.out = full_out[:T]
            b.capture()
            # about 0.2 s per window
            t0 = time.perf_counter()
            with torch.cuda.stream(b.stream):
                b.replay_steps(b.nslots)
            torch.cuda.synchronize(device)
            est = max((time.perf_counter() - t0) / b.nslots, 1e-6)
            steps = int(min(20000, max(b.nslots, 0.2 / est)))
            ms, per, _ = b.run(args.warmup, steps, None, 0.0)
            rows.append({"T": T, "path": name, "us_per_layer": round(ms * 1e3, 2),
                         "tokens_per_s": round(T / (ms * 1e-3), 1), "windows": len(per),
                         "steps_per_window": steps})
            print(f"T={T:4d} {name:9s} {ms * 1e3:10.2f} us", file=sys.stderr, flush=True)
    b.free()
    print(json.dumps({"sweep": rows, "workload": f"{base.name} shapes, T = 1..{tmax}",
                      "l2": f"{args.ncopy} weight copies x {args.nbatch} batches rotated"}),
          flush=True)
    return 0


REF_BUDGET_S = 120.0  # cap on the reference arm's timed oracle work


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cfg = workloads.CONFIGS[args.config]
    # warm-up: one oracle token, untimed
    oracle_sample(cfg, budget_s=0.0, max_tokens=max(0, min(args.warmup, 1)))
    # one token per step, bounded: at most REF_BUDGET_S of oracle work, so the arm ends within
    # a few minutes whatever --steps is (the oracle takes ~0.13 s per decode1 token)
    n, sec = oracle_sample(cfg, budget_s=REF_BUDGET_S, max_tokens=args.steps)
    tps = n / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": round(tps, 4), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec / n * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (fp64 router)", "data": "synthetic",
        "config": config_dict(cfg, args.ncopy, args.nbatch),
        "step": "one token of the workload through the oracle",
        "parallelism": "rank 0 only, one host thread",
        "steps_timed": n,
        "cpu_baseline": {"value": round(tps, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} tokens of {cfg.name}, one per step, single thread "
                                   f"(at most {REF_BUDGET_S:.0f} s of oracle work)",
                         **host_cpu()},
        "e2e": {"value": round(tps, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def host_cpu():
    """The host the oracle ran on: processor name (best effort) and its core count."""
    name = ""
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "hardware", "cpu part") and ":" in ln:
                    name = ln.split(":", 1)[1].strip()
                    if key == "model name":
                        break
    except OSError:
        pass
    return {"cpu": name or platform.processor() or platform.machine(), "nproc": os.cpu_count()}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=HEADLINE, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--secondary", default=SECONDARY,
                    help="comma-separated extra configs in the same line ('none': no extra config)")
    ap.add_argument("--secondary-steps", type=int, default=0,
                    help="steps per timed window of each extra config (0: a per-config default)")
    ap.add_argument("--ncopy", type=int, default=8)
    ap.add_argument("--nbatch", type=int, default=8)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--fmt", default="w4", choices=["w4", "w8"],
                    help="expert weights of the headline config: int4 (W4A16) or fp8 (W8A8)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the layer against T on each forced expert path (one JSON line)")
    ap.add_argument("--no-w8a8", action="store_true",
                    help="skip the W8A8 timings of the prefill configs")
    ap.add_argument("--min-time", type=float, default=MIN_TIMED_S,
                    help="repeat timed windows for at least this many seconds (>= 5 windows)")
    ap.add_argument("--flags", type=int, default=0,
                    help="moe_dims_t.flags for the headline config (1: force GEMV, 2: force grouped)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)

    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = f"cuda:{local}"
    pk, pk_kind = peaks()
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local]) \
        if "CUDA_VISIBLE_DEVICES" in os.environ else local

    if args.sweep:
        return run_sweep(args, device, gpu_index)
    if world > 1:
        dist.barrier()
    main_res = measure_config(args.config, device, args.warmup, args.steps, args.ncopy,
                              args.nbatch, pk, pk_kind, gpu_index, flags=args.flags,
                              min_time=args.min_time, fmt=args.fmt)
    sec_names = [] if args.secondary in ("", "none", '""') else \
        [n for n in args.secondary.split(",") if n and n != args.config]
    sec_res = []
    for name in sec_names:
        steps = args.secondary_steps or SECONDARY_STEPS.get(name, 100)
        # the skewed config also runs without the grouped kernel's CTA scheduling
        ab = 0x4 if workloads.CONFIGS[name].bias == "zipf" else None
        r = measure_config(name, device, args.warmup, steps, args.ncopy, args.nbatch, pk, pk_kind,
                           gpu_index, ab_flags=ab, min_time=args.min_time)
        if name in W8A8_CONFIGS and not args.no_w8a8:
            r["w8"] = measure_config(name, device, args.warmup, steps, args.ncopy, args.nbatch, pk,
                                     pk_kind, gpu_index, min_time=args.min_time, fmt="w8")
        sec_res.append(r)
    ms = max_over_ranks(main_res["ms"], device)
    cfg = main_res["cfg"]
    value = world * cfg.T / (ms * 1e-3)

    cpu = None
    if rank == 0 and world == 1 and args.cpu_budget > 0:
        n, sec = oracle_sample(cfg, args.cpu_budget, 10 ** 6)
        cpu = {"value": round(n / sec, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
               "sample": f"{n} single tokens of {cfg.name} (router + {cfg.k} experts + shared), "
                         f"{sec:.1f} s of single-thread CPU work", **host_cpu()}

    if rank == 0:
        roof = (roofline_of(main_res, ms, pk, pk_kind) if args.fmt == "w4" else
                w8a8_entry(main_res, main_res, pk, pk_kind)["roofline"])
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "us_per_layer": round(ms * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": ("int4 weights x bf16 activations, f32 accumulate" if args.fmt == "w4" else
                      "e4m3 weights x e4m3 activations, f32 accumulate"),
            "data": "synthetic (seeded generator, random weights of the layer's shapes)",
            "config": config_dict(cfg, args.ncopy, args.nbatch),
            "parallelism": f"{world} replicas, no collective" if world > 1 else "single GPU",
            "timing": timing_dict(main_res),
            "roofline": roof,
            "active_experts_mean": float(np.mean(main_res["active"])),
            "clocks": main_res["clocks"],
            "e2e": e2e_dict(main_res) if args.fmt == "w4" else None,
            "gpu_launches": kernels_per_step(cfg, args.flags, args.fmt) * args.steps,
            "kernels_per_step": kernels_per_step(cfg, args.flags, args.fmt),
            "cpu_baseline": cpu,
            "peaks": f"{pk_kind} (MEASURED_PEAKS.json)" if pk_kind == "measured" else "fallback",
        }
        if sec_res:
            line["secondary"] = [secondary_entry(r, pk, pk_kind) for r in sec_res]
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
