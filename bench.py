#!/usr/bin/env python3
"""MoE-layer throughput on one GB300 per rank.

Workload (default): the decode verify window -- one MoE layer, 4 tokens,
hidden 2048, 512 experts top-10, expert intermediate 512, a shared expert
(intermediate 512, sigmoid gate), 4-bit block-scaled weights, Zipf(1.1)
router bias, 50% of the experts resident in cache slots and the rest in
device staging slots.  One step = one pass of the hot path over a fresh
4-token window: router, top-k, expert groups with the residency lookup and
the heat-counter update (done by the grouping kernel), gate/up, down, and the
combine with the gated shared expert.
The timed steps go through 8 layers of this shape in turn (as a model's layers
follow one another), so each step's weights -- about 40 MB per layer, 320 MB in
all, against a 129 MB L2 -- are not in L2 when it runs; the K steps are timed
back to back with one CUDA-event pair.  The per-kernel durations behind the
roofline come from a separate pass on one layer with the L2 evicted before
every step (a 256 MB write, then a 256 MB read of another buffer).

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
the same workload instead (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

DEFAULT_WORKLOAD = "decode_t4_h2048_e512_k10"


# ------------------------------------------------------------------ replicas
def max_over_ranks(values, world: int, device: str = "cuda"):
    """Each value's maximum over the ranks: a job's time is its slowest replica's.  Needs the
    process group initialised when world > 1 (its backend must handle `device`)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_tokens_per_s(tokens_per_step: int, steps: int, world: int, job_ms: float) -> float:
    """Whole-job throughput: every replica's tokens over the slowest replica's time."""
    return tokens_per_step * steps * world / (job_ms / 1e3)


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-prefill", action="store_true", help="skip the secondary prefill-chunk measurement")
    p.add_argument("--layers", type=int, default=8,
                   help="layers of the workload's shape stepped through in turn (1 for small profiling runs)")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle sample budget for cpu_baseline")
    p.add_argument("--large", action="store_true",
                   help="also time the 4096-hidden, 256-expert top-6 model: its 4096-token prefill chunk and "
                        "batch-64 decode")
    p.add_argument("--no-stack", action="store_true", help="skip the 48-layer decode stack schedule")
    p.add_argument("--no-mixed", action="store_true",
                   help="skip the 8-layer prefill-then-decode run of the 4096-hidden model")
    p.add_argument("--stack-steps", type=int, default=2048)
    return p.parse_args()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", self.gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(self.rows),
                "power_w_max": max((float(r[3]) for r in self.rows if r[3].replace(".", "").isdigit()), default=None)}


def gpu_id_for(dev) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ------------------------------------------------------------- oracle leg
class OracleRunner:
    """The CPU oracle on windows of the workload, with the expert weights generated
    up front (input preparation, outside any timing)."""

    def __init__(self, w):
        from serving_router_top_gb300 import inputs as I
        self.w, self.I = w, I
        s = w.shape
        self.li = I.layer_inputs(w)
        self.experts = [I.expert_of(w, 0, e) for e in range(s.E)]
        mask = I.resident_mask(w.seed, 0, s.E, w.resident_frac)
        self.resid = np.where(mask, np.cumsum(mask) - 1, -1).astype(np.int32)
        self.stage = np.where(~mask, np.cumsum(~mask) - 1, -1).astype(np.int32)
        self.calls = 0

    def call(self, T: int) -> int:
        """One oracle layer call on a fresh window of T tokens; returns T."""
        from oracle import layer as olayer
        s, li = self.w.shape, self.li
        x = self.I.activations(self.w.seed, 1000 + self.calls, T, s.H)
        olayer.moe_layer(x, li.w_router, li.bias, s.k, self.experts.__getitem__, s.H, s.I, resid=self.resid,
                         stage=self.stage, shared=li.shared, I_shared=s.I_shared,
                         w_shared_gate_bits=li.w_shared_gate)
        self.calls += 1
        return T

    def sample(self, seconds: float, T=None):
        """Calls until ~`seconds` elapse: (tokens/s, tokens, calls, wall seconds)."""
        T = self.w.T if T is None else T
        tokens = calls = 0
        t0 = time.perf_counter()
        while True:
            tokens += self.call(T)
            calls += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return tokens / el, tokens, calls, el


def oracle_sample(w, seconds: float):
    return OracleRunner(w).sample(seconds)


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = w.shape
    cores = os.cpu_count()
    runner = OracleRunner(w)
    # size each step so warm-up + steps finish in about two and a half minutes
    t_call = runner.sample(0.0)[3]
    per_step = 150.0 / max(1, args.steps + args.warmup)
    T = w.T if t_call <= per_step else 1
    for _ in range(args.warmup):
        runner.call(T)
    t0 = time.perf_counter()
    tokens = 0
    for _ in range(args.steps):
        tokens += runner.call(T)
    el = time.perf_counter() - t0
    value = tokens / el
    sample = (f"{args.steps} oracle layer calls of {T} token(s) each (fp64 numpy, seeded windows of "
              f"{w.name}); expert weights pre-generated")
    out = {"impl": "reference", "metric": "moe_layer_tokens_per_s", "value": value, "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": w.name, "tokens_per_window": w.T, "hidden": s.H, "experts": s.E, "top_k": s.k,
                      "intermediate": s.I, "shared_intermediate": s.I_shared},
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ ours
class L2Flush:
    """Evicts the L2 (129 MB) before a timed step: a 256 MB write, then a 256 MB read
    of another buffer, so the write-back of the written lines happens here and not
    inside the next step (between real layers the L2 holds clean weight lines)."""

    def __init__(self):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(64 << 20, dtype=torch.int32, device="cuda")
        self.sink = torch.zeros((), dtype=torch.int32, device="cuda")

    def __call__(self):
        import torch
        self.w.zero_()
        torch.amax(self.r, dim=0, out=self.sink)



def algorithmic_bytes(st, G: int, T: int) -> dict:
    """Bytes each decode kernel must move at minimum for one window with G routed groups."""
    H, I_, E, k, Is = st.H, st.I, st.E, st.k, st.I_shared
    gu = G * 2 * I_ * (H // 2 + H // 16) + (2 * Is * (H // 2 + H // 16) if Is else 0)
    gu += T * H * 2 + (T * k + (T if Is else 0)) * I_ * 4           # activations in, h out
    dn = G * H * (I_ // 2 + I_ // 16) + (H * (Is // 2 + Is // 16) if Is else 0)
    dn += (T * k + (T if Is else 0)) * (I_ * 4 + H * 4)               # h in, o out
    router = E * H * 2 + T * H * 2 + T * E * 4
    # the single-kernel decode moves all of it (h stays on chip between its phases only
    # through L2, so its h traffic is counted as for the separate kernels)
    return {"gateup_decode": gu, "down_decode": dn, "router": router, "decode_fused": gu + dn + router}


def prefill_flops(st, T: int) -> dict:
    """Dense-equivalent FLOPs of the prefill GEMMs for a T-token chunk (every token's k experts + shared)."""
    H, I_, E, k, Is = st.H, st.I, st.E, st.k, st.I_shared
    return {"router": 2 * T * H * (E + (1 if Is else 0)),
            "gateup_gemm": 2 * (T * k * 2 * I_ * H + T * 2 * Is * H),
            "down_gemm": 2 * (T * k * H * I_ + T * H * Is)}


KERNEL_SOURCES = {"gateup_decode": "k_gemv.cu", "down_decode": "k_gemv.cu", "router": "k_route.cu",
                  "decode_fused": "k_decode.cu",
                  "gateup_gemm": "k_prefill.cu", "down_gemm": "k_prefill.cu"}


def source_sha1(name: str) -> str:
    import hashlib
    with open(os.path.join(ROOT, "serving_router_top_gb300", "csrc", name), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


def profiled_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary of `workload`
    (a line 'bench-traffic: kernel=K source=F sha1=S bytes=N'), or None when there is
    none or the kernel's source has changed since the counters were taken."""
    import glob
    import re
    pat = re.compile(r"bench-traffic:\s*kernel=(\S+)\s+source=(\S+)\s+sha1=(\w+)\s+bytes=(\d+)")
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", f"*{workload}*.md"))):
        with open(path) as f:
            for line in f:
                m = pat.search(line)
                if m and m.group(1) == kernel:
                    try:
                        if source_sha1(m.group(2)) == m.group(3):
                            return int(m.group(4))
                    except OSError:
                        pass
                    return None
    return None


def kernel_time_pass(st, step, set_input, flusher, steps: int, stream, groups_out=None):
    """Per-kernel durations (CUDA events recorded on the launching stream around each
    kernel, captured into a graph of the step) averaged over `steps` flushed steps.
    Kept out of the timed region: the event nodes lengthen the step.  When `groups_out`
    is a list, the routed-group count of every one of those steps is appended to it
    (the algorithmic bytes behind the durations are those of the same windows)."""
    import torch
    from serving_router_top_gb300 import moe
    ngroups = moe.device_view(st.ws.view.num_groups, (1,), "int32", st.ws)
    st.ws.set_profiling(True)
    set_input(0)
    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    sums, per_step = {}, 0
    for i in range(steps):
        set_input(i)
        flusher()
        g.replay()
        times = st.ws.kernel_times()
        per_step = len(times)
        if groups_out is not None:
            groups_out.append(int(ngroups.item()))
        for name, ms in times:
            sums[name] = sums.get(name, 0.0) + ms
    torch.cuda.synchronize()
    st.ws.set_profiling(False)
    del g
    return {n: v / steps for n, v in sums.items()}, per_step


def measure_policy(st, xs, ys, T, stream, n=16):
    """The cache policies' device costs on the bench's cache (CUDA events on the launching
    stream, medians over n calls): the heat policy's planning round over all layers, and the
    global LRU's per-call plan (K = 32 victims) and its execution (unmap, blob copies from the
    backing pool on a copy stream, publish), each after a real layer call whose groups it
    uses.  Run after the timed region: the LRU admissions change the residency."""
    import torch
    from serving_router_top_gb300 import moe
    K = 32
    plan = torch.zeros(96 * 5, dtype=torch.int32, device="cuda")
    n_dev = torch.zeros(1, dtype=torch.int32, device="cuda")
    copy_stream = torch.cuda.Stream()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    heat_ms, plan_ms, apply_ms, admitted = [], [], [], 0
    with torch.cuda.stream(stream):
        for _ in range(n):
            a, b = ev(), ev()
            a.record(stream)
            moe.cache_plan_swaps(st.cache, 1.5, 96, 0.7, plan, n_dev, stream=stream)
            b.record(stream)
            b.synchronize()
            heat_ms.append(a.elapsed_time(b))
        for i in range(n):
            layer = i % st.L
            st.forward(layer, xs[i % len(xs)], ys[layer], T, y_is_fp32=False, stream=stream)
            a, b, c = ev(), ev(), ev()
            a.record(stream)
            moe.cache_lru_plan(st.cache, st.ws, layer, K, plan, n_dev, stream=stream)
            b.record(stream)
            moe.moe_cache_apply_lru(st.cache, plan, n_dev, compute=stream, copy=copy_stream)
            c.record(stream)
            c.synchronize()
            plan_ms.append(a.elapsed_time(b))
            apply_ms.append(b.elapsed_time(c))
            admitted += int(n_dev.item())
    rc = moe.moe_sync_status(st.ws)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device error in the policy pass: {moe.strerror(rc)}")
    return {"heat_plan_round_us": 1e3 * statistics.median(heat_ms),
            "heat_plan_scope": f"{st.L} layers x {st.E} experts, threshold 1.5, at most 96 swaps, decay 0.7",
            "lru_plan_us": 1e3 * statistics.median(plan_ms),
            "lru_apply_us": 1e3 * statistics.median(apply_ms),
            "lru_admitted_per_call": admitted / n, "lru_K": K, "slots": st.cache.view.nslots,
            "note": "CUDA events on the launching stream; the LRU's apply includes the blob copies of its "
                    "admissions (the decode window's misses)"}


def prefill_timing(st, w, T, peaks, xs):
    """One prefill chunk of T tokens through layer 0 of st: CUDA graph, L2 flushed before each of
    20 replays, events on the launching stream; per-kernel times from a separate pass."""
    import torch
    from serving_router_top_gb300 import moe
    s = w.shape
    x_in = torch.empty_like(xs[0])
    y = torch.zeros((T, s.H), dtype=torch.int16, device="cuda")
    flusher = L2Flush()
    stream = torch.cuda.Stream()

    def step():
        st.forward(0, x_in, y, T, y_is_fp32=False, mode=moe.MOE_MODE_PREFILL, stream=stream)

    def set_input(i):
        x_in.copy_(xs[i % 2])

    with torch.cuda.stream(stream):
        set_input(0)
        step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        for i in range(3):
            set_input(i)
            flusher()
            g.replay()
        torch.cuda.synchronize()
        n = 20
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            set_input(i)
            flusher()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in ev) / n
        kt, _ = kernel_time_pass(st, step, set_input, flusher, 10, stream)
    rc = moe.moe_sync_status(st.ws)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device error in prefill measurement: {moe.strerror(rc)}")
    fl = prefill_flops(st, T)
    peak = float(peaks["bf16_tflops"])
    gemms = {}
    for name in ("router", "gateup_gemm", "down_gemm"):
        if name in kt:
            tf = fl[name] / (kt[name] / 1e3) / 1e12
            gemms[name] = {"us": 1e3 * kt[name], "tflops": tf, "frac": tf / peak}
    total = sum(fl.values())
    return {"workload": w.name, "tokens": T, "tokens_per_s": T / (ms / 1e3), "ms_per_layer": ms,
            "tflops_dense_equiv": total / (ms / 1e3) / 1e12, "peak_tflops": peak,
            "peak_source": "measured bf16_tflops (burst); the GEMMs run kind::f16 on bf16/f16 operands",
            "kernels_us": {n: 1e3 * v for n, v in kt.items()}, "gemms": gemms,
            "timing": f"{n} steps, CUDA graph, L2 flushed before each"}


def measure_prefill(args, peaks):
    """A short measurement of the prefill chunk (8192 tokens through one layer), then the
    same chunk with the layer's experts streamed through the staging pool."""
    import torch
    from serving_router_top_gb300 import inputs as I
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["prefill_t8192_h2048_e512_k10"]
    s, T = w.shape, w.T
    st = ModelState(w)
    xs = [torch.from_numpy(I.activations(w.seed, 20_000 + i, T, s.H).view(np.int16)).cuda() for i in range(2)]
    out = prefill_timing(st, w, T, peaks, xs)
    del st
    torch.cuda.empty_cache()
    out["streamed"] = {f"{src}_{nb}buf": measure_prefill_streamed(w, xs, on_device, buffers=nb)
                       for src, on_device in (("device", True), ("pinned_host", False)) for nb in (2, 1)}
    out["layers_streamed"] = measure_layers_streamed()
    return out


def measure_large(peaks, layers: int = 2, T_decode: int = 64, steps: int = 200):
    """The 4096-hidden, 256-expert top-6 model (I = I_shared = 2048), all experts resident:
    its 4096-token prefill chunk through one layer, and batch-64 decode stepping through
    `layers` layers in turn (their weights, 3.6 GB per layer, exceed the L2), captured as
    graphs of `layers` steps and timed back to back with one event pair."""
    import torch
    from serving_router_top_gb300 import inputs as I, moe
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["large_h4096_e256_k6"]
    s = w.shape
    st = ModelState(w, layers=layers)
    xs = [torch.from_numpy(I.activations(w.seed, 30_000 + i, w.T, s.H).view(np.int16)).cuda() for i in range(2)]
    pre = prefill_timing(st, w, w.T, peaks, xs)
    wins = [torch.from_numpy(I.activations(w.seed, 40_000 + i, T_decode, s.H).view(np.int16)).cuda()
            for i in range(4 * layers)]
    ys = [torch.zeros((T_decode, s.H), dtype=torch.int16, device="cuda") for _ in range(layers)]
    stream = torch.cuda.Stream()

    def steps_of(j):
        for l in range(layers):
            st.forward(l, wins[(j * layers + l) % len(wins)], ys[l], T_decode, y_is_fp32=False,
                       mode=moe.MOE_MODE_DECODE, stream=stream)

    with torch.cuda.stream(stream):
        steps_of(0)
        torch.cuda.synchronize()
        graphs = []
        for j in range(4):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                steps_of(j)
            graphs.append(g)
        for j in range(8):
            graphs[j % 4].replay()
        torch.cuda.synchronize()
        reps = max(1, steps // layers)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for j in range(reps):
            graphs[j % 4].replay()
        e1.record(stream)
        torch.cuda.synchronize()
    rc = moe.moe_sync_status(st.ws)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device error in the large-model measurement: {moe.strerror(rc)}")
    us = 1e3 * e0.elapsed_time(e1) / (reps * layers)
    out = {"workload": w.name, "prefill": pre,
           "decode": {"tokens_per_window": T_decode, "us_per_layer_step": us,
                      "tokens_per_s": T_decode / (us / 1e6), "layers_stepped": layers,
                      "timing": f"{reps * layers} layer steps in graphs of {layers}, back to back, one event pair"}}
    del st
    torch.cuda.empty_cache()
    return out


def measure_stack(Ts=(1, 2, 4, 8, 16), steps: int = 2048, layers: int = 48):
    """The 48-layer decode stack as specified: every step a fresh window of T tokens through
    48 layers (residual + RMSNorm between them, the heat update inside each layer's grouping),
    a planning round with its swaps every 256 steps, the router biases re-drawn every 512
    steps; 30% of the 48 x 512 experts resident in cache slots, every expert also staged.
    One graph of a whole step, replayed; the batch sizes run one after another on one cache."""
    import torch
    from serving_router_top_gb300 import inputs as I, moe
    from serving_router_top_gb300.stack import DecodeStack, run_schedule
    w = I.WORKLOADS["stack48_decode_h2048_e512_k10"]
    t0 = time.perf_counter()
    stk = DecodeStack(w, layers=layers, maxT=max(Ts), plan_every=256, drift_every=512)
    build_s = time.perf_counter() - t0
    st = stk.st
    stream = torch.cuda.Stream()
    blob = moe.moe_blob_bytes(st.H, st.I)
    fixed = st.E * st.H * 2 + blob  # router rows and the shared expert, every layer call
    out = {"workload": w.name, "layers": layers, "steps": steps, "slots": st.cache.view.nslots,
           "plan_every": 256, "drift_every": 512, "by_batch": {}}
    for T in Ts:
        windows = torch.from_numpy(np.stack([I.activations(w.seed, 50_000 + T * 100 + i, T, st.H)
                                             for i in range(16)]).view(np.int16)).cuda()
        win32 = (windows.view(torch.int16).to(torch.int32) << 16).view(torch.float32).contiguous()
        stats0 = st.cache.stats()
        ms, swaps, _, _ = run_schedule(stk, T, steps, win32, stream)
        groups = int((st.cache.stats() - stats0)[:, 0].sum())
        nbytes = groups * blob + steps * layers * fixed
        out["by_batch"][str(T)] = {"tokens_per_s": T * steps / (ms / 1e3), "ms": ms,
                                   "us_per_layer_step": 1e3 * ms / (steps * layers),
                                   "weight_GBps": nbytes / (ms / 1e3) / 1e9, "swaps_applied": swaps,
                                   "mean_groups_per_layer_call": groups / (steps * layers)}
    rc = moe.moe_sync_status(st.ws)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device error in the stack run: {moe.strerror(rc)}")
    out["build_s"] = build_s
    out["timing"] = ("CUDA events around each batch size's whole schedule (graph replays, the planning rounds "
                     "and drift between them); weight_GBps counts every distinct expert a layer call reads, "
                     "its router rows and the shared expert")
    del stk, st
    torch.cuda.empty_cache()
    return out


def measure_mixed(layers: int = 8, Tp: int = 4096, Td: int = 64, steps: int = 256):
    """The 4096-hidden, 256-expert top-6 model, all 8 layers resident: a 4096-token prefill
    chunk through the 8 layers, then 256 decode steps of 64 tokens (one graph per step)."""
    import torch
    from serving_router_top_gb300 import inputs as I, moe
    from serving_router_top_gb300.stack import DecodeStack, run_prefill_then_decode
    w = I.WORKLOADS["large_h4096_e256_k6"]
    t0 = time.perf_counter()
    stk = DecodeStack(w, layers=layers, maxT=Tp, plan_every=0, drift_every=0, stage_all=False)
    build_s = time.perf_counter() - t0
    st = stk.st
    stream = torch.cuda.Stream()
    to32 = lambda b: (torch.from_numpy(b.view(np.int16)).cuda().to(torch.int32) << 16).view(torch.float32)
    prompt = to32(I.activations(w.seed, 60_000, Tp, st.H))
    wins = torch.stack([to32(I.activations(w.seed, 61_000 + i, Td, st.H)) for i in range(8)])
    pre_ms, dec_ms, _, _ = run_prefill_then_decode(stk, prompt, wins, steps, stream)
    rc = moe.moe_sync_status(st.ws)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device error in the mixed run: {moe.strerror(rc)}")
    out = {"workload": w.name, "layers": layers, "prefill_tokens": Tp, "decode_batch": Td, "decode_steps": steps,
           "prefill_ms": pre_ms, "prefill_tokens_per_s": Tp / (pre_ms / 1e3),
           "decode_ms": dec_ms, "decode_tokens_per_s": Td * steps / (dec_ms / 1e3),
           "decode_us_per_layer_step": 1e3 * dec_ms / (steps * layers), "build_s": build_s,
           "timing": "CUDA events: the prefill chunk through every layer, then the decode steps (graph replays)"}
    del stk, st
    torch.cuda.empty_cache()
    return out


def measure_layers_streamed(layers: int = 4, n: int = 5):
    """Layers of the 8192-token prefill chunk with each layer's 512 experts streamed whole
    into one half of the staging pool one layer ahead (two buffers) or into one buffer (each
    copy waits for the previous layer), from pinned host memory and from HBM."""
    import torch
    from serving_router_top_gb300 import inputs as I, moe
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["prefill_t8192_h2048_e512_k10"]
    s, T = w.shape, w.T
    out = {"workload": w.name, "layers": layers}
    for on_device in (False, True):
        st = ModelState(w, layers=layers, resident=np.zeros((layers, s.E), dtype=bool), stage_rest=False, nslots=1,
                        nstaging=2 * s.E, backing_on_device=on_device)
        x0 = (torch.from_numpy(I.activations(w.seed, 70_000, T, s.H).view(np.int16)).cuda().to(torch.int32)
              << 16).view(torch.float32)
        xn = torch.zeros((T, s.H), dtype=torch.int16, device="cuda")
        y = torch.zeros((T, s.H), dtype=torch.int16, device="cuda")
        stream, copy = torch.cuda.Stream(), torch.cuda.Stream()
        descs = [st.layers[l].desc for l in range(layers)]
        # one layer's blobs copied alone (after a first, page-mapping copy), and beside a bf16
        # GEMM loop on the compute stream: what the copy engine delivers with and without
        # busy SMs
        nb = s.E * moe.moe_blob_bytes(s.H, s.I)
        stag = moe.device_view(st.cache.view.staging, (nb,), "uint8", st.cache)
        src = st.backing[:nb]
        A = torch.randn(4096, 4096, dtype=torch.bfloat16, device="cuda")
        for beside in (False, False, True):
            with torch.cuda.stream(copy):
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(copy)
                stag.copy_(src, non_blocking=True)
                c1.record(copy)
            if beside:
                with torch.cuda.stream(stream):
                    for _ in range(40):
                        A @ A
            torch.cuda.synchronize()
            key = f"{'device' if on_device else 'pinned_host'}_copy_{'beside_gemm' if beside else 'alone'}_GBps"
            out[key] = nb / (c0.elapsed_time(c1) / 1e3) / 1e9
        del A
        for buffers in (2, 1):
            with torch.cuda.stream(stream):
                x = x0.clone()
                moe.moe_layers_forward_streamed(descs, x, xn, y, T, st.cache, st.ws, buffers=buffers, stream=stream,
                                                copy_stream=copy)
                torch.cuda.synchronize()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(n):
                    x.copy_(x0)
                    moe.moe_layers_forward_streamed(descs, x, xn, y, T, st.cache, st.ws, buffers=buffers,
                                                    stream=stream, copy_stream=copy)
                e1.record(stream)
                torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / (n * layers)
            out[f"{'device' if on_device else 'pinned_host'}_{buffers}buf"] = {
                "ms_per_layer": ms, "tokens_per_s": T / (ms / 1e3),
                "weight_GBps": s.E * moe.moe_blob_bytes(s.H, s.I) / (ms / 1e3) / 1e9}
        rc = moe.moe_sync_status(st.ws)
        if rc != moe.MOE_OK:
            raise RuntimeError(f"device error in the layer-streamed prefill: {moe.strerror(rc)}")
        del st
        torch.cuda.empty_cache()
    out["timing"] = (f"{n} calls of {layers} layers back to back, events on the compute stream; per layer: "
                     "residual + RMSNorm, router, top-k, groups, the expert GEMMs on the layer's staged half")
    return out


def measure_prefill_streamed(w, xs, on_device: bool, U: int = 64, n: int = 8, buffers: int = 2):
    """The same chunk with every expert of the layer streamed from the backing pool (HBM, or
    pinned host memory over the host link) through the staging pool in units of U experts:
    with two buffers the copies on a second stream overlap the grouped GEMMs of the previous
    unit; with one, each copy waits for them (the second buffer off)."""
    import torch
    from serving_router_top_gb300 import moe
    from serving_router_top_gb300.model import ModelState
    s, T = w.shape, w.T
    st = ModelState(w, resident=np.zeros((1, s.E), dtype=bool), stage_rest=False, nslots=1, nstaging=2 * U,
                    backing_on_device=on_device)
    x_in = xs[0]
    y = torch.zeros((T, s.H), dtype=torch.int16, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(2):
            st.forward_streamed(0, x_in, y, T, U, y_is_fp32=False, stream=stream, buffers=buffers)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            st.forward_streamed(0, xs[i % 2], y, T, U, y_is_fp32=False, stream=stream, buffers=buffers)
        e1.record(stream)
        torch.cuda.synchronize()
    rc = moe.moe_sync_status(st.ws)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device error in streamed prefill: {moe.strerror(rc)}")
    ms = e0.elapsed_time(e1) / n
    nbytes = s.E * moe.moe_blob_bytes(s.H, s.I)
    out = {"backing": "device" if on_device else "pinned host", "units": f"{(s.E + U - 1) // U} of {U} experts",
           "buffers": buffers,
           "ms_per_layer": ms, "tokens_per_s": T / (ms / 1e3), "weight_GBps": nbytes / (ms / 1e3) / 1e9,
           "timing": f"{n} calls back to back, events on the compute stream (its last wait covers the copies)"}
    del st
    torch.cuda.empty_cache()
    return out


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    from serving_router_top_gb300 import build, inputs as I, moe
    from serving_router_top_gb300.model import ModelState

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        dist.barrier()
    s = w.shape
    T = w.T
    # NL layers of the workload's shape, stepped through in turn as a model would:
    # their weights (about 40 MB each) exceed the L2, so no step finds its
    # weights cached and no flush is needed between timed steps.
    NL = max(1, args.layers)
    # every expert also has a staging copy, so that an expert the policy pass (after the
    # timed steps) evicts stays reachable; lookups take a resident slot first, so the timed
    # steps see the same sources either way
    st = ModelState(w, layers=NL, stage_all=True)
    st.ws.set_fused_heat(True)  # the heat update runs inside the grouping kernel of each call
    P = 8 * NL  # distinct windows, resident in HBM before the timed region
    xs_host = [torch.from_numpy(I.activations(w.seed, 10_000 * rank + i, T, s.H).view(np.int16)).pin_memory()
               for i in range(P)]
    xs = [x.cuda() for x in xs_host]
    ys = [torch.zeros((T, s.H), dtype=torch.int16, device="cuda") for _ in range(NL)]  # bf16 output bits
    stream = torch.cuda.Stream()

    def layer_step(l, x):
        """One step: one layer call on a window, its heat update included (fused into the grouping)."""
        st.forward(l, x, ys[l], T, y_is_fp32=False, stream=stream)

    K = args.steps
    full, rem = K // NL, K % NL

    copy_stream = torch.cuda.Stream()

    def capture(n_layers, first_window, with_copies=False, x_pins=None, y_pins=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            if not with_copies:
                for l in range(n_layers):
                    layer_step(l, xs[first_window + l])
            else:
                # host copies on a second stream of the same graph: every window comes in up
                # front, each output goes back as soon as its layer call is done, so the
                # copies overlap the calls of the other layers (their windows are independent)
                fork = torch.cuda.Event()
                fork.record(stream)
                copy_stream.wait_event(fork)
                ev_in = [torch.cuda.Event() for _ in range(n_layers)]
                ev_out = [torch.cuda.Event() for _ in range(n_layers)]
                with torch.cuda.stream(copy_stream):
                    for l in range(n_layers):
                        xs[first_window + l].copy_(x_pins[l], non_blocking=True)
                        ev_in[l].record(copy_stream)
                for l in range(n_layers):
                    stream.wait_event(ev_in[l])
                    layer_step(l, xs[first_window + l])
                    ev_out[l].record(stream)
                with torch.cuda.stream(copy_stream):
                    for l in range(n_layers):
                        copy_stream.wait_event(ev_out[l])
                        y_pins[l].copy_(ys[l], non_blocking=True)
                join = torch.cuda.Event()
                join.record(copy_stream)
                stream.wait_event(join)
        return g

    # The C-ABI calls allocate nothing and never synchronise, so whole runs of
    # steps are captured as CUDA graphs and replayed.
    with torch.cuda.stream(stream):
        for l in range(NL):
            layer_step(l, xs[l])
        torch.cuda.synchronize()
        graphs = [capture(NL, j * NL) for j in range(P // NL)]
        g_rem = capture(rem, 0) if rem else None
        for i in range(max(1, (args.warmup + NL - 1) // NL)):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
    rc = moe.moe_sync_status(st.ws)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device error during warm-up: {moe.strerror(rc)}")

    # ---- timed region: exactly K steps back to back, one event pair on the launching stream
    sampler = ClockSampler(gpu_id_for(local))
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for r in range(full):
            graphs[r % len(graphs)].replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = e0.elapsed_time(e1)
    time.sleep(0.2)
    sampler.stop()
    rc = moe.moe_sync_status(st.ws)
    if rc != moe.MOE_OK:
        raise RuntimeError(f"device error in timed region: {moe.strerror(rc)}")

    # ---- per-kernel durations for the roofline (separate pass: layer 0, L2 evicted before each step)
    flusher = L2Flush()
    x_in = torch.empty_like(xs[0])
    G_steps = []
    with torch.cuda.stream(stream):
        kt, per_step = kernel_time_pass(st, lambda: layer_step(0, x_in), lambda i: x_in.copy_(xs[i % P]), flusher,
                                        min(K, 300), stream, groups_out=G_steps)
    G = statistics.mean(G_steps)  # the mean over the same windows whose durations are averaged
    launches = per_step * K  # the forward's kernels (the heat update inside the grouping), every step

    # ---- end to end through the C ABI with host buffers: each step's window is
    # copied from pinned host memory and its output copied back, inside the
    # graph and the timed region (on a second stream of the graph, overlapping the
    # other layers' calls); the host fills the pinned inputs between replays.
    x_pins = [torch.empty_like(xs_host[0]).pin_memory() for _ in range(NL)]
    y_pins = [torch.empty((T, s.H), dtype=torch.int16).pin_memory() for _ in range(NL)]
    with torch.cuda.stream(stream):
        g2 = capture(NL, 0, True, x_pins, y_pins)
        g2_rem = capture(rem, 0, True, x_pins, y_pins) if rem else None
        e2e_ms = 0.0
        for r in range(full + (1 if rem else 0)):
            n = NL if r < full else rem
            for l in range(n):
                x_pins[l].copy_(xs_host[(r * NL + l) % P])
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            (g2 if r < full else g2_rem).replay()
            b.record(stream)
            b.synchronize()
            e2e_ms += a.elapsed_time(b)
    torch.cuda.synchronize()

    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], world)
    value = job_tokens_per_s(T, args.steps, world, total_ms)
    e2e_value = job_tokens_per_s(T, args.steps, world, e2e_ms)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peaks, src = measured_peaks()
    by = algorithmic_bytes(st, G, T)
    dom = max((n for n in kt if n in by), key=lambda n: kt[n])
    if per_step == 1:
        # one kernel per step: its average launch duration is the timed region's own, the
        # event pair bracketing exactly K launches of it (the gaps between them count too)
        avg_ms = total_ms / args.steps
        duration = (f"the timed region's CUDA events / its {args.steps} launches (one kernel per step; the "
                    f"gaps between launches count against it)")
    else:
        avg_ms = kt[dom]
        duration = ("CUDA events around the kernel on its stream, separate pass of "
                    f"{min(args.steps, 300)} steps with the L2 evicted before each")
    achieved = by[dom] / (avg_ms / 1e3) / 1e9
    peak = float(peaks["hbm_gbs"])
    traffic = profiled_traffic(w.name, dom)
    clocks = sampler.summary()
    out = {
        "metric": "moe_layer_tokens_per_s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e2m1 weights; f16 x f16 -> f32 math", "data": "synthetic",
        "config": {"workload": w.name, "tokens_per_window": T, "hidden": s.H, "experts": s.E, "top_k": s.k,
                   "intermediate": s.I, "shared_intermediate": s.I_shared, "zipf_s": w.zipf_s,
                   "resident_frac": w.resident_frac, "layers_stepped": NL,
                   "l2": f"not flushed: the timed steps go through {NL} layers of this shape in turn, whose weights "
                         f"(about 40 MB each, {40 * NL} MB in all) exceed the 129 MB L2" if NL >= 4 else
                         f"{NL} layer(s) only: weights may stay in L2 (profiling run, not a bench number)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": f"{src} hbm_gbs",
                     "algorithmic_bytes_per_launch": by[dom], "avg_launch_us": avg_ms * 1e3,
                     "mean_routed_groups": G,
                     "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum of the committed ncu summary "
                                       "of this kernel (profiles/), used only while the kernel's source file "
                                       "matches the SHA-1 recorded there; not measured in this run",
                     "duration": duration,
                     "cold_launch_us": {n: 1e3 * v for n, v in kt.items()},
                     "cold_launch_note": "each kernel with the L2 evicted before every step (separate pass of "
                                         f"{min(args.steps, 300)} steps on one layer): the launch with no weight "
                                         "byte cached"},
        "kernels_us_per_step": {n: 1e3 * v for n, v in kt.items()},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * s.H * 2,
                "d2h_bytes_per_step": T * s.H * 2,
                "note": "each window copied in from pinned host memory and each output copied back inside the "
                        "timed graph replays, on a second stream of the graph (overlapping the other layers' "
                        "calls); the host refills the pinned inputs between replays"},
        "gpu_launches": launches,
    }
    with torch.cuda.stream(stream):
        out["policy"] = measure_policy(st, xs, ys, T, stream)
    if not args.no_prefill:
        out["prefill"] = measure_prefill(args, peaks)
    if args.large:
        out["large"] = measure_large(peaks)
    if not args.no_stack:
        out["stack"] = measure_stack(steps=args.stack_steps)
    if not args.no_mixed:
        out["mixed"] = measure_mixed()
    if not args.no_cpu_baseline:
        v, tok, calls, el = oracle_sample(w, args.cpu_seconds)
        out["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                               "sample": f"{calls} oracle layer calls x {w.T} tokens ({tok} tokens, {el:.1f} s), "
                                         f"fp64 numpy (BLAS threads over the host's cores), same workload, "
                                         f"seeded windows"}
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    from serving_router_top_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
