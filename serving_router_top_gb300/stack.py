"""Layer stacks: MoE layers in sequence over an fp32 residual stream, with the cache
policy running beside them.

Per step and layer: residual add of the previous layer's output and RMS
normalisation (moe_residual_rmsnorm), the layer forward (moe_layer_forward) with
its heat update inside the grouping; every ``plan_every`` steps a planning round
(cache_plan_swaps) and its copies and publication (moe_cache_apply_swaps, on a
copy stream beside the compute stream); every ``drift_every`` steps the routers'
Zipf biases are re-drawn (the hot set drifts).  This module only sequences C-ABI
calls; every step runs in libmoe's kernels.
"""
from __future__ import annotations

from typing import Callable, Optional

import numpy as np
import torch

from . import inputs as I
from . import moe
from .model import ModelState


class DecodeStack:
    def __init__(self, w: I.Workload, layers: Optional[int] = None, maxT: Optional[int] = None,
                 plan_every: int = 256, drift_every: int = 512, threshold: float = 1.5, max_swaps: int = 96,
                 decay: float = 0.7, eps: float = 1e-6, stage_all: bool = True):
        self.w = w
        self.st = ModelState(w, layers=layers, maxT=maxT, stage_all=stage_all)
        self.st.ws.set_fused_heat(True)  # the heat update runs inside each layer call's grouping
        s = w.shape
        self.L, self.H, self.k = self.st.L, s.H, s.k
        self.maxT = self.st.maxT
        self.plan_every, self.drift_every = plan_every, drift_every
        self.threshold, self.max_swaps, self.decay, self.eps = threshold, max_swaps, decay, eps
        dev = "cuda"
        self.xn = torch.zeros((self.maxT, self.H), dtype=torch.int16, device=dev)
        self.ys = [torch.zeros((self.maxT, self.H), dtype=torch.int16, device=dev) for _ in range(self.L)]
        self.plan = torch.zeros(max(max_swaps, 1) * 5, dtype=torch.int32, device=dev)
        self.n_plan = torch.zeros(1, dtype=torch.int32, device=dev)
        self.copy_stream = torch.cuda.Stream()
        self.epoch = 0
        self.ids_log: Optional[torch.Tensor] = None

    def set_epoch(self, epoch: int) -> None:
        """Re-draw every layer's router bias for drift epoch ``epoch`` (host copies into the
        bias tensors the layer calls read)."""
        self.epoch = epoch
        s = self.w.shape
        for l in range(self.L):
            b = I.zipf_bias(self.w.seed, l, s.E, self.w.zipf_s, epoch)
            self.st.layers[l].bias.copy_(torch.from_numpy(b))
            self.st.layers[l].host.bias = b

    def enable_ids_log(self, T: int) -> None:
        """Keep every layer call's top-k ids on the device (int32 [L, T, k] per step, appended by
        log_step); a step graph captured afterwards copies them too."""
        self.log_T = T
        self.ids_step = torch.zeros((self.L, T, self.k), dtype=torch.int32, device="cuda")

    def layers_pass(self, x_res: torch.Tensor, T: int, stream=None,
                    after_layer: Optional[Callable[[int], None]] = None) -> None:
        """All layers on the residual stream x_res (fp32 [T, H], updated in place), ending with
        the residual add of the last layer and its normalisation."""
        st = self.st
        prev = None
        topk = moe.device_view(st.ws.view.topk_ids, (self.maxT * self.k,), "int32", st.ws)
        for l in range(self.L):
            moe.moe_residual_rmsnorm(x_res, prev, self.xn, T, self.H, self.eps, stream=stream)
            st.forward(l, self.xn, self.ys[l], T, y_is_fp32=False, stream=stream)
            if getattr(self, "ids_step", None) is not None:
                self.ids_step[l].view(-1)[:T * self.k].copy_(topk[:T * self.k])
            if after_layer is not None:
                after_layer(l)
            prev = self.ys[l]
        moe.moe_residual_rmsnorm(x_res, prev, self.xn, T, self.H, self.eps, stream=stream)

    def maybe_drift(self, index: int) -> None:
        if self.drift_every and index % self.drift_every == 0 and index // self.drift_every != self.epoch:
            self.set_epoch(index // self.drift_every)

    def plan_round(self, index: int, after_plan: Optional[Callable[[], None]] = None, stream=None) -> bool:
        """After step `index`: a planning round and its swaps when the schedule says so."""
        if not (self.plan_every and (index + 1) % self.plan_every == 0):
            return False
        st = self.st
        compute = torch.cuda.current_stream() if stream is None else stream
        moe.cache_plan_swaps(st.cache, self.threshold, self.max_swaps, self.decay, self.plan, self.n_plan,
                             stream=compute)
        if after_plan is not None:
            after_plan()
        moe.moe_cache_apply_swaps(st.cache, self.plan, self.n_plan, compute, self.copy_stream)
        return True

    def step(self, x_res: torch.Tensor, T: int, index: int,
             after_layer: Optional[Callable[[int], None]] = None,
             after_plan: Optional[Callable[[], None]] = None) -> None:
        """One decode step of all layers on the residual stream x_res (fp32 [T, H], updated in place)."""
        self.maybe_drift(index)
        self.layers_pass(x_res, T, after_layer=after_layer)
        self.plan_round(index, after_plan)


def run_schedule(stk: DecodeStack, T: int, steps: int, windows: torch.Tensor, stream: torch.cuda.Stream,
                 log_ids: bool = False):
    """The decode schedule on a graph of one step: each step starts from a fresh window of
    token rows (windows fp32 [n, T, H], step s takes window s % n) and runs every layer; the
    planning rounds and the drift happen between replays, where the schedule puts them.
    Returns (elapsed ms of the whole schedule, swaps applied, ids log as numpy [steps, L, T, k]
    or None, plans as a list of numpy moe_swap arrays)."""
    x_res = torch.zeros((T, stk.H), dtype=torch.float32, device="cuda")
    src = torch.zeros_like(x_res)
    if log_ids:
        stk.enable_ids_log(T)
        log = torch.zeros((steps, stk.L, T, stk.k), dtype=torch.int32, device="cuda")
    else:
        stk.ids_step = None
    with torch.cuda.stream(stream):
        src.copy_(windows[0])
        x_res.copy_(src)
        stk.layers_pass(x_res, T, stream=stream)  # warm-up (first-call set-up outside the capture)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            x_res.copy_(src)
            stk.layers_pass(x_res, T, stream=stream)
        torch.cuda.synchronize()
    # the warm-up call added heat: start the schedule from a clean policy state
    stk.st.cache.tables()[2].zero_()
    swaps, plans = 0, []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_win = windows.shape[0]
    with torch.cuda.stream(stream):
        e0.record(stream)
        for s in range(steps):
            stk.maybe_drift(s)
            src.copy_(windows[s % n_win])
            g.replay()
            if log_ids:
                log[s].copy_(stk.ids_step)
            if stk.plan_round(s, stream=stream):
                n = int(stk.n_plan.item())  # one synchronisation per planning round
                swaps += n
                plans.append(stk.plan.cpu().numpy().view(moe.SWAP_DTYPE)[:n].copy())
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    return ms, swaps, (log.cpu().numpy() if log_ids else None), plans


def run_prefill_then_decode(stk: DecodeStack, prompt: torch.Tensor, decode_windows: torch.Tensor, steps: int,
                            stream: torch.cuda.Stream):
    """A mixed run: a prompt chunk (fp32 [Tp, H] residual rows) through every layer in the
    prefill path, then `steps` decode steps of decode_windows.shape[1] tokens each (step s
    starts from window s % n).  Returns (prefill ms, decode ms)."""
    Tp, Td = prompt.shape[0], decode_windows.shape[1]
    x_pre = prompt.clone()
    x_dec = torch.zeros((Td, stk.H), dtype=torch.float32, device="cuda")
    src = torch.zeros_like(x_dec)
    with torch.cuda.stream(stream):
        src.copy_(decode_windows[0])
        x_dec.copy_(src)
        stk.layers_pass(x_dec, Td, stream=stream)  # first-call set-up of the decode path
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            x_dec.copy_(src)
            stk.layers_pass(x_dec, Td, stream=stream)
        torch.cuda.synchronize()
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        e0.record(stream)
        stk.layers_pass(x_pre, Tp, stream=stream)
        e1.record(stream)
        for s in range(steps):
            src.copy_(decode_windows[s % decode_windows.shape[0]])
            g.replay()
        e2.record(stream)
        torch.cuda.synchronize()
    return e0.elapsed_time(e1), e1.elapsed_time(e2), x_pre, x_dec
