"""The decode-stack workload: MoE layers in sequence over an fp32 residual stream,
with the cache policy running beside them.

Per step and layer: residual add of the previous layer's output and RMS
normalisation (moe_residual_rmsnorm), the layer forward (moe_layer_forward), its
heat update (cache_heat_update); every ``plan_every`` steps a planning round
(cache_plan_swaps) and its copies and publication (moe_cache_apply_swaps, on a
copy stream beside the compute stream); every ``drift_every`` steps the
routers' Zipf biases are re-drawn (the hot set drifts).  This module only
sequences C-ABI calls; every step runs in libmoe's kernels.
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
                 decay: float = 0.7, eps: float = 1e-6):
        self.w = w
        self.st = ModelState(w, layers=layers, maxT=maxT, stage_all=True)
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

    def set_epoch(self, epoch: int) -> None:
        """Re-draw every layer's router bias for drift epoch ``epoch``."""
        self.epoch = epoch
        s = self.w.shape
        for l in range(self.L):
            b = I.zipf_bias(self.w.seed, l, s.E, self.w.zipf_s, epoch)
            self.st.layers[l].bias.copy_(torch.from_numpy(b))
            self.st.layers[l].host.bias = b

    def step(self, x_res: torch.Tensor, T: int, index: int,
             after_layer: Optional[Callable[[int], None]] = None,
             after_plan: Optional[Callable[[], None]] = None) -> None:
        """One decode step of all layers on the residual stream x_res (fp32 [T, H], updated in place)."""
        if self.drift_every and index % self.drift_every == 0 and index // self.drift_every != self.epoch:
            self.set_epoch(index // self.drift_every)
        st, ws = self.st, self.st.ws
        prev = None
        for l in range(self.L):
            moe.moe_residual_rmsnorm(x_res, prev, self.xn, T, self.H, self.eps)
            st.forward(l, self.xn, self.ys[l], T, y_is_fp32=False)
            moe.cache_heat_update(st.cache, ws.view.topk_ids, T, self.k, l)
            if after_layer is not None:
                after_layer(l)
            prev = self.ys[l]
        moe.moe_residual_rmsnorm(x_res, prev, self.xn, T, self.H, self.eps)
        if self.plan_every and (index + 1) % self.plan_every == 0:
            moe.cache_plan_swaps(st.cache, self.threshold, self.max_swaps, self.decay, self.plan, self.n_plan)
            if after_plan is not None:
                after_plan()
            moe.moe_cache_apply_swaps(st.cache, self.plan, self.n_plan, torch.cuda.current_stream(),
                                      self.copy_stream)
