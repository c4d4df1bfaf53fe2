"""Device-side set-up of a synthetic workload: backing store, expert cache,
per-layer router/shared-expert weights and a workspace.

This is set-up code around the C ABI (host logic: generate, pack, copy); the
layer itself runs only in libmoe's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional

import numpy as np
import torch

from . import inputs as I
from . import moe


def to_device(a: np.ndarray, device="cuda") -> torch.Tensor:
    """numpy array -> torch device tensor holding the same bytes (uint16 -> int16, uint8 stays uint8)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


def pack(ex: I.Expert, H: int, I_: int, out: Optional[np.ndarray] = None) -> np.ndarray:
    return moe.moe_pack_expert(ex.gate, ex.up, ex.down, H, I_, ex.gscale, out)


@dataclasses.dataclass
class LayerWeights:
    layer: int
    host: I.LayerInputs
    w_router: torch.Tensor
    bias: torch.Tensor
    w_shared_gate: Optional[torch.Tensor]
    shared_blob: Optional[torch.Tensor]
    desc: moe.moe_layer_desc


class ModelState:
    """All device state of one workload.

    ``resident``/``staged``: bool [L, E] masks (default: the workload's
    resident fraction as a seeded subset, everything else staged when
    ``stage_rest``; ``stage_all`` stages every expert, so that experts the
    cache policy swaps out stay reachable through the staging table).  ``backing_on_device``: keep the full expert pool in HBM
    (else page-locked host memory that kernels read directly).
    """

    def __init__(self, w: I.Workload, layers: Optional[int] = None, resident: Optional[np.ndarray] = None,
                 staged: Optional[np.ndarray] = None, stage_rest: bool = True, nslots: Optional[int] = None,
                 nstaging: Optional[int] = None, backing_on_device: bool = True, maxT: Optional[int] = None,
                 device: str = "cuda", stage_all: bool = False):
        self.w = w
        s = w.shape
        self.L = L = w.layers if layers is None else layers
        self.H, self.I, self.E, self.k, self.I_shared = s.H, s.I, s.E, s.k, s.I_shared
        self.blob_bytes = moe.moe_blob_bytes(s.H, s.I)
        if resident is None:
            resident = np.stack([I.resident_mask(w.seed, l, s.E, w.resident_frac) for l in range(L)])
        self.resident = np.asarray(resident, dtype=bool).reshape(L, s.E)
        if stage_all:  # every expert also in a staging slot: an expert swapped out stays reachable
            staged = np.ones_like(self.resident)
        elif staged is None:
            staged = ~self.resident if stage_rest else np.zeros_like(self.resident)
        self.staged = np.asarray(staged, dtype=bool).reshape(L, s.E)
        if not stage_all:
            self.staged &= ~self.resident
        self.backing = self._build_backing(backing_on_device, device)
        nslots = int(self.resident.sum()) if nslots is None else nslots
        nstaging = int(self.staged.sum()) if nstaging is None else nstaging
        self.cache = moe.Cache(L, s.E, s.H, s.I, nslots, nstaging, self.backing, backing_on_device)
        self.cache.fill(self.resident.astype(np.uint8))
        if self.staged.any():
            self.cache.fill(self.staged.astype(np.uint8), staging=True)
        self.layers: List[LayerWeights] = [self._layer(l, device) for l in range(L)]
        self.maxT = w.T if maxT is None else maxT
        self.ws = moe.Workspace(self.maxT, s.H, s.I, s.E, s.k, s.I_shared)

    def _build_backing(self, on_device: bool, device: str) -> torch.Tensor:
        s, L, nb = self.w.shape, self.L, self.blob_bytes
        total = L * s.E * nb
        if on_device:
            backing = torch.empty(total, dtype=torch.uint8, device=device)
        else:
            backing = torch.empty(total, dtype=torch.uint8, pin_memory=True)
        layer_buf = np.empty(s.E * nb, dtype=np.uint8)
        for l in range(L):
            for e, ex in I.experts_of_layer(self.w, l):
                pack(ex, s.H, s.I, layer_buf[e * nb:(e + 1) * nb])
            backing[l * s.E * nb:(l + 1) * s.E * nb].copy_(torch.from_numpy(layer_buf), non_blocking=False)
        if on_device:
            torch.cuda.synchronize()
        return backing

    def _layer(self, l: int, device: str) -> LayerWeights:
        s = self.w.shape
        li = I.layer_inputs(self.w, layer=l)
        w_router = to_device(li.w_router, device)
        bias = to_device(li.bias, device)
        wsg = to_device(li.w_shared_gate, device) if li.w_shared_gate is not None else None
        sblob = to_device(pack(li.shared, s.H, s.I_shared), device) if li.shared is not None else None
        desc = moe.layer_desc(w_router, bias, wsg, sblob, l, s.H, s.I, s.E, s.k, s.I_shared)
        return LayerWeights(l, li, w_router, bias, wsg, sblob, desc)

    def resid_table(self) -> np.ndarray:
        r, _, _ = self.cache.tables()
        return r.cpu().numpy()

    def stage_table(self) -> np.ndarray:
        _, st, _ = self.cache.tables()
        return st.cpu().numpy()

    def expert_host(self, layer: int, e: int) -> I.Expert:
        return I.expert_of(self.w, layer, e)

    def forward(self, layer: int, x: torch.Tensor, y: torch.Tensor, T: int, y_is_fp32: bool = True,
                mode: int = moe.MOE_MODE_AUTO, stream=None) -> None:
        moe.moe_layer_forward(self.layers[layer].desc, x, y, y_is_fp32, T, self.cache, self.ws, mode, stream)

    def forward_streamed(self, layer: int, x: torch.Tensor, y: torch.Tensor, T: int, U: int,
                         y_is_fp32: bool = True, stream=None, buffers: int = 2) -> None:
        """Prefill forward with the layer's experts streamed from the backing pool through the
        staging pool in units of U (needs at least buffers*U staging slots; buffers = 1 lets
        each copy wait for the previous unit's GEMMs)."""
        if getattr(self, "_copy_stream", None) is None:
            self._copy_stream = torch.cuda.Stream()
        moe.moe_layer_forward_streamed(self.layers[layer].desc, x, y, y_is_fp32, T, self.cache, self.ws, U,
                                       stream, self._copy_stream, buffers=buffers)
