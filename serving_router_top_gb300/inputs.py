"""Seeded synthetic workloads for the slot-addressed MoE layer.

This module is the one place that both the CUDA path and the CPU oracle take
their inputs from.  It draws random numbers and lays them out in the canonical
byte formats; it holds none of the layer's arithmetic (no decoding, no
routing, no FFN, no policy).  Everything is a pure function of
``(seed, tensor tag, layer, expert)``, so any sub-part of a large workload can
be regenerated on its own (the oracle checks sampled experts of a 29 GB model
without materialising the rest).

Canonical weight format (the NVFP4 row layout described on the PLE offload
page, "packed 文件" / "一个 160 维向量在 packed 文件中占 90 字节"): a matrix of
``rows x cols`` values is stored as ``rows`` byte rows; each row holds
``cols/2`` code bytes (two 4-bit E2M1 codes per byte, the low nibble being the
even column) followed by ``cols/16`` FP8-E4M3 block-scale bytes, one per 16
consecutive columns.  One FP32 global scale per matrix rides beside it.
Row width is therefore ``9*cols/16`` bytes.

Input recipe (stated once here; the design notes repeat it):
  * codes: uniform bytes (two independent uniform 4-bit codes);
  * block scales: E4M3 bytes ``(e<<3)|m`` with ``e`` uniform in 3..6 and ``m``
    uniform in 0..7, i.e. values ``2^(e-7)*(1+m/8)`` spread over
    ``[2^-4, 2^0)`` one octave at a time (log-uniform at octave grain);
  * global scales: 1.0 (the edge-case workload: 0.375, 2.0, 1.25 for gate, up, down,
    and block scales over the whole non-negative E4M3 range, see ``packed_matrix``);
  * activations x: N(0,1) rounded to bf16 (round-to-nearest-even);
  * router weights W_r: N(0, std) in bf16, std 0.02 (or 1/sqrt(H) where a
    workload asks for unit-variance logits);
  * shared-expert gate vector w_sg: N(0, 0.02) in bf16;
  * per-expert Zipf bias: ``-s * ln(rank)``, ``rank`` a seeded permutation of
    ``1..E`` per layer (and per drift epoch);
  * residency: a seeded uniform subset of the experts of each layer.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Tuple

import numpy as np

# Tensor tags keep the sub-streams of one seed apart.
TAG_X, TAG_WR, TAG_BIAS, TAG_WSG, TAG_GATE, TAG_UP, TAG_DOWN, TAG_RESID, TAG_SHARED, TAG_TRACE = range(1, 11)
SHARED_EXPERT_ID = 1 << 20  # expert id used for the shared expert's sub-stream


def rng(seed: int, *ids: int) -> np.random.Generator:
    """Independent PCG64 stream for ``(seed, *ids)`` (numpy SeedSequence mixing)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed)] + [int(i) & 0xFFFFFFFF for i in ids])))


def round_f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even.  Input recipe step only."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def normal_bf16(g: np.random.Generator, shape, std: float) -> np.ndarray:
    return round_f32_to_bf16_bits((g.standard_normal(shape) * std).astype(np.float32))


def packed_row_bytes(cols: int) -> int:
    return cols // 2 + cols // 16


def random_bytes(g: np.random.Generator, n: int) -> np.ndarray:
    """n uniform bytes: the little-endian bytes of raw 64-bit PCG64 outputs."""
    words = g.bit_generator.random_raw((n + 7) // 8).astype("<u8", copy=False)
    return words.view(np.uint8)[:n]


# Scale-byte recipes.  "octaves": exponent field 3..6, any mantissa (the default).
# "edge": the whole non-negative E4M3 range with its ends over-represented -- zero
# (0x00), subnormals (0x01..0x07), the largest normal 448 (0x7E) and the rest of
# the normal range (0x08..0x7D) -- to reach the ends of the format's value range.
SCALE_RECIPES = ("octaves", "edge")


def packed_matrix(g: np.random.Generator, rows: int, cols: int, scales: str = "octaves") -> np.ndarray:
    """One matrix in the canonical packed-row format, uint8 ``[rows, 9*cols/16]``.

    Codes are raw random bytes.  "octaves" scales: each scale byte takes 5 random
    bits, two picking the exponent field e in 3..6 and three the mantissa field m in
    0..7.  "edge" scales: a random byte picks 0x00 (1 in 16), a subnormal 0x01..0x07
    (2 in 16), 0x7E (1 in 16), else a uniform byte of 0x08..0x7D; the sign bit stays 0.
    """
    assert cols % 16 == 0, cols
    assert scales in SCALE_RECIPES, scales
    codes = random_bytes(g, rows * cols // 2).reshape(rows, cols // 2)
    r = random_bytes(g, rows * cols // 16).reshape(rows, cols // 16)
    if scales == "octaves":
        sc = (((r & 3) + 3) << 3) | ((r >> 2) & 7)
    else:
        kind = r & 15
        rest = random_bytes(g, rows * cols // 16).reshape(rows, cols // 16)
        sc = np.where(kind == 0, 0,
             np.where(kind <= 2, 1 + rest % 7,
             np.where(kind == 3, 0x7E, 0x08 + rest % (0x7E - 0x08)))).astype(np.uint8)
    return np.concatenate([codes, sc.astype(np.uint8)], axis=1)


@dataclasses.dataclass(frozen=True)
class LayerShape:
    H: int          # hidden size
    I: int          # routed-expert intermediate size
    E: int          # routed experts per layer
    k: int          # experts per token
    I_shared: int   # shared-expert intermediate size (0 = no shared expert)


@dataclasses.dataclass
class Expert:
    """One expert's three matrices in canonical packed rows."""
    gate: np.ndarray   # [I, 9H/16]
    up: np.ndarray     # [I, 9H/16]
    down: np.ndarray   # [H, 9I/16]
    gscale: Tuple[float, float, float] = (1.0, 1.0, 1.0)


def expert_weights(seed: int, layer: int, expert: int, H: int, I: int, scales: str = "octaves",
                   gscale: Tuple[float, float, float] = (1.0, 1.0, 1.0)) -> Expert:
    return Expert(
        gate=packed_matrix(rng(seed, TAG_GATE, layer, expert), I, H, scales),
        up=packed_matrix(rng(seed, TAG_UP, layer, expert), I, H, scales),
        down=packed_matrix(rng(seed, TAG_DOWN, layer, expert), H, I, scales),
        gscale=tuple(float(np.float32(v)) for v in gscale),
    )


def shared_expert_weights(seed: int, layer: int, H: int, I_shared: int, scales: str = "octaves",
                          gscale: Tuple[float, float, float] = (1.0, 1.0, 1.0)) -> Expert:
    return expert_weights(seed, layer, SHARED_EXPERT_ID, H, I_shared, scales, gscale)


def activations(seed: int, step: int, T: int, H: int) -> np.ndarray:
    """bf16 bits ``[T, H]``, N(0,1)."""
    return normal_bf16(rng(seed, TAG_X, step), (T, H), 1.0)


def router_weights(seed: int, layer: int, E: int, H: int, std: float) -> np.ndarray:
    return normal_bf16(rng(seed, TAG_WR, layer), (E, H), std)


def shared_gate_weights(seed: int, layer: int, H: int) -> np.ndarray:
    return normal_bf16(rng(seed, TAG_WSG, layer), (H,), 0.02)


def zipf_bias(seed: int, layer: int, E: int, s: float, epoch: int = 0) -> np.ndarray:
    """float32 ``[E]``: ``-s*ln(rank[e])`` with a seeded rank permutation; zeros when s == 0."""
    if s == 0.0:
        return np.zeros(E, dtype=np.float32)
    rank = rng(seed, TAG_BIAS, layer, epoch).permutation(E) + 1
    return (-s * np.log(rank.astype(np.float64))).astype(np.float32)


def resident_mask(seed: int, layer: int, E: int, frac: float) -> np.ndarray:
    """bool ``[E]``: a uniform subset of ``round(frac*E)`` experts."""
    n = int(round(frac * E))
    mask = np.zeros(E, dtype=bool)
    mask[rng(seed, TAG_RESID, layer).permutation(E)[:n]] = True
    return mask


def routing_trace(seed: int, L: int, E: int, k: int, T: int, steps: int, drift_every: int, s: float):
    """Synthetic decode routing: for each step and layer (in that order), int32 ``[T, k]``
    distinct expert ids per token, drawn without replacement with probability proportional
    to ``rank^-s`` (Gumbel keys on ``zipf_bias``); the ranks are re-drawn every
    ``drift_every`` steps, so the hot set drifts.  Yields ``(step, layer, ids)``."""
    for step in range(steps):
        epoch = step // drift_every
        for layer in range(L):
            bias = zipf_bias(seed, layer, E, s, epoch).astype(np.float64)
            g = rng(seed, TAG_TRACE, step, layer).gumbel(size=(T, E))
            yield step, layer, np.argsort(-(bias[None, :] + g), axis=1)[:, :k].astype(np.int32)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: LayerShape
    T: int                    # tokens per layer call
    layers: int = 1
    zipf_s: float = 0.0
    router_std: float = 0.02
    resident_frac: float = 1.0
    seed: int = 0
    description: str = ""
    scales: str = "octaves"                                  # block-scale recipe (SCALE_RECIPES)
    gscale: Tuple[float, float, float] = (1.0, 1.0, 1.0)     # FP32 global scales of gate, up, down


# The five workload shapes of the method's evaluation, plus small variants
# sized for exhaustive oracle comparison.
WORKLOADS: Dict[str, Workload] = {
    "layer_t8_h256_e16_k2": Workload(
        "layer_t8_h256_e16_k2", LayerShape(H=256, I=128, E=16, k=2, I_shared=0), T=8,
        description="single MoE layer, 8 tokens, hidden 256, 16 experts top-2, I=128, no shared expert, all resident"),
    "decode_t4_h2048_e512_k10": Workload(
        "decode_t4_h2048_e512_k10", LayerShape(H=2048, I=512, E=512, k=10, I_shared=512), T=4,
        zipf_s=1.1, resident_frac=0.5,
        description="decode verify window: 4 tokens, hidden 2048, 512 experts top-10, I=512, shared expert I=512, "
                    "Zipf(1.1) router bias, 50% of experts resident, the rest in device staging slots"),
    "stack48_decode_h2048_e512_k10": Workload(
        "stack48_decode_h2048_e512_k10", LayerShape(H=2048, I=512, E=512, k=10, I_shared=512), T=16, layers=48,
        zipf_s=1.1, resident_frac=0.3,
        description="48-layer decode stack (RMSNorm + residual), batch 1..16, Zipf-hot routing drifting every 512 steps, "
                    "cache of 30% of 48x512 slots, heat every step, planning every 256 steps"),
    "prefill_t8192_h2048_e512_k10": Workload(
        "prefill_t8192_h2048_e512_k10", LayerShape(H=2048, I=512, E=512, k=10, I_shared=512), T=8192,
        description="prefill chunk: 8192 tokens, hidden 2048, 512 experts top-10, I=512, shared expert, "
                    "weights streamed through two staging slots"),
    "large_h4096_e256_k6": Workload(
        "large_h4096_e256_k6", LayerShape(H=4096, I=2048, E=256, k=6, I_shared=2048), T=4096, layers=8,
        zipf_s=1.0, router_std=1.0 / math.sqrt(4096),
        description="8 layers, hidden 4096, 256 experts top-6, I=2048, shared expert I=2048, all resident (~29 GB); "
                    "4096-token prefill then batch-64 decode"),
}


def small_workload(T=5, H=128, I=64, E=12, k=3, I_shared=64, zipf_s=0.5, resident_frac=1.0, seed=1, layers=1,
                   scales="octaves", gscale=(1.0, 1.0, 1.0)) -> Workload:
    """Ragged small shapes for exhaustive oracle checks."""
    return Workload(f"small_t{T}_h{H}_e{E}_k{k}", LayerShape(H=H, I=I, E=E, k=k, I_shared=I_shared), T=T,
                    layers=layers, zipf_s=zipf_s, resident_frac=resident_frac, seed=seed, scales=scales,
                    gscale=tuple(gscale))


def edge_workload(T=6, H=256, I=128, E=24, k=4, I_shared=128, seed=11, resident_frac=0.5) -> Workload:
    """The format's edge cases on a small layer: block scales over the whole non-negative
    E4M3 range (zero, subnormals, 448) and distinct non-unit global scales per matrix."""
    return small_workload(T=T, H=H, I=I, E=E, k=k, I_shared=I_shared, zipf_s=0.7, resident_frac=resident_frac,
                          seed=seed, scales="edge", gscale=(0.375, 2.0, 1.25))


def expert_of(w: Workload, layer: int, e: int) -> Expert:
    """Routed expert e of a layer of workload w, with the workload's scale recipe."""
    return expert_weights(w.seed, layer, e, w.shape.H, w.shape.I, w.scales, w.gscale)


@dataclasses.dataclass
class LayerInputs:
    """Everything one MoE layer call needs, in canonical formats (host numpy)."""
    x: np.ndarray                 # bf16 bits [T, H]
    w_router: np.ndarray          # bf16 bits [E, H]
    bias: np.ndarray              # float32 [E]
    w_shared_gate: Optional[np.ndarray]  # bf16 bits [H] or None
    shared: Optional[Expert]
    layer: int


def layer_inputs(w: Workload, layer: int = 0, step: int = 0, epoch: int = 0, T: Optional[int] = None) -> LayerInputs:
    s = w.shape
    T = w.T if T is None else T
    has_shared = s.I_shared > 0
    return LayerInputs(
        x=activations(w.seed, step, T, s.H),
        w_router=router_weights(w.seed, layer, s.E, s.H, w.router_std),
        bias=zipf_bias(w.seed, layer, s.E, w.zipf_s, epoch),
        w_shared_gate=shared_gate_weights(w.seed, layer, s.H) if has_shared else None,
        shared=shared_expert_weights(w.seed, layer, s.H, s.I_shared, w.scales, w.gscale) if has_shared else None,
        layer=layer,
    )


def experts_of_layer(w: Workload, layer: int):
    """Generator over ``(expert id, Expert)`` of one layer."""
    for e in range(w.shape.E):
        yield e, expert_of(w, layer, e)
