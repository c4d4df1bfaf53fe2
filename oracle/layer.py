"""The MoE layer forward over a slot-addressed expert cache (oracle; test infrastructure only).

Sources (page titles as headed in the source material):
  * Strata expert paths (hanayo.cn, "显存里缓存的是什么？"): an expert's identity
    is (layer, expert); the router picks each token's experts and their merge
    weights; 48 layers x 512 experts, top-10.
  * Same page, "路由以后，专家怎样分工？": a resident expert is found through the
    slot table and computed on the GPU; every path produces the expert output
    vector; outputs of a token are multiplied by their routing weights and
    summed, then the gated shared-expert contribution (same input) is added;
    repeated experts of one layer and window form one group that records its
    input and output positions.
  * Same page, "CPU 怎样把剩下的专家算完？": an expert computes gate/up, the
    activation, then the down projection.
  * Same page, "哪些专家能长期留在显存？": the residency table maps
    (layer, expert) to a slot or returns a special value when not resident.
  * FreeToken reading notes (zhongzhuzhou.org), section 3.2: CPU and GPU
    partial results merge exactly -- the layer output is the plain weighted sum.
  * Strata page, "还有一条会改变输出的路径：跳过尾部专家" (optional tail skip):
    with a threshold of 7 on zero-based ranks, an expert that is not resident
    and that every token of the window choosing it ranks 7th or later adds
    nothing; one token ranking it higher, or residency, keeps it; the other
    weights are not renormalised, so the output moves by minus the skipped
    experts' weighted outputs.

Readings where the pages are silent (each listed in the design notes):
  * top-k: softmax over all E then renormalise over the k chosen equals a
    softmax over the chosen logits; selection is on the fp32 logits with ties
    to the lower expert id; the output order is weight descending.
  * groups: one group per distinct expert, ascending expert id; entries by
    ascending token; an entry's output position is ``t*k + r`` (r = rank).
  * residency sentinel: -1.  A non-resident expert may sit in a staging slot
    (second table); neither -> MISSING.
  * shared-expert gate: ``sigmoid(x . w_sg)``; activation SiLU(z) = z/(1+e^-z).
  * tail skip: an entry's rank is its position r in the token's list (weight
    descending); "not resident" means staged or missing, and a skipped
    expert that is also missing is not an error.  Off unless asked for.
"""
from __future__ import annotations

import dataclasses
from typing import Callable, Dict, List, Optional, Tuple

import numpy as np

from .formats import bf16_value, dequantize

MISSING = -1
SRC_RESIDENT, SRC_STAGED, SRC_MISSING, SRC_SKIPPED = 0, 1, -1, 2


class OracleError(RuntimeError):
    pass


def router_logits(x_bits: np.ndarray, w_router_bits: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    """``l[t,e] = sum_h x[t,h] * W_r[e,h] + bias[e]`` in fp64, rounded once to fp32."""
    x = bf16_value(x_bits)
    w = bf16_value(w_router_bits)
    l = x @ w.T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    return l.astype(np.float32)


def top_k(logits: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray]:
    """Top-k per token with renormalised softmax weights.

    Returns ``ids`` int32 ``[T,k]`` (weight descending, ties to the lower id)
    and ``w`` fp64 ``[T,k]`` with ``w_r = exp(l_r - l_0) / sum_j exp(l_j - l_0)``
    over the chosen k (equal to softmax over all E renormalised over the k).
    """
    l = np.asarray(logits, dtype=np.float32)
    if np.isnan(l).any():
        raise OracleError("NaN logit")
    T, E = l.shape
    if not 1 <= k <= E:
        raise OracleError("k out of range")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    expert = np.arange(E)
    for t in range(T):
        order = np.lexsort((expert, -l[t].astype(np.float64)))[:k]  # by (-l, e)
        ids[t] = order
        sel = l[t, order].astype(np.float64)
        p = np.exp(sel - sel[0])
        w[t] = p / p.sum()
    return ids, w


@dataclasses.dataclass
class Groups:
    experts: np.ndarray   # int32 [G], ascending
    off: np.ndarray       # int32 [G+1]
    ent_tok: np.ndarray   # int32 [T*k]
    ent_pos: np.ndarray   # int32 [T*k], t*k + r

    @property
    def num_groups(self) -> int:
        return int(self.experts.size)


def expert_groups(ids: np.ndarray) -> Groups:
    """Dedupe the (token, rank) selections of one layer and window into expert groups."""
    ids = np.asarray(ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.ravel()
    pos = np.arange(T * k)
    order = np.lexsort((pos, flat))            # expert ascending, then position (= token) ascending
    experts, counts = np.unique(flat, return_counts=True)
    off = np.concatenate([[0], np.cumsum(counts)])
    return Groups(experts.astype(np.int32), off.astype(np.int32),
                  (order // k).astype(np.int32), order.astype(np.int32))


def lookup(experts: np.ndarray, layer: int, E: int, resid: np.ndarray,
           stage: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """(layer, expert) -> (slot, source): resident slot, else staging slot, else MISSING."""
    flat = layer * E + np.asarray(experts, dtype=np.int64)
    slot = np.asarray(resid, dtype=np.int32)[flat].copy()
    src = np.where(slot >= 0, SRC_RESIDENT, SRC_MISSING).astype(np.int32)
    if stage is not None:
        st = np.asarray(stage, dtype=np.int32)[flat]
        use = (slot < 0) & (st >= 0)
        slot[use] = st[use]
        src[use] = SRC_STAGED
    slot[src == SRC_MISSING] = MISSING
    return slot, src


def tail_skip_mask(groups: Groups, src: np.ndarray, k: int, min_rank: int) -> np.ndarray:
    """Groups dropped by the tail skip (Strata page, "跳过尾部专家").

    Group g is dropped when its expert is not resident and every entry has a
    zero-based rank ``pos % k`` of at least ``min_rank``.  ``min_rank <= 0``
    drops nothing.
    """
    G = groups.num_groups
    drop = np.zeros(G, dtype=bool)
    if min_rank <= 0:
        return drop
    for g in range(G):
        ranks = groups.ent_pos[groups.off[g]:groups.off[g + 1]] % k
        drop[g] = src[g] != SRC_RESIDENT and int(ranks.min()) >= min_rank
    return drop


def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def sigmoid(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


@dataclasses.dataclass
class DenseExpert:
    """An expert's matrices dequantised to fp64."""
    gate: np.ndarray  # [I, H]
    up: np.ndarray    # [I, H]
    down: np.ndarray  # [H, I]


def dequantize_expert(ex, H: int, I: int) -> DenseExpert:
    g, u, d = ex.gscale
    return DenseExpert(dequantize(ex.gate, H, g), dequantize(ex.up, H, u), dequantize(ex.down, I, d))


def swiglu_expert(x: np.ndarray, de: DenseExpert) -> np.ndarray:
    """gate/up, SiLU(gate)*up, down projection, all fp64.  ``x`` is ``[n, H]``."""
    g = x @ de.gate.T
    u = x @ de.up.T
    return (silu(g) * u) @ de.down.T


@dataclasses.dataclass
class LayerResult:
    y: np.ndarray            # fp64 [T, H]
    logits: np.ndarray       # fp32 [T, E]
    ids: np.ndarray          # int32 [T, k]
    w: np.ndarray            # fp64 [T, k]
    groups: Groups
    slot: np.ndarray         # int32 [G]
    src: np.ndarray          # int32 [G]
    o: np.ndarray            # fp64 [T*k, H] routed expert outputs by position
    shared: Optional[np.ndarray]   # fp64 [T, H] shared expert output
    gamma: Optional[np.ndarray]    # fp64 [T] shared gate


def moe_layer(x_bits: np.ndarray, w_router_bits: Optional[np.ndarray], bias: Optional[np.ndarray], k: int,
              get_expert: Callable[[int], object], H: int, I: int, layer: int = 0,
              resid: Optional[np.ndarray] = None, stage: Optional[np.ndarray] = None,
              shared=None, I_shared: int = 0, w_shared_gate_bits: Optional[np.ndarray] = None,
              logits: Optional[np.ndarray] = None, x_values: Optional[np.ndarray] = None,
              tail_skip: int = 0) -> LayerResult:
    """One MoE layer forward, in the order the Strata page walks it.

    ``get_expert(e)`` returns the canonical-format weights of routed expert e
    of this layer.  ``logits`` (fp32) replaces the router when given.
    ``x_values`` (fp64 ``[T,H]``) overrides the decoded bf16 input, for callers
    that feed an already-normalised activation.  ``tail_skip > 0`` drops the
    groups ``tail_skip_mask`` names: their source becomes SRC_SKIPPED, their
    slot MISSING, and their entries' outputs stay zero.
    """
    x = bf16_value(x_bits) if x_values is None else np.asarray(x_values, dtype=np.float64)
    T = x.shape[0]
    if logits is None:
        logits = router_logits(x_bits, w_router_bits, bias)
    E = logits.shape[1]
    ids, w = top_k(logits, k)
    groups = expert_groups(ids)
    if resid is None:
        resid = np.arange((layer + 1) * E, dtype=np.int32)  # all resident
    slot, src = lookup(groups.experts, layer, E, resid, stage)
    drop = tail_skip_mask(groups, src, k, tail_skip)
    src[drop] = SRC_SKIPPED
    slot[drop] = MISSING
    if (src == SRC_MISSING).any():
        raise OracleError("expert neither resident nor staged")
    o = np.zeros((T * k, H), dtype=np.float64)
    for gi, e in enumerate(groups.experts):
        if drop[gi]:
            continue
        a, b = groups.off[gi], groups.off[gi + 1]
        toks = groups.ent_tok[a:b]
        o[groups.ent_pos[a:b]] = swiglu_expert(x[toks], dequantize_expert(get_expert(int(e)), H, I))
    y = np.zeros((T, H), dtype=np.float64)
    for r in range(k):                               # routing-weighted combine, rank order
        y += w[:, r:r + 1] * o[np.arange(T) * k + r]
    s = gamma = None
    if shared is not None:
        s = swiglu_expert(x, dequantize_expert(shared, H, I_shared))
        gamma = sigmoid(x @ bf16_value(w_shared_gate_bits))
        y = gamma[:, None] * s + y
    return LayerResult(y, logits, ids, w, groups, slot, src, o, s, gamma)


def rmsnorm(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """RMSNorm with unit weight: ``x / sqrt(mean(x^2) + eps)`` per row."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
