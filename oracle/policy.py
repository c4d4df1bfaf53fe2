"""Adaptive expert-cache policy (oracle; test infrastructure only).

Source: Strata expert paths (hanayo.cn), section "哪些专家能长期留在显存？":
  * the policy accumulates how often each expert is routed to and decays the
    history periodically;
  * within one layer it pairs hot experts outside the cache with cold experts
    inside it, and schedules a swap only when the heat difference reaches the
    threshold;
  * all candidates are sorted by heat difference and capped per round;
  * worked example: A (not resident) heat 10, B (resident) heat 8,
    difference 2 >= 1.5, so the pair is a candidate; defaults are threshold
    1.5, at most 96 swaps per round, decay 0.7 applied to the old heats after
    an adjustment round;
  * new weights become visible only after their copy completes; an old slot is
    reused only after earlier readers are done.

The counters are fp32 and the policy is defined on them, so this module
computes the exact fp32 operation sequence (numpy float32: one rounding per
operation, no fused multiply-add):
  heat update : heat = fl32(heat + fl32(count))        once per step and layer
  difference  : d = fl32(heat[hot] - heat[cold]);  swap iff d >= 1.5f
  decay       : heat = fl32(heat * 0.7f)               all entries, once per round

Readings (listed in the design notes): the count is +1 per (token, rank)
selection; pairing ranks the layer's non-resident experts by heat descending
(id ascending) and its resident experts by heat ascending (id ascending) and
pairs them i-th with i-th while the difference reaches the threshold; the
merged candidates are ordered by (difference desc, layer asc, hot id asc) and
the first ``max_swaps`` kept; decay runs once per planning round, after
planning, even when no swap was planned.
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np

F32 = np.float32
THRESHOLD = F32(1.5)
MAX_SWAPS = 96
DECAY = F32(0.7)


@dataclasses.dataclass(frozen=True)
class Swap:
    layer: int
    hot_expert: int    # not resident, to be brought in
    cold_expert: int   # resident, to be evicted
    slot: int          # the cold expert's slot, reused by the hot one
    diff: float        # fl32(heat[hot] - heat[cold])


def heat_update(heat: np.ndarray, ids: np.ndarray, layer: int, E: int) -> None:
    """Add this step's per-expert selection counts of one layer, in place."""
    assert heat.dtype == F32
    cnt = np.bincount(np.asarray(ids, dtype=np.int64).ravel(), minlength=E)[:E]
    row = heat[layer * E:(layer + 1) * E]
    row[:] = row + cnt.astype(F32)


def plan_swaps(heat: np.ndarray, resid: np.ndarray, L: int, E: int,
               threshold: float = THRESHOLD, max_swaps: int = MAX_SWAPS) -> List[Swap]:
    """Hot-out/cold-in pairing per layer, merged, sorted and capped.  Does not decay."""
    assert heat.dtype == F32
    thr = F32(threshold)
    cands = []
    for l in range(L):
        h = heat[l * E:(l + 1) * E]
        r = np.asarray(resid[l * E:(l + 1) * E])
        hot = sorted(np.flatnonzero(r < 0), key=lambda e: (-float(h[e]), int(e)))
        cold = sorted(np.flatnonzero(r >= 0), key=lambda e: (float(h[e]), int(e)))
        for a, b in zip(hot, cold):
            d = F32(h[a] - h[b])
            if not d >= thr:
                break
            cands.append(Swap(l, int(a), int(b), int(r[b]), float(d)))
    cands.sort(key=lambda s: (-s.diff, s.layer, s.hot_expert))
    return cands[:max_swaps]


def decay(heat: np.ndarray, factor: float = DECAY) -> None:
    """heat = fl32(heat * factor) for every entry, in place."""
    assert heat.dtype == F32
    heat[:] = heat * F32(factor)


def plan_round(heat: np.ndarray, resid: np.ndarray, L: int, E: int, threshold: float = THRESHOLD,
               max_swaps: int = MAX_SWAPS, factor: float = DECAY) -> List[Swap]:
    """One adjustment round: plan, then decay all heats."""
    plan = plan_swaps(heat, resid, L, E, threshold, max_swaps)
    decay(heat, factor)
    return plan


def apply_swaps(resid: np.ndarray, plan: List[Swap], E: int) -> None:
    """Residency after a round's copies have landed: cold unmapped, hot published in its slot."""
    for s in plan:
        assert resid[s.layer * E + s.cold_expert] == s.slot
        resid[s.layer * E + s.cold_expert] = -1
        resid[s.layer * E + s.hot_expert] = s.slot
