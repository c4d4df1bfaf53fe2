"""Global LRU expert cache (oracle; test infrastructure only).

Source: FreeToken reading notes (zhongzhuzhou.org):
  * section 3.3: one LRU cache shared by every layer, over (layer, expert): a
    hit refreshes the expert's recency, a fill admits the newly chosen expert,
    and eviction removes the least recently used one;
  * section 4: victim selection does not rescan the cache per eviction -- one
    pass finds the K least recently used candidate slots and the miss path
    consumes the first q <= K of them, so finding victims costs the same
    whatever the number of misses.

Readings (listed in the design notes):
  * recency is kept per slot: ``tick[slot]`` is the number of the last layer
    call that used the slot (its hits, or the call that admitted an expert
    into it); calls are numbered 1, 2, ... by a clock; 0 means never used;
  * one call: the clock advances, the call's hits are refreshed, then its
    misses -- groups neither resident nor dropped by the tail skip, in group
    order (ascending expert id) -- are admitted into the victims, which are the
    K slots the call did not use, empty slots first (in slot order), then by
    (tick, slot) ascending; q = min(misses, victims) admissions, the i-th miss
    taking the i-th victim;
  * an admitted expert takes the slot (tick = the call's clock); the expert it
    evicts, if any, loses its residency; a miss beyond the first K stays out
    until a later call admits it.
"""
from __future__ import annotations

import dataclasses
from typing import List, Sequence

import numpy as np

from .layer import SRC_MISSING, SRC_RESIDENT, SRC_STAGED


@dataclasses.dataclass(frozen=True)
class LruSwap:
    layer: int        # layer of the admitted expert
    hot_expert: int   # admitted expert
    cold_flat: int    # evicted expert as layer * E + expert, or -1 for an empty slot
    slot: int


@dataclasses.dataclass
class LruState:
    tick: np.ndarray  # int64 [nslots]
    clock: int = 0


def new_state(nslots: int) -> LruState:
    return LruState(np.zeros(nslots, dtype=np.int64), 0)


def victims(state: LruState, slot_owner: np.ndarray, K: int) -> List[int]:
    """The K slots not used by the current call: empty ones by slot, then the others by (tick, slot)."""
    cand = [s for s in range(state.tick.size) if state.tick[s] < state.clock]
    cand.sort(key=lambda s: (0, 0, s) if slot_owner[s] < 0 else (1, int(state.tick[s]), s))
    return cand[:K]


def plan_call(state: LruState, slot_owner: np.ndarray, layer: int, experts: Sequence[int], src: Sequence[int],
              slot: Sequence[int], K: int, E: int) -> List[LruSwap]:
    """One layer call: refresh its hits, then pair its misses with the victims.

    ``experts``, ``src``, ``slot`` are the call's groups in group order (as the
    grouping writes them).  Updates ``state`` (clock, ticks of the hits and of
    the slots taken); the residency tables change in ``apply``.
    """
    state.clock += 1
    for s, sl in zip(src, slot):
        if s == SRC_RESIDENT:
            state.tick[sl] = state.clock
    misses = [int(e) for e, s in zip(experts, src) if s in (SRC_STAGED, SRC_MISSING)]
    v = victims(state, slot_owner, K)
    plan = []
    for i in range(min(len(misses), len(v))):
        owner = int(slot_owner[v[i]])
        plan.append(LruSwap(layer, misses[i], owner, v[i]))
        state.tick[v[i]] = state.clock
    return plan


def apply(resid: np.ndarray, slot_owner: np.ndarray, plan: List[LruSwap], E: int) -> None:
    """Evict, then admit: the residency table and the slot owners after the copies land."""
    for p in plan:
        if p.cold_flat >= 0:
            assert resid[p.cold_flat] == p.slot
            resid[p.cold_flat] = -1
        slot_owner[p.slot] = -1
    for p in plan:
        f = p.layer * E + p.hot_expert
        resid[f] = p.slot
        slot_owner[p.slot] = f
