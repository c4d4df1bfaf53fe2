"""Miss rates of cache policies on a synthetic routing trace (oracle; test infrastructure only).

The FreeToken reading notes (section 5.3) replay the same decode routing traces
through three placement policies and report the share of expert reads that
miss: a global LRU, a placement updated at prefill time, and a static split.
The real traces are not available; this module replays a synthetic drifting
Zipf trace (``inputs.routing_trace``) through the policies this repository
implements, from the same initial residency:

  * ``lru``    -- the global LRU of ``oracle.lru`` (a call's misses are admitted
                  into the K least recently used slots);
  * ``heat``   -- the Strata heat policy of ``oracle.policy`` (counts every step,
                  a planning round with decay every ``plan_every`` steps);
  * ``static`` -- the initial residency, never changed.

A lookup is one group (one distinct expert of one layer call); it misses when
the expert is not resident at the time of the call.

    python -m oracle.policy_study      # the table of the design notes
"""
from __future__ import annotations

import numpy as np

from serving_router_top_gb300 import inputs

from . import layer as olayer
from . import lru as olru
from . import policy as opol


def simulate(policy: str, L: int, E: int, k: int, T: int, nslots: int, steps: int, drift_every: int, s: float,
             seed: int = 0, K: int = 32, plan_every: int = 256) -> float:
    """Miss rate of `policy` over the trace; every policy starts from the same seeded residency."""
    g = np.random.default_rng(seed)
    resid = np.full(L * E, -1, dtype=np.int32)
    owner = np.full(nslots, -1, dtype=np.int32)
    for slot, f in enumerate(g.permutation(L * E)[:nslots]):
        resid[f] = slot
        owner[slot] = f
    heat = np.zeros(L * E, dtype=np.float32)
    state = olru.new_state(nslots)
    lookups = misses = 0
    for step, layer, ids in inputs.routing_trace(seed, L, E, k, T, steps, drift_every, s):
        grp = olayer.expert_groups(ids)
        slot, src = olayer.lookup(grp.experts, layer, E, resid)
        lookups += grp.num_groups
        misses += int((src != olayer.SRC_RESIDENT).sum())
        if policy == "lru":
            plan = olru.plan_call(state, owner, layer, grp.experts, src, slot, K, E)
            olru.apply(resid, owner, plan, E)
        elif policy == "heat":
            opol.heat_update(heat, ids, layer, E)
            if layer == L - 1 and (step + 1) % plan_every == 0:
                opol.apply_swaps(resid, opol.plan_round(heat, resid, L, E), E)
        elif policy != "static":
            raise ValueError(policy)
    return misses / max(1, lookups)


def study(L=8, E=512, k=10, T=4, steps=1024, drift_every=256, s=1.1, fracs=(0.37, 0.11), seed=0):
    rows = []
    for frac in fracs:
        nslots = int(round(frac * L * E))
        rows.append((frac, nslots, {p: simulate(p, L, E, k, T, nslots, steps, drift_every, s, seed)
                                    for p in ("lru", "heat", "static")}))
    return rows


if __name__ == "__main__":
    import time
    t0 = time.time()
    L, E, k, T, steps, drift, s = 8, 512, 10, 4, 1024, 256, 1.1
    print(f"trace: {L} layers x {E} experts, top-{k}, {T} tokens per call, {steps} steps, "
          f"Zipf s={s}, hot set re-drawn every {drift} steps")
    print("| cache (share of the pool) | slots | global LRU | heat policy | static |")
    print("|---|---:|---:|---:|---:|")
    for frac, nslots, r in study(L, E, k, T, steps, drift, s):
        print(f"| {frac:.0%} | {nslots} | {r['lru']:.1%} | {r['heat']:.1%} | {r['static']:.1%} |")
    print(f"({time.time() - t0:.0f} s)")
