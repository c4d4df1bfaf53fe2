"""Cache-policy miss rates on a synthetic drifting Zipf routing trace (oracle only, CPU).

FreeToken reading notes, section 5.3: replaying the same decode routing through a
global LRU, a periodically updated placement and a static one, the LRU misses
least and the static placement most.  The synthetic trace stands in for the
real ones."""
import numpy as np

from oracle import policy_study
from serving_router_top_gb300 import inputs


def test_routing_trace_shapes_and_distinct_ids():
    seen = 0
    for step, layer, ids in inputs.routing_trace(0, 3, 40, 5, 4, 6, 3, 1.1):
        assert ids.shape == (4, 5) and ids.dtype == np.int32
        assert all(len(set(row)) == 5 for row in ids) and ids.min() >= 0 and ids.max() < 40
        seen += 1
    assert seen == 18
    a = [ids for _, _, ids in inputs.routing_trace(1, 2, 64, 4, 2, 4, 2, 1.1)]
    b = [ids for _, _, ids in inputs.routing_trace(1, 2, 64, 4, 2, 4, 2, 1.1)]
    assert all(np.array_equal(x, y) for x, y in zip(a, b))   # seeded


def test_lru_misses_least_static_most():
    kw = dict(L=4, E=64, k=6, T=4, nslots=60, steps=200, drift_every=50, s=1.1)
    lru = policy_study.simulate("lru", **kw)
    heat = policy_study.simulate("heat", plan_every=32, **kw)
    static = policy_study.simulate("static", **kw)
    assert lru < heat <= static, (lru, heat, static)


def test_full_cache_never_misses():
    """A slot for every expert: everything starts resident and no policy misses."""
    kw = dict(L=2, E=16, k=3, T=2, nslots=32, steps=30, drift_every=10, s=1.1)
    assert all(policy_study.simulate(p, **kw) == 0.0 for p in ("lru", "heat", "static"))
