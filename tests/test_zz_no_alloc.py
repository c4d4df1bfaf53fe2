"""cache_plan_swaps_noalloc (planner on caller-owned tables, static scratch, no allocation)
against cache_plan_swaps on the same tables: identical plans, counts and decayed heats,
on two calls in a row.  Collected last, so it also runs after every other test in one process."""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import policy as opol
from serving_router_top_gb300 import moe

F32 = np.float32


def _make_cache(L, E, resident, H=64, I=32, seed=0):
    nb = moe.moe_blob_bytes(H, I)
    g = np.random.default_rng(seed)
    backing = torch.from_numpy(g.integers(0, 256, size=L * E * nb, dtype=np.uint8)).cuda()
    c = moe.Cache(L, E, H, I, int(resident.sum()), 0, backing, True)
    c.fill(resident.astype(np.uint8))
    return c, backing


def _plan_of(plan, n):
    cnt = int(n.item())
    return cnt, plan.cpu().numpy().view(moe.SWAP_DTYPE)[:cnt].copy()


@pytest.fixture(scope="module")
def lib():
    """The library built from this checkout (a fresh process has not built it yet)."""
    from serving_router_top_gb300 import build
    build.build()
    return moe.load()


def _heats(g, L, E, nonfinite=False):
    heat = (g.integers(0, 12, size=L * E) * F32(0.5)).astype(F32)
    heat[g.random(L * E) < 0.1] *= F32(0.7)
    if nonfinite:  # NaN and +inf heats, and inf on both sides of a pair (inf - inf = NaN)
        idx = g.choice(L * E, size=max(4, L * E // 50), replace=False)
        heat[idx[0::3]] = np.nan
        heat[idx[1::3]] = np.inf
        heat[idx[2::3]] = -np.inf
    return heat


def _check_pair_of_calls(L, E, seed, nonfinite=False):
    g = np.random.default_rng(seed)
    resident = g.random((L, E)) < 0.3
    c, _backing = _make_cache(L, E, resident)
    resid_t, _, heat_t = c.tables()
    heat = _heats(g, L, E, nonfinite)
    heat_t.copy_(torch.from_numpy(heat))
    # the caller's own copies of the tables
    my_heat = torch.from_numpy(heat.copy()).cuda()
    my_resid = resid_t.clone()
    cap = 96
    for call in range(2):
        prev = heat.copy()
        plan_a = torch.zeros(cap * 5, dtype=torch.int32, device="cuda")
        n_a = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        plan_b = torch.zeros(cap * 5, dtype=torch.int32, device="cuda")
        n_b = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        moe.cache_plan_swaps(c, 1.5, cap, 0.7, plan_a, n_a)
        moe.cache_plan_swaps_noalloc(my_heat, my_resid, L, E, 1.5, cap, 0.7, plan_b, n_b)
        torch.cuda.synchronize()
        na, pa = _plan_of(plan_a, n_a)
        nb, pb = _plan_of(plan_b, n_b)
        assert na == nb, (call, na, nb)
        if call == 0:
            assert na > 0  # the tables above give candidates on the first call
        assert np.array_equal(pa, pb), call
        # every entry names a real pair of this call's tables
        assert ((pb["layer"] >= 0) & (pb["layer"] < L)).all(), call
        assert ((pb["hot_expert"] >= 0) & (pb["hot_expert"] < E)).all(), call
        assert ((pb["cold_expert"] >= 0) & (pb["cold_expert"] < E)).all(), call
        assert (pb["slot"] >= 0).all(), call
        np.testing.assert_array_equal(heat_t.cpu().numpy(), my_heat.cpu().numpy())
        # every heat decayed exactly once more than before the call
        heat = (heat * F32(0.7)).astype(F32)
        np.testing.assert_array_equal(my_heat.cpu().numpy(), heat)
        if not nonfinite:  # and, on finite heats, the oracle's plan of the heats before the call
            ref = opol.plan_swaps(prev, my_resid.cpu().numpy(), L, E, max_swaps=cap)
            assert [(r.layer, r.hot_expert, r.cold_expert, r.slot) for r in ref] == \
                [tuple(int(v) for v in (e["layer"], e["hot_expert"], e["cold_expert"], e["slot"])) for e in pb], call
    return c


@pytest.mark.gpu
def test_noalloc_matches_cache_plan_swaps_large_then_small(lib):
    """Two calls in a row at 48 x 512, then two at 3 x 37: the smaller calls run on a scratch
    that still holds the larger calls' keys and partners, and must not read them."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _check_pair_of_calls(48, 512, 6)
    _check_pair_of_calls(3, 37, 5)


@pytest.mark.gpu
def test_noalloc_matches_cache_plan_swaps_small_then_large(lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _check_pair_of_calls(3, 37, 7)
    _check_pair_of_calls(48, 512, 8)


@pytest.mark.gpu
def test_noalloc_nonfinite_heats_after_a_larger_call(lib):
    """NaN and infinite heats end a layer's pairing at the first pair whose difference fails
    the threshold test; the plan then holds only pairs this call wrote, even though a larger
    call left other keys in the shared scratch."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    _check_pair_of_calls(48, 512, 9)
    _check_pair_of_calls(6, 200, 10, nonfinite=True)


def test_noalloc_rejects_sizes_beyond_the_static_scratch(lib):
    """Checked before anything reaches the device: the Python wrapper raises, the C entry returns EINVAL."""
    for L, E in [(1025, 4), (64, 1025), (40, 1000), (1024, 33)]:
        with pytest.raises(ValueError, match="static scratch"):
            moe.cache_plan_swaps_noalloc(16, 16, L, E, 1.5, 96, 0.7, 16, 16)
    cfg = moe.moe_policy_cfg(1.5, 96, 0.7)
    fake = C.c_void_p(256)  # never dereferenced: the size check comes first
    for L, E in [(1025, 4), (64, 1025), (40, 1000), (1024, 33), (0, 8), (8, 0)]:
        assert lib.cache_plan_swaps_noalloc(fake, fake, L, E, C.byref(cfg), fake, fake, None) == moe.MOE_EINVAL
    assert lib.cache_plan_swaps_noalloc(fake, fake, 8, 8, None, fake, fake, None) == moe.MOE_EINVAL
