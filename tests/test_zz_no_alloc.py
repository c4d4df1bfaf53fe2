"""cache_plan_swaps_noalloc (planner on caller-owned tables, static scratch, no allocation)
against cache_plan_swaps on the same tables: identical plans, counts and decayed heats,
on two calls in a row.  Collected last, so it also runs after every other test in one process."""
import ctypes as C

import numpy as np
import pytest
import torch

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


@pytest.mark.gpu
@pytest.mark.parametrize("L,E,seed", [(3, 37, 5), (48, 512, 6)])
def test_noalloc_matches_cache_plan_swaps_twice(L, E, seed):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_router_top_gb300 import build
    build.build()
    g = np.random.default_rng(seed)
    resident = g.random((L, E)) < 0.3
    c, _backing = _make_cache(L, E, resident)
    resid_t, _, heat_t = c.tables()
    heat = (g.integers(0, 12, size=L * E) * F32(0.5)).astype(F32)
    heat[g.random(L * E) < 0.1] *= F32(0.7)
    heat_t.copy_(torch.from_numpy(heat))
    # the caller's own copies of the tables
    my_heat = torch.from_numpy(heat.copy()).cuda()
    my_resid = resid_t.clone()
    cap = 96
    for call in range(2):
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
        assert np.array_equal(heat_t.cpu().numpy(), my_heat.cpu().numpy()), call
        # every heat decayed exactly once more than before the call
        heat = (heat * F32(0.7)).astype(F32)
        assert np.array_equal(my_heat.cpu().numpy(), heat), call


def test_noalloc_rejects_sizes_beyond_the_static_scratch():
    """Checked before anything reaches the device: the Python wrapper raises, the C entry returns EINVAL."""
    for L, E in [(1025, 4), (64, 1025), (40, 1000), (1024, 33)]:
        with pytest.raises(ValueError, match="static scratch"):
            moe.cache_plan_swaps_noalloc(16, 16, L, E, 1.5, 96, 0.7, 16, 16)
    lib = moe.load()
    cfg = moe.moe_policy_cfg(1.5, 96, 0.7)
    fake = C.c_void_p(256)  # never dereferenced: the size check comes first
    for L, E in [(1025, 4), (64, 1025), (40, 1000), (1024, 33), (0, 8), (8, 0)]:
        assert lib.cache_plan_swaps_noalloc(fake, fake, L, E, C.byref(cfg), fake, fake, None) == moe.MOE_EINVAL
    assert lib.cache_plan_swaps_noalloc(fake, fake, 8, 8, None, fake, fake, None) == moe.MOE_EINVAL
