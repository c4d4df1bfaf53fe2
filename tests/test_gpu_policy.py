"""GPU parity of the cache policy (heat update, swap planning with decay, swap execution)
against the fp32 oracle: plans and heats bit-exact, residency equal to the plan applied."""
import numpy as np
import pytest
import torch

from oracle import policy as opol
from serving_router_top_gb300 import moe
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def make_cache(L, E, resident, H=64, I=32, seed=0):
    """A cache whose backing blobs are distinct random bytes, with `resident` [L,E] admitted."""
    nb = moe.moe_blob_bytes(H, I)
    g = np.random.default_rng(seed)
    backing = torch.from_numpy(g.integers(0, 256, size=L * E * nb, dtype=np.uint8)).cuda()
    c = moe.Cache(L, E, H, I, int(resident.sum()), 0, backing, True)
    c.fill(resident.astype(np.uint8))
    return c, backing, nb


def set_heat(c, heat):
    _, _, h = c.tables()
    h.copy_(torch.from_numpy(heat))


def run_plan(c, thr=1.5, cap=96, decay=0.7):
    plan = torch.zeros(max(cap, 1) * 5, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.cache_plan_swaps(c, thr, cap, decay, plan, n)
    torch.cuda.synchronize()
    cnt = int(n.item())
    arr = plan.cpu().numpy().view(moe.SWAP_DTYPE)[:cnt]
    return arr, plan, n


def plans_equal(got, ref):
    assert len(got) == len(ref), (len(got), len(ref))
    for a, b in zip(got, ref):
        assert (int(a["layer"]), int(a["hot_expert"]), int(a["cold_expert"]), int(a["slot"])) == \
               (b.layer, b.hot_expert, b.cold_expert, b.slot)
        assert F32(a["diff"]) == F32(b.diff)


def test_heat_update_bit_exact():
    L, E, k, T = 3, 40, 5, 17
    resident = np.zeros((L, E), dtype=bool)
    c, _, _ = make_cache(L, E, resident)
    g = np.random.default_rng(1)
    heat = (g.random(L * E) * 50).astype(F32)
    set_heat(c, heat)
    ref = heat.copy()
    for step in range(20):
        layer = step % L
        ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        moe.cache_heat_update(c, torch.from_numpy(ids).cuda(), T, k, layer)
        opol.heat_update(ref, ids, layer, E)
    torch.cuda.synchronize()
    assert np.array_equal(c.tables()[2].cpu().numpy(), ref)


@pytest.mark.parametrize("T", [17, 600])   # one-CTA grouping, and the multi-CTA passes (T*k > 4096)
def test_fused_heat_in_grouping_bit_exact(T):
    """moe_group with the workspace's fused heat on adds exactly the oracle's heat update;
    off, the heats stay as they were."""
    L, E, k = 3, 40, 8
    resident = np.zeros((L, E), dtype=bool)
    resident[:, ::3] = True
    c, _, _ = make_cache(L, E, resident)
    ws = moe.Workspace(T, 64, 64, E, k, 0)
    g = np.random.default_rng(T)
    heat = (g.random(L * E) * 50).astype(F32)
    set_heat(c, heat)
    ref = heat.copy()
    ws.set_fused_heat(True)
    for step in range(6):
        layer = step % L
        ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        moe.moe_group(torch.from_numpy(ids).cuda(), T, k, E, layer, c, ws)
        opol.heat_update(ref, ids, layer, E)
    torch.cuda.synchronize()
    assert moe.moe_sync_status(ws) in (moe.MOE_OK, moe.MOE_EMISSING)
    assert np.array_equal(c.tables()[2].cpu().numpy(), ref)
    ws.set_fused_heat(False)
    moe.moe_group(torch.from_numpy(ids).cuda(), T, k, E, 0, c, ws)
    torch.cuda.synchronize()
    assert np.array_equal(c.tables()[2].cpu().numpy(), ref)


def test_fused_heat_in_layer_forward_bit_exact():
    """The decode window's fused top-k + grouping kernel adds the heat update of its ids."""
    from serving_router_top_gb300 import inputs as I
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["decode_t4_h2048_e512_k10"]
    st = ModelState(w, layers=2)
    E = w.shape.E
    g = np.random.default_rng(7)
    heat = (g.random(2 * E) * 20).astype(F32)
    set_heat(st.cache, heat)
    ref = heat.copy()
    st.ws.set_fused_heat(True)
    y = torch.zeros((w.T, w.shape.H), dtype=torch.float32, device="cuda")
    for step in range(4):
        layer = step % 2
        x = torch.from_numpy(I.activations(w.seed, step, w.T, w.shape.H).view(np.int16)).cuda()
        st.forward(layer, x, y, w.T)
        ids = st.ws.routing(w.T)[1].cpu().numpy()
        opol.heat_update(ref, ids, layer, E)
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    assert np.array_equal(st.cache.tables()[2].cpu().numpy(), ref)


@pytest.mark.parametrize("L,E,seed", [(1, 4, 0), (3, 37, 1), (8, 256, 2), (48, 512, 3)])
def test_plan_swaps_bit_exact(L, E, seed):
    g = np.random.default_rng(seed)
    resident = g.random((L, E)) < 0.3
    c, _, _ = make_cache(L, E, resident)
    # integer-valued heats with many ties and exact-threshold differences, then decayed values
    heat = (g.integers(0, 12, size=L * E) * F32(0.5)).astype(F32)
    heat[g.random(L * E) < 0.1] *= F32(0.7)
    set_heat(c, heat)
    resid = c.tables()[0].cpu().numpy()
    ref_heat = heat.copy()
    ref = opol.plan_round(ref_heat, resid, L, E)
    got, _, _ = run_plan(c)
    plans_equal(got, ref)
    assert np.array_equal(c.tables()[2].cpu().numpy(), ref_heat)


def test_plan_worked_example_and_cap():
    E = 4
    resident = np.array([[False, True, False, False]])
    c, _, _ = make_cache(1, E, resident)
    set_heat(c, np.array([10, 8, 0, 0], dtype=F32))
    got, _, _ = run_plan(c)
    assert len(got) == 1 and int(got[0]["hot_expert"]) == 0 and int(got[0]["cold_expert"]) == 1
    assert F32(got[0]["diff"]) == F32(2.0)
    assert c.tables()[2].cpu().numpy().tolist() == [F32(7.0), F32(5.6), 0, 0]
    # decay-only round: nothing left to pair
    set_heat(c, np.array([1, 0, 0, 0], dtype=F32))
    got, _, _ = run_plan(c)
    assert len(got) == 0 and c.tables()[2].cpu().numpy()[0] == F32(0.7)
    # cap: 100 candidates -> 96
    L, E = 4, 64
    res = np.zeros((L, E), dtype=bool)
    res[:, 32:57] = True
    c2, _, _ = make_cache(L, E, res)
    heat = np.zeros(L * E, dtype=F32)
    g = np.random.default_rng(5)
    for l in range(L):
        heat[l * E:l * E + 25] = (2 + g.integers(0, 1000, 25)).astype(F32)
    set_heat(c2, heat)
    resid = c2.tables()[0].cpu().numpy()
    ref = opol.plan_swaps(heat.copy(), resid, L, E)
    got, _, _ = run_plan(c2)
    assert len(ref) == 96
    plans_equal(got, ref)


def test_apply_swaps_publishes_after_copy():
    L, E = 2, 24
    g = np.random.default_rng(7)
    resident = g.random((L, E)) < 0.4
    c, backing, nb = make_cache(L, E, resident)
    heat = g.integers(0, 20, size=L * E).astype(F32)
    set_heat(c, heat)
    resid_before = c.tables()[0].cpu().numpy()
    ref_plan = opol.plan_swaps(heat.copy(), resid_before, L, E)
    got, plan, n = run_plan(c)
    plans_equal(got, ref_plan)
    copy = torch.cuda.Stream()
    moe.moe_cache_apply_swaps(c, plan, n, torch.cuda.current_stream(), copy)
    torch.cuda.synchronize()
    ref_resid = resid_before.copy()
    opol.apply_swaps(ref_resid, ref_plan, E)
    resid = c.tables()[0].cpu().numpy()
    assert np.array_equal(resid, ref_resid)
    # every resident slot holds exactly its expert's backing blob
    pool = moe.device_view(c.view.slots, (c.nslots * nb,), "uint8", c)
    for f in np.flatnonzero(resid >= 0):
        s = int(resid[f])
        assert torch.equal(pool[s * nb:(s + 1) * nb], backing[f * nb:(f + 1) * nb]), f


# ------------------------------------------------------------ global LRU
# (FreeToken reading notes, 3.3 and 4: one LRU for all layers; K victims per pass)

def _zipf_ids(g, T, k, E, perm, s=1.1):
    p = 1.0 / np.arange(1, E + 1) ** s
    p = p[np.argsort(perm)]
    p /= p.sum()
    return np.stack([g.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("L,E,nslots,T,k,K,calls", [
    (3, 24, 10, 2, 3, 4, 60),       # a small pool, K below the misses of many calls
    (4, 64, 40, 4, 6, 32, 80),      # empty slots at the start, admissions across layers
    (2, 512, 300, 4, 10, 32, 40),   # the decode window's routing shape
])
def test_lru_plans_and_residency_bit_exact(L, E, nslots, T, k, K, calls):
    from oracle import layer as olayer, lru
    H, I_ = 64, 64
    nb = moe.moe_blob_bytes(H, I_)
    g = np.random.default_rng(nslots)
    backing = torch.from_numpy(g.integers(0, 256, size=L * E * nb, dtype=np.uint8)).cuda()
    c = moe.Cache(L, E, H, I_, nslots, 0, backing, True)
    resident = np.zeros((L, E), dtype=bool)
    resident[0, : nslots // 2] = True             # half the slots filled, the rest empty
    c.fill(resident.astype(np.uint8))
    ws = moe.Workspace(T, H, I_, E, k, 0)
    plan = torch.zeros(K * 5, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    resid_o = c.tables()[0].cpu().numpy().copy()
    view = moe.device_view(c.view.slot_owner, (nslots,), "int32", c)
    owner_o = view.cpu().numpy().copy()
    st = lru.new_state(nslots)
    tick_t, clock_t = c.lru_tables()
    perm = g.permutation(E)
    for i in range(calls):
        layer = i % L
        if i % 20 == 0:
            perm = g.permutation(E)                  # the hot set drifts
        ids = _zipf_ids(g, T, k, E, perm)
        moe.moe_group(torch.from_numpy(ids).cuda(), T, k, E, layer, c, ws)
        moe.cache_lru_plan(c, ws, layer, K, plan, n)
        moe.moe_cache_apply_lru(c, plan, n)
        torch.cuda.synchronize()
        assert moe.moe_sync_status(ws) in (moe.MOE_OK, moe.MOE_EMISSING)   # misses have no staging copy here
        grp = olayer.expert_groups(ids)
        slot, src = olayer.lookup(grp.experts, layer, E, resid_o)
        ref = lru.plan_call(st, owner_o, layer, grp.experts, src, slot, K, E)
        lru.apply(resid_o, owner_o, ref, E)
        cnt = int(n.item())
        got = plan.cpu().numpy().view(moe.SWAP_DTYPE)[:cnt]
        assert cnt == len(ref), (i, cnt, len(ref))
        for a, b in zip(got, ref):
            assert (int(a["layer"]), int(a["hot_expert"]), int(a["cold_expert"]), int(a["slot"])) == \
                   (b.layer, b.hot_expert, b.cold_flat, b.slot), i
        assert np.array_equal(tick_t.cpu().numpy().astype(np.int64), st.tick), i
        assert int(clock_t.item()) == st.clock
        assert np.array_equal(c.tables()[0].cpu().numpy(), resid_o), i
        assert np.array_equal(view.cpu().numpy(), owner_o), i
    # the admitted blobs are the backing store's
    slots_t = moe.device_view(c.view.slots, (nslots * nb,), "uint8", c)
    for s in g.choice(nslots, 5, replace=False):
        f = int(owner_o[s])
        if f >= 0:
            assert torch.equal(slots_t[s * nb:(s + 1) * nb], backing[f * nb:(f + 1) * nb])


def test_lru_plan_rejects_bad_k():
    c, _, _ = make_cache(1, 8, np.ones((1, 8), dtype=bool))
    ws = moe.Workspace(2, 64, 64, 8, 2, 0)
    plan = torch.zeros(40 * 5, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    for K in (0, 33):
        with pytest.raises(moe.MoeError):
            moe.cache_lru_plan(c, ws, 0, K, plan, n)


def test_publish_after_copy_race_with_layer_calls():
    """Publish-after-copy under a delayed copy (Strata page, "哪些专家能长期留在显存？": new weights
    become visible only after their copy completes).  The copy stream first runs a timed spin
    (about 0.1 s), so the swap's blob copy lands long after the compute stream could otherwise
    run the layer calls queued behind moe_cache_apply_swaps.  Those calls route every token to
    the swapped-in expert; each output must equal the oracle's, and the last call's lookup must
    find that expert resident in the reused slot: the calls ran after the publish, which waited
    for the copy, so none of them read the slot while it still held the evicted expert."""
    from oracle import layer as olayer
    from serving_router_top_gb300 import inputs as I
    from serving_router_top_gb300.model import ModelState
    T, E = 4, 16
    w = I.small_workload(T=T, H=256, I=128, E=E, k=3, I_shared=128, zipf_s=0.0, resident_frac=0.5, seed=21)
    st = ModelState(w, stage_all=True)   # every expert also staged: the evicted one stays reachable
    resid0 = st.resid_table()[:E]
    A = int(np.flatnonzero(resid0 < 0)[0])    # hot, not resident
    B = int(np.flatnonzero(resid0 >= 0)[0])   # cold, resident
    heat = np.where(resid0 >= 0, F32(100.0), F32(0.0)).astype(F32)
    heat[A], heat[B] = F32(10.0), F32(8.0)    # the page's worked example: 10 - 8 = 2 >= 1.5
    set_heat(st.cache, heat)
    bias = st.layers[0].bias
    bias[A] = 50.0                            # every token's first choice is A
    got, plan, n = run_plan(st.cache)
    assert [(int(s["hot_expert"]), int(s["cold_expert"]), int(s["slot"])) for s in got] == [(A, B, int(resid0[B]))]
    compute = torch.cuda.current_stream()
    copy = torch.cuda.Stream()
    with torch.cuda.stream(copy):
        torch.cuda._sleep(200_000_000)        # ~0.1 s at 2 GHz, bounded: a delay, not a wait
    moe.moe_cache_apply_swaps(st.cache, plan, n, compute, copy)
    xs = [I.activations(w.seed, 50 + i, T, w.shape.H) for i in range(6)]
    ys = [torch.zeros((T, w.shape.H), dtype=torch.float32, device="cuda") for _ in xs]
    for xb, y in zip(xs, ys):
        st.forward(0, torch.from_numpy(xb.view(np.int16)).cuda(), y, T, mode=moe.MOE_MODE_DECODE)
    torch.cuda.synchronize()
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    exp_, _, slot, src, _, _ = st.ws.groups(T)
    gi = int(np.flatnonzero(exp_ == A)[0])
    assert src[gi] == moe.MOE_SRC_RESIDENT and slot[gi] == int(resid0[B])
    li = st.layers[0].host
    bias_h = li.bias.copy()
    bias_h[A] = np.float32(50.0)
    for xb, y in zip(xs, ys):
        logits = olayer.router_logits(xb, li.w_router, bias_h)
        ref = olayer.moe_layer(xb, li.w_router, bias_h, st.k, lambda e: st.expert_host(0, e), st.H, st.I,
                               resid=st.resid_table(), stage=st.stage_table(), shared=li.shared,
                               I_shared=st.I_shared, w_shared_gate_bits=li.w_shared_gate, logits=logits)
        assert (ref.ids[:, 0] == A).all()
        U.assert_close_layer(y.cpu().numpy(), ref.y)
