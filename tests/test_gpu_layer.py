"""GPU parity of the whole layer (router -> top-k -> groups -> lookup -> experts -> combine)
against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import layer as olayer
from serving_router_top_gb300 import inputs as I
from serving_router_top_gb300 import moe
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def run_layer(st, x_bits, T, bf16_out=False, layer=0, mode=moe.MOE_MODE_AUTO):
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    if bf16_out:
        y = torch.zeros((T, st.H), dtype=torch.int16, device="cuda")
    else:
        y = torch.zeros((T, st.H), dtype=torch.float32, device="cuda")
    st.forward(layer, x, y, T, y_is_fp32=not bf16_out, mode=mode)
    rc = moe.moe_sync_status(st.ws)
    assert rc == moe.MOE_OK, moe.strerror(rc)
    return U.y_to_numpy(y, bf16_out)


def check_layer(st, T, bf16_out=False, step=0, layer=0, tail_skip=0, mode=moe.MOE_MODE_AUTO):
    x_bits = I.activations(st.w.seed, step, T, st.H)
    y = run_layer(st, x_bits, T, bf16_out, layer, mode)
    logits_t, ids_t, w_t = st.ws.routing(T)
    logits = logits_t.cpu().numpy()
    ids = ids_t.cpu().numpy()
    w = w_t.cpu().numpy()
    li = st.layers[layer].host
    # router logits: within the fp32-accumulation bound of the oracle's
    ref_logits = olayer.router_logits(x_bits, li.w_router, li.bias)
    bound = U.logits_bound(x_bits, li.w_router, li.bias)
    assert np.all(np.abs(logits.astype(np.float64) - ref_logits) <= bound)
    # top-k on the same fp32 logits: bit-exact ids, weights to fp32 rounding
    ref_ids, ref_w = olayer.top_k(logits, st.k)
    assert np.array_equal(ids, ref_ids)
    assert np.allclose(w, ref_w, rtol=1e-5, atol=1e-7)
    # top-k on the oracle's own logits differs only at near-ties
    o_ids, _ = olayer.top_k(ref_logits, st.k)
    for t in np.flatnonzero((o_ids != ids).any(axis=1)):
        srt = np.sort(ref_logits[t].astype(np.float64))[::-1]
        gaps = np.abs(np.diff(srt[: st.k + 1]))
        assert gaps.min() <= 2 * bound[t].max(), t
    # the rest of the layer on identical routing
    ref = U.oracle_layer_from_state(st, layer, x_bits, logits, tail_skip=tail_skip)
    exp_, off, slot, src, ent_tok, ent_pos = st.ws.groups(T)
    assert np.array_equal(exp_, ref.groups.experts)
    assert np.array_equal(off, ref.groups.off)
    assert np.array_equal(ent_tok, ref.groups.ent_tok)
    assert np.array_equal(ent_pos, ref.groups.ent_pos)
    assert np.array_equal(slot, ref.slot)
    assert np.array_equal(src, ref.src)
    return U.assert_close_layer(y, ref.y, bf16_out), ref


def test_layer_t8_h256_e16_k2():
    st_ = I.WORKLOADS["layer_t8_h256_e16_k2"]
    from serving_router_top_gb300.model import ModelState
    st = ModelState(st_)
    for step in range(3):
        check_layer(st, st_.T, step=step)
    check_layer(st, st_.T, bf16_out=True, step=5)


@pytest.mark.parametrize("T,H,I_,E,k,Is,frac", [
    (1, 128, 64, 12, 3, 64, 1.0),
    (5, 128, 64, 12, 3, 64, 0.5),      # ragged token count, half staged
    (7, 256, 128, 40, 7, 64, 0.25),    # shared intermediate narrower than routed
    (33, 64, 64, 9, 9, 0, 1.0),        # k == E, no shared expert, narrowest rows
    (64, 1024, 256, 64, 6, 256, 0.5),
    (3, 4096, 2048, 16, 2, 2048, 1.0),  # the large-expert row widths
    (2, 128, 64, 1, 1, 64, 1.0),        # a single routed expert (weight 1) and the shared one
    (8, 256, 128, 40, 7, 64, 0.5),      # the largest window of the decode GEMVs
    (9, 256, 128, 40, 7, 64, 0.5),      # the smallest window of the streaming kernels
])
def test_layer_small_shapes(T, H, I_, E, k, Is, frac):
    """The decode kernels at every window size (forced past 32 tokens, where AUTO takes the
    prefill kernels), then AUTO on fewer tokens than the workspace was sized for."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=H, I=I_, E=E, k=k, I_shared=Is, zipf_s=0.8, resident_frac=frac, seed=T + E)
    st = ModelState(w)
    check_layer(st, T, mode=moe.MOE_MODE_DECODE)
    check_layer(st, max(1, T // 2), step=1)


@pytest.mark.parametrize("T,H,I_,E,k,Is,frac", [
    (1, 128, 64, 12, 3, 64, 1.0),
    (5, 128, 64, 12, 3, 64, 0.5),
    (7, 256, 128, 40, 7, 64, 0.25),
    (8, 256, 128, 40, 7, 64, 0.5),      # the largest window of the chain's GEMVs
    (12, 512, 256, 64, 6, 256, 0.5),    # the chain's streaming kernel below 32 tokens
    (4, 2048, 512, 512, 10, 512, 0.5),  # the decode window's shapes
])
def test_layer_decode_chain(T, H, I_, E, k, Is, frac):
    """The chain of decode kernels (router, top-k + groups, gate/up, down, combine), which the
    single kernel replaces by default: every shape against the oracle, fp32 and bf16 out."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=H, I=I_, E=E, k=k, I_shared=Is, zipf_s=0.8, resident_frac=frac, seed=2 * T + E)
    st = ModelState(w)
    st.ws.set_decode_path(moe.MOE_DECODE_CHAIN)
    st.ws.set_profiling(True)
    check_layer(st, T, mode=moe.MOE_MODE_DECODE)
    assert "decode_fused" not in [n for n, _ in st.ws.kernel_times()]
    st.ws.set_profiling(False)
    check_layer(st, T, bf16_out=True, step=1, mode=moe.MOE_MODE_DECODE)


def test_layer_decode_t4_h2048_e512_k10():
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["decode_t4_h2048_e512_k10"]
    st = ModelState(w)
    rel, ref = check_layer(st, w.T)
    assert (ref.src == moe.MOE_SRC_STAGED).any() and (ref.src == moe.MOE_SRC_RESIDENT).any()
    check_layer(st, w.T, bf16_out=True, step=1)
    stats = st.cache.stats()
    assert stats[0, 0] == stats[0, 1] + stats[0, 2] and stats[0, 3] == 0


# ------------------------------------------------------------ tail skip
# (Strata page, "跳过尾部专家"): a non-resident expert that every choosing token
# ranks at or past the threshold is dropped; no renormalisation.

def test_tail_skip_decode_window():
    """The page's threshold (7, zero-based ranks) on the verify window: groups, sources and
    slots bit-exact, y within tolerance of the oracle's layer with the same groups dropped,
    and the drops counted."""
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["decode_t4_h2048_e512_k10"]
    st = ModelState(w)
    st.ws.set_tail_skip(7)
    n_skip = 0
    for step in range(4):
        _, ref = check_layer(st, w.T, step=step, tail_skip=7)
        n_skip += int((ref.src == olayer.SRC_SKIPPED).sum())
    assert n_skip > 0
    stats = st.cache.stats()
    assert stats[0, 4] == n_skip and stats[0, 3] == 0
    assert stats[0, 0] == stats[0, 1] + stats[0, 2] + stats[0, 4]
    st.ws.set_tail_skip(0)
    _, ref = check_layer(st, w.T, step=0)
    assert not (ref.src == olayer.SRC_SKIPPED).any()


@pytest.mark.parametrize("T,R", [(5, 1), (8, 2), (64, 2)])   # GEMV path, and the streaming kernel past 8 tokens
def test_tail_skip_small_windows(T, R):
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=256, I=128, E=24, k=4, I_shared=128, zipf_s=0.6, resident_frac=0.5, seed=11 + T)
    st = ModelState(w)
    st.ws.set_tail_skip(R)
    n_skip = 0
    for step in range(3):
        _, ref = check_layer(st, T, step=step, tail_skip=R, mode=moe.MOE_MODE_DECODE)
        n_skip += int((ref.src == olayer.SRC_SKIPPED).sum())
    assert n_skip > 0


def _split_ids(rng, T, k, R, low, high):
    """Each token's ranks 0..R-1 from `low`, ranks R..k-1 from `high` (distinct within a row)."""
    ids = np.zeros((T, k), dtype=np.int32)
    for t in range(T):
        ids[t, :R] = rng.choice(low, R, replace=False)
        ids[t, R:] = rng.choice(high, k - R, replace=False)
    return ids


@pytest.mark.parametrize("T", [100, 600])   # one-CTA grouping, and the three multi-CTA passes (T*k > 4096)
def test_tail_skip_grouping_missing_experts(T):
    """Every non-resident expert is missing (no staging) but chosen only at ranks >= R: with the
    tail skip at R the grouping drops them all and records no error; off, MOE_EMISSING.  Groups
    and sources bit-exact against the oracle's lookup and drop rule on both grouping paths."""
    from serving_router_top_gb300.model import ModelState
    E, k, R = 64, 8, 5
    w = I.small_workload(T=T, H=128, I=64, E=E, k=k, I_shared=0, resident_frac=0.5, seed=5)
    st = ModelState(w, stage_rest=False)
    resid = st.resid_table()
    res_e = np.flatnonzero(resid[:E] >= 0)
    non_e = np.flatnonzero(resid[:E] < 0)
    assert len(res_e) >= R and len(non_e) >= k - R
    ids = _split_ids(np.random.default_rng(T), T, k, R, res_e, non_e)
    ids_t = torch.from_numpy(ids).cuda()
    st.ws.set_tail_skip(R)
    moe.moe_group(ids_t, T, k, E, 0, st.cache, st.ws)
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    g = olayer.expert_groups(ids)
    slot, src = olayer.lookup(g.experts, 0, E, resid, st.stage_table())
    drop = olayer.tail_skip_mask(g, src, k, R)
    src[drop] = olayer.SRC_SKIPPED
    slot[drop] = olayer.MISSING
    assert drop.sum() == len(set(ids[:, R:].ravel()))
    exp_, off, gslot, gsrc, ent_tok, ent_pos = st.ws.groups(T)
    assert np.array_equal(exp_, g.experts) and np.array_equal(off, g.off)
    assert np.array_equal(ent_tok, g.ent_tok) and np.array_equal(ent_pos, g.ent_pos)
    assert np.array_equal(gslot, slot) and np.array_equal(gsrc, src)
    assert st.cache.stats()[0, 4] == drop.sum()
    # one token ranking a missing expert above R keeps it: an error again
    ids2 = ids.copy()
    ids2[0, 0], ids2[0, R] = ids2[0, R], ids2[0, 0]
    moe.moe_group(torch.from_numpy(ids2).cuda(), T, k, E, 0, st.cache, st.ws)
    assert moe.moe_sync_status(st.ws) == moe.MOE_EMISSING
    st.ws.set_tail_skip(0)
    moe.moe_group(ids_t, T, k, E, 0, st.cache, st.ws)
    assert moe.moe_sync_status(st.ws) == moe.MOE_EMISSING


def test_tail_skip_rejects_negative_rank():
    from serving_router_top_gb300.model import ModelState
    st = ModelState(I.small_workload(T=2, H=128, I=64, E=8, k=2, I_shared=0))
    with pytest.raises(moe.MoeError):
        st.ws.set_tail_skip(-1)


@pytest.mark.parametrize("T,E,k", [(4, 512, 10), (12, 64, 10), (32, 64, 6)])
def test_fused_topk_group_all_ties(T, E, k):
    """Router weights zeroed and no bias: every logit is 0, so each token takes experts
    0..k-1 with weights 1/k (ties to the lower id), through the fused top-k + grouping."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=128, I=64, E=E, k=k, I_shared=0, zipf_s=0.0, resident_frac=1.0, seed=2)
    st = ModelState(w)
    st.layers[0].w_router.zero_()
    st.layers[0].bias.zero_()
    x = torch.from_numpy(I.activations(w.seed, 0, T, 128).view(np.int16)).cuda()
    y = torch.zeros((T, 128), dtype=torch.float32, device="cuda")
    st.forward(0, x, y, T, mode=moe.MOE_MODE_DECODE)
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    _, ids_t, w_t = st.ws.routing(T)
    assert np.array_equal(ids_t.cpu().numpy(), np.tile(np.arange(k, dtype=np.int32), (T, 1)))
    assert np.all(w_t.cpu().numpy() == np.float32(1.0) / np.float32(k))
    exp_, off, _, _, ent_tok, _ = st.ws.groups(T)
    assert exp_.tolist() == list(range(k)) and off.tolist() == [T * r for r in range(k + 1)]
    assert ent_tok.tolist() == list(range(T)) * k


def test_empty_window_is_a_no_op():
    """T = 0 through every call: MOE_OK, nothing written."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=4, H=128, I=64, E=8, k=2, I_shared=64, resident_frac=0.5, seed=4)
    st = ModelState(w)
    x = torch.zeros((4, 128), dtype=torch.int16, device="cuda")
    y = torch.full((4, 128), 7.0, dtype=torch.float32, device="cuda")
    for mode in (moe.MOE_MODE_DECODE, moe.MOE_MODE_PREFILL, moe.MOE_MODE_AUTO):
        st.forward(0, x, y, 0, mode=mode)
    ids = torch.zeros((4, 2), dtype=torch.int32, device="cuda")
    moe.moe_group(ids, 0, 2, 8, 0, st.cache, st.ws)
    moe.cache_heat_update(st.cache, ids, 0, 2, 0)
    torch.cuda.synchronize()
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    assert bool((y == 7.0).all())
    assert float(st.cache.tables()[2].abs().sum()) == 0.0   # no heat added


def test_missing_expert_is_reported():
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=6, H=128, I=64, E=12, k=3, I_shared=0, resident_frac=0.25, seed=3)
    st = ModelState(w, stage_rest=False)
    x = torch.from_numpy(I.activations(w.seed, 0, 6, 128).view(np.int16)).cuda()
    y = torch.zeros((6, 128), dtype=torch.float32, device="cuda")
    st.forward(0, x, y, 6)
    assert moe.moe_sync_status(st.ws) == moe.MOE_EMISSING
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK  # cleared


def test_route_same_logits_mode_ties_and_nan():
    U.require_gpu()
    T, E, k = 9, 37, 5
    g = np.random.default_rng(0)
    logits = g.integers(-2, 3, size=(T, E)).astype(np.float32)  # many exact ties
    lt = torch.from_numpy(logits).cuda()
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_route(None, None, None, lt, T, 0, E, k, ids, w, err)
    torch.cuda.synchronize()
    ref_ids, ref_w = olayer.top_k(logits, k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.allclose(w.cpu().numpy(), ref_w, rtol=1e-6)
    assert int(err.item()) == 0
    logits[2, 4] = np.nan
    moe.moe_route(None, None, None, torch.from_numpy(logits).cuda(), T, 0, E, k, ids, w, err)
    torch.cuda.synchronize()
    assert int(err.item()) == moe.MOE_ENAN


def test_group_rejects_out_of_range_ids():
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=4, H=64, I=64, E=8, k=2, I_shared=0)
    st = ModelState(w)
    ids = torch.tensor([[0, 1], [2, 9], [3, 4], [5, 6]], dtype=torch.int32, device="cuda")
    moe.moe_group(ids, 4, 2, 8, 0, st.cache, st.ws)
    assert moe.moe_sync_status(st.ws) == moe.MOE_ERANGE


def test_large_expert_layer_decode_batch64_all_tokens():
    """One layer of the 4096-hidden, 256-expert top-6 model (I = I_shared = 2048) decoding a batch of
    64 tokens: every token against the oracle, plus the router, routing and groups as check_layer --
    on the decode kernels (the streaming expert tiles) and under AUTO (the grouped GEMMs, which
    AUTO takes from 32 tokens on)."""
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["large_h4096_e256_k6"]
    st = ModelState(w, layers=1, maxT=64)
    check_layer(st, 64, step=7, mode=moe.MOE_MODE_DECODE)
    st.ws.set_profiling(True)
    check_layer(st, 64, step=8)
    assert "gateup_gemm" in [n for n, _ in st.ws.kernel_times()]
    st.ws.set_profiling(False)


@pytest.mark.parametrize("T", [6, 20])   # the decode GEMVs; the streaming kernel past 8 tokens
def test_layer_edge_format(T):
    """Zero, subnormal and 448 block scales and global scales 0.375 / 2.0 / 1.25 (gate, up, down)
    through the decode path, fp32 and bf16 output."""
    from serving_router_top_gb300.model import ModelState
    w = I.edge_workload(T=T)
    st = ModelState(w)
    check_layer(st, T)
    check_layer(st, T, bf16_out=True, step=1)


@pytest.mark.parametrize("T,H,I_,E,k,frac", [
    (1, 2048, 512, 512, 10, 0.5),   # eight warps per token
    (4, 2048, 512, 512, 10, 0.5),   # the decode window: eight warps per token
    (8, 256, 128, 40, 7, 0.5),      # four warps per token, E not a multiple of the slices
    (12, 256, 128, 1000, 10, 0.5),  # two warps per token, 32 logits per lane, 120 entries
    (3, 128, 64, 16, 16, 1.0),      # k = E = 16: every expert
    (16, 256, 128, 64, 6, 0.4),     # two warps per token
    (16, 256, 128, 64, 8, 0.5),     # 128 entries
    (32, 256, 128, 40, 7, 0.6),     # one warp per token, E not a multiple of the slices
])
def test_fused_topk_group_equals_separate_kernels(T, H, I_, E, k, frac):
    """The decode forward's single-CTA top-k + grouping (several warps per token) gives the
    same ids, weights (bit for bit) and groups as the separate top-k kernel and grouping call
    on the same logits."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=H, I=I_, E=E, k=k, I_shared=0, zipf_s=1.0, resident_frac=frac, seed=7 * T + E)
    st = ModelState(w)
    x = torch.from_numpy(I.activations(w.seed, 3, T, H).view(np.int16)).cuda()
    y = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    st.forward(0, x, y, T, mode=moe.MOE_MODE_DECODE)
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    logits_t, ids_t, w_t = st.ws.routing(T)
    logits = logits_t.clone()
    fused_ids, fused_w = ids_t.cpu().numpy().copy(), w_t.cpu().numpy().copy()
    fused_groups = st.ws.groups(T)
    ids = torch.zeros((T, k), dtype=torch.int32, device="cuda")
    wts = torch.zeros((T, k), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_route(None, None, None, logits, T, 0, E, k, ids, wts, err)
    moe.moe_group(ids, T, k, E, 0, st.cache, st.ws)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(ids.cpu().numpy(), fused_ids)
    assert np.array_equal(wts.cpu().numpy().view(np.uint32), fused_w.view(np.uint32))
    for a, b in zip(st.ws.groups(T), fused_groups):
        assert np.array_equal(a, b)
    # and both are the oracle's top-k on these logits
    ref_ids, _ = olayer.top_k(logits.cpu().numpy(), k)
    assert np.array_equal(fused_ids, ref_ids)
