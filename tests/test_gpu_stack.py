"""GPU parity of the decode-stack workload: layers in sequence over an fp32 residual stream
(residual + RMSNorm between layers), heat updates every step, planning and swaps every few
steps, router biases re-drawn every few steps (drift).

Checked against the oracle:
  * the cache policy replayed in full from the GPU's own top-k ids: every plan, the heats
    and the residency table bit-exact;
  * RMSNorm of the residual stream within one bf16 unit;
  * teacher-forced layer outputs at sampled (step, layer) points, on the GPU's input,
    logits and residency tables of that moment.
The layer shape is the workload's (hidden 2048, 512 experts top-10, I 512, shared expert,
30% of the slots resident); the depth and schedule are scaled down for a test."""
import numpy as np
import pytest
import torch

from oracle import formats, layer as olayer, policy as opol
from serving_router_top_gb300 import inputs as I
from serving_router_top_gb300 import moe
from tests import gpu_util as U

pytestmark = pytest.mark.gpu
F32 = np.float32


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def _bf16_ulp(a):
    a = np.abs(np.asarray(a, dtype=np.float64))
    return np.exp2(np.floor(np.log2(np.maximum(a, 1e-38))) - 7)


@pytest.mark.parametrize("T,steps,sample", [(16, 12, [(5, 1), (10, 2)]), (1, 8, [(6, 0)])])
def test_decode_stack_policy_and_layers(T, steps, sample):
    from serving_router_top_gb300.stack import DecodeStack
    w = I.WORKLOADS["stack48_decode_h2048_e512_k10"]
    L, plan_every, drift_every = 3, 4, 6
    stk = DecodeStack(w, layers=L, maxT=16, plan_every=plan_every, drift_every=drift_every)
    st = stk.st
    E, H, k = st.E, st.H, st.k
    resid0 = st.resid_table().copy()
    ids_log = {}
    samples = {}
    plans = []
    cur = {"step": 0}

    def after_layer(l):
        s = cur["step"]
        logits_t, ids_t, _ = st.ws.routing(T)
        ids_log[(s, l)] = ids_t.cpu().numpy().copy()
        if (s, l) in sample:
            samples[(s, l)] = dict(xn=stk.xn[:T].cpu().numpy().view(np.uint16).copy(),
                                   x_res=x_res.cpu().numpy().astype(np.float64),
                                   y=stk.ys[l][:T].cpu().numpy().view(np.uint16).copy(),
                                   logits=logits_t.cpu().numpy().copy(),
                                   resid=st.resid_table().copy(), stage=st.stage_table().copy(),
                                   bias=st.layers[l].host.bias.copy())

    def after_plan():
        n = int(stk.n_plan.item())
        plans.append(stk.plan.cpu().numpy().view(moe.SWAP_DTYPE)[:n].copy())

    x_res = torch.from_numpy(formats.bf16_value(I.activations(w.seed, 99, T, H)).astype(F32)).cuda()
    resid_after = []
    for s in range(steps):
        cur["step"] = s
        stk.step(x_res, T, s, after_layer=after_layer, after_plan=after_plan)
        torch.cuda.synchronize()
        if plan_every and (s + 1) % plan_every == 0:
            resid_after.append(st.resid_table().copy())
        rc = moe.moe_sync_status(st.ws)
        assert rc == moe.MOE_OK, moe.strerror(rc)

    # ---- the policy, replayed in the oracle from the GPU's own routing
    heat = np.zeros(L * E, dtype=F32)
    resid = resid0.copy()
    pi = 0
    for s in range(steps):
        for l in range(L):
            opol.heat_update(heat, ids_log[(s, l)], l, E)
        if (s + 1) % plan_every == 0:
            ref = opol.plan_round(heat, resid, L, E, 1.5, 96, 0.7)
            got = plans[pi]
            assert len(got) == len(ref), (s, len(got), len(ref))
            for a, b in zip(got, ref):
                assert (int(a["layer"]), int(a["hot_expert"]), int(a["cold_expert"]), int(a["slot"])) == \
                       (b.layer, b.hot_expert, b.cold_expert, b.slot)
                assert F32(a["diff"]) == F32(b.diff)
            opol.apply_swaps(resid, ref, E)
            assert np.array_equal(resid_after[pi], resid), s
            pi += 1
    assert pi > 0 and sum(len(p) for p in plans) > 0  # the schedule did plan some swaps
    assert np.array_equal(st.cache.tables()[2].cpu().numpy(), heat)

    # ---- RMSNorm of the residual stream and teacher-forced layers at the sampled points
    for (s, l), d in samples.items():
        ref_xn = olayer.rmsnorm(d["x_res"])
        got_xn = formats.bf16_value(d["xn"])
        assert np.all(np.abs(got_xn - ref_xn) <= _bf16_ulp(ref_xn)), (s, l)
        li = st.layers[l].host
        ref = olayer.moe_layer(d["xn"], li.w_router, d["bias"], k, lambda e: st.expert_host(l, e), H, st.I,
                               layer=l, resid=d["resid"], stage=d["stage"], shared=li.shared, I_shared=st.I_shared,
                               w_shared_gate_bits=li.w_shared_gate, logits=d["logits"])
        assert np.array_equal(olayer.top_k(d["logits"], k)[0], ids_log[(s, l)])
        U.assert_close_layer(formats.bf16_value(d["y"]), ref.y, bf16_out=True, what=f"y at step {s} layer {l}")


def _to32(bits):
    return torch.from_numpy(formats.bf16_value(bits).astype(F32)).cuda()


def test_stack48_full_schedule_policy_replay():
    """The 48-layer decode stack as specified (hidden 2048, 512 experts top-10, 30% of the 48 x 512
    slots resident, 2048 steps of 4 tokens, planning every 256 steps, drift every 512), run as
    graph replays of whole steps: every plan of the eight rounds, the decayed heats and the
    residency table equal the oracle's replay of the policy on the run's own routing; then
    teacher-forced layers at three depths of one more step, on the cache the schedule left."""
    from serving_router_top_gb300.stack import DecodeStack, run_schedule
    w = I.WORKLOADS["stack48_decode_h2048_e512_k10"]
    T, steps, L = 4, 2048, 48
    stk = DecodeStack(w, layers=L, maxT=16, plan_every=256, drift_every=512)
    st = stk.st
    E, H, k = st.E, st.H, st.k
    resid0 = st.resid_table().copy()
    wins = torch.stack([_to32(I.activations(w.seed, 7000 + i, T, H)) for i in range(16)])
    stream = torch.cuda.Stream()
    ms, swaps, log, plans = run_schedule(stk, T, steps, wins, stream, log_ids=True)
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    assert len(plans) == steps // 256 and swaps > 0
    heat = np.zeros(L * E, dtype=F32)
    resid = resid0.copy()
    for s in range(steps):
        for l in range(L):
            opol.heat_update(heat, log[s, l], l, E)
        if (s + 1) % 256 == 0:
            ref = opol.plan_round(heat, resid, L, E, 1.5, 96, 0.7)
            got = plans[(s + 1) // 256 - 1]
            assert len(got) == len(ref), s
            for a, b in zip(got, ref):
                assert (int(a["layer"]), int(a["hot_expert"]), int(a["cold_expert"]), int(a["slot"])) == \
                       (b.layer, b.hot_expert, b.cold_expert, b.slot)
            opol.apply_swaps(resid, ref, E)
    assert np.array_equal(st.cache.tables()[2].cpu().numpy(), heat)
    assert np.array_equal(st.resid_table(), resid)
    # one more step, teacher-forced checks at three depths
    sample = {0: None, 23: None, 47: None}
    x_res = wins[3].clone()

    def after_layer(l):
        if l in sample:
            logits_t, _, _ = st.ws.routing(T)
            sample[l] = dict(xn=stk.xn[:T].cpu().numpy().view(np.uint16).copy(),
                             y=stk.ys[l][:T].cpu().numpy().view(np.uint16).copy(),
                             logits=logits_t.cpu().numpy().copy(), resid=st.resid_table().copy(),
                             stage=st.stage_table().copy(), bias=st.layers[l].host.bias.copy())

    stk.layers_pass(x_res, T, after_layer=after_layer)
    torch.cuda.synchronize()
    for l, d in sample.items():
        li = st.layers[l].host
        ref = olayer.moe_layer(d["xn"], li.w_router, d["bias"], k, lambda e: st.expert_host(l, e), H, st.I,
                               layer=l, resid=d["resid"], stage=d["stage"], shared=li.shared, I_shared=st.I_shared,
                               w_shared_gate_bits=li.w_shared_gate, logits=d["logits"])
        U.assert_close_layer(formats.bf16_value(d["y"]), ref.y, bf16_out=True, what=f"y at layer {l}")
    del stk, st
    torch.cuda.empty_cache()


def test_mixed_prefill_then_decode_large_model():
    """The 4096-hidden, 256-expert top-6 model (8 layers, all resident): a 4096-token prefill
    chunk through all 8 layers, then decode steps at batch 64; teacher-forced checks of sampled
    layers in both phases (prefill: 16 sampled tokens; decode: every token), each on the
    GPU's own input rows and logits of that layer."""
    from serving_router_top_gb300.stack import DecodeStack
    w = I.WORKLOADS["large_h4096_e256_k6"]
    Tp, Td, L = 4096, 64, 8
    stk = DecodeStack(w, layers=L, maxT=Tp, plan_every=0, drift_every=0, stage_all=False)
    st = stk.st
    H, k = st.H, st.k
    toks = np.random.default_rng(3).choice(Tp, 16, replace=False)
    checks = []

    def sampler(layers, rows):
        def after_layer(l):
            if l in layers:
                T = rows
                logits_t, _, _ = st.ws.routing(T)
                checks.append(dict(l=l, T=T, xn=stk.xn[:T].cpu().numpy().view(np.uint16).copy(),
                                   y=stk.ys[l][:T].cpu().numpy().view(np.uint16).copy(),
                                   logits=logits_t.cpu().numpy().copy()))
        return after_layer

    x_pre = _to32(I.activations(w.seed, 60_000, Tp, H))
    stk.layers_pass(x_pre, Tp, after_layer=sampler({0, 5}, Tp))
    x_dec = _to32(I.activations(w.seed, 61_000, Td, H))
    for s in range(3):
        stk.layers_pass(x_dec, Td, after_layer=sampler({2, 7} if s == 2 else set(), Td))
    torch.cuda.synchronize()
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    for d in checks:
        li = st.layers[d["l"]].host
        sel = toks if d["T"] == Tp else np.arange(d["T"])
        ref = olayer.moe_layer(d["xn"][sel], li.w_router, li.bias, k, lambda e: st.expert_host(d["l"], e), H, st.I,
                               layer=d["l"], shared=li.shared, I_shared=st.I_shared,
                               w_shared_gate_bits=li.w_shared_gate, logits=d["logits"][sel])
        U.assert_close_layer(formats.bf16_value(d["y"][sel]), ref.y, bf16_out=True,
                             what=f"y at layer {d['l']}, {d['T']} tokens")
    del stk, st
    torch.cuda.empty_cache()
