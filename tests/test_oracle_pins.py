"""Pins of the CPU oracle to facts fixed outside itself: the pages' printed values,
library decoders, brute force on tiny inputs, closed forms and invariants."""
import itertools

import numpy as np
import pytest
import scipy.special
import torch

from oracle import formats, layer, policy, side
from serving_router_top_gb300 import inputs
from tests.conftest import read_golden

F32 = np.float32


# ---------------------------------------------------------------- formats

def test_fp4_table_matches_page():
    mags = [float(v) for v in read_golden("fp4_magnitudes.txt")[0]]
    codes = np.arange(16, dtype=np.uint8)
    vals = formats.e2m1_value(codes)
    for c in range(16):
        expect = mags[c & 7] * (-1.0 if c & 8 else 1.0)
        assert vals[c] == expect or (expect == 0 and vals[c] == 0), (c, vals[c], expect)


def test_e4m3_all_codes_match_torch_decoder():
    b = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(b).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = formats.e4m3_value(b)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert nan.sum() == 2  # S.1111.111 only: no infinities
    assert np.array_equal(ref[~nan], got[~nan])


def test_bf16_decode_matches_torch():
    bits = np.random.default_rng(3).integers(0, 1 << 16, 4096).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = formats.bf16_value(bits)
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok]) and np.array_equal(np.isnan(ref), np.isnan(got))


def test_nibble_order_low_first():
    # the page names the low 4 bits first: byte 0x2F holds code 0xF then code 0x2
    assert formats.unpack_codes(np.array([[0x2F]], dtype=np.uint8)).tolist() == [[0xF, 0x2]]


def test_packed_row_arithmetic_matches_page():
    g = {r[0]: int(r[1]) for r in read_golden("packed_row.txt")}
    cols = g["values_per_row"]
    assert cols // 2 == g["code_bytes"] and cols // g["block_size"] == g["scale_bytes"]
    assert inputs.packed_row_bytes(cols) == g["row_bytes"]
    assert g["heads_per_token"] * inputs.packed_row_bytes(cols) == g["packed_bytes_per_token"]
    assert g["heads_per_token"] * cols * 2 == g["bf16_bytes_per_token"]
    assert round(100 * g["packed_bytes_per_token"] / g["bf16_bytes_per_token"]) == g["packed_over_bf16_percent"]
    # a 16-head packed token of 160-value rows dequantises to 16 x 160 values
    packed = inputs.packed_matrix(inputs.rng(0, 99), 16, cols)
    assert packed.nbytes == g["packed_bytes_per_token"]
    assert formats.dequantize(packed, cols).shape == (16, 160)


def test_dequant_chain_against_torch_fp8_and_page_table():
    """value = FP4 value x FP8 block scale x FP32 global scale, checked with an independent
    decoder for the scales (torch) and the page's table for the codes."""
    cols, rows = 64, 7
    packed = inputs.packed_matrix(inputs.rng(0, 5), rows, cols)
    mags = [float(v) for v in read_golden("fp4_magnitudes.txt")[0]]
    gscale = 0.375
    got = formats.dequantize(packed, cols, gscale)
    sc = torch.from_numpy(packed[:, cols // 2:].copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for r in range(rows):
        for c in range(cols):
            byte = packed[r, c // 2]
            code = (byte & 0xF) if c % 2 == 0 else (byte >> 4)
            v = mags[code & 7] * (-1 if code & 8 else 1) * sc[r, c // 16] * gscale
            assert got[r, c] == v


def test_dequant_is_exact_in_bf16():
    """FP4 (2 significant bits) x E4M3 (4 significant bits) fits bf16's 8 bits:
    the dequantised weights of the generated scale range are bf16-exact."""
    packed = inputs.packed_matrix(inputs.rng(0, 6), 64, 256)
    v = formats.dequantize(packed, 256).astype(np.float32)
    as_bf16 = torch.from_numpy(v).to(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(v, as_bf16)


# ---------------------------------------------------------------- router / top-k

def _brute_topk_set(l, k):
    """Among all k-subsets, the one with the largest logit sum, then the smallest id sum
    (integer logits, so sums are exact)."""
    best = None
    for sub in itertools.combinations(range(len(l)), k):
        key = (sum(int(l[i]) for i in sub), -sum(sub))
        if best is None or key > best[0]:
            best = (key, sub)
    return set(best[1])


@pytest.mark.parametrize("E", [1, 2, 5, 8, 12])
def test_topk_brute_force_tiny(E):
    g = np.random.default_rng(E)
    for k in range(1, E + 1):
        for _ in range(6):
            l = g.integers(-3, 4, size=(3, E)).astype(np.float32)   # many ties
            ids, w = layer.top_k(l, k)
            for t in range(3):
                assert set(ids[t].tolist()) == _brute_topk_set(l[t], k)
                # order: logit descending, ties by id ascending
                keys = [(-float(l[t, e]), int(e)) for e in ids[t]]
                assert keys == sorted(keys)
                assert abs(w[t].sum() - 1.0) < 1e-15


def test_topk_all_equal_logits():
    ids, w = layer.top_k(np.zeros((2, 9), dtype=F32), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 2
    assert np.allclose(w, 0.25, rtol=0, atol=1e-16)


def test_topk_weights_equal_full_softmax_renormalised():
    g = np.random.default_rng(7)
    l = g.standard_normal((16, 40)).astype(F32) * 3
    ids, w = layer.top_k(l, 6)
    p = scipy.special.softmax(l.astype(np.float64), axis=1)
    sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
    ref = sel / sel.sum(axis=1, keepdims=True)
    assert np.allclose(w, ref, rtol=1e-13, atol=0)
    assert np.all(np.diff(w, axis=1) <= 0)


def test_topk_nan_is_an_error():
    l = np.zeros((1, 4), dtype=F32)
    l[0, 2] = np.nan
    with pytest.raises(layer.OracleError):
        layer.top_k(l, 2)


def test_router_logits_against_torch_float64():
    x = inputs.normal_bf16(inputs.rng(0, 1), (5, 96), 1.0)
    wr = inputs.normal_bf16(inputs.rng(0, 2), (11, 96), 0.02)
    bias = inputs.zipf_bias(0, 0, 11, 1.1)
    tx = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
    tw = torch.from_numpy(wr.view(np.int16)).view(torch.bfloat16).double()
    ref = (tx @ tw.T + torch.from_numpy(bias).double()).float().numpy()
    assert np.array_equal(layer.router_logits(x, wr, bias), ref)


# ---------------------------------------------------------------- groups / lookup

def _brute_groups(ids, E):
    T, k = ids.shape
    experts, off, tok, pos = [], [0], [], []
    for e in range(E):
        n = 0
        for t in range(T):
            for r in range(k):
                if ids[t, r] == e:
                    tok.append(t)
                    pos.append(t * k + r)
                    n += 1
        if n:
            experts.append(e)
            off.append(off[-1] + n)
    return experts, off, tok, pos


@pytest.mark.parametrize("T,E,k", [(1, 4, 1), (5, 12, 3), (9, 16, 2), (33, 40, 7), (3, 5, 5)])
def test_groups_brute_force(T, E, k):
    g = np.random.default_rng(T * 100 + E)
    ids = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    gr = layer.expert_groups(ids)
    experts, off, tok, pos = _brute_groups(ids, E)
    assert gr.experts.tolist() == experts
    assert gr.off.tolist() == off
    assert gr.ent_tok.tolist() == tok
    assert gr.ent_pos.tolist() == pos
    assert gr.off[-1] == T * k


def test_lookup_resident_staged_missing():
    E = 6
    resid = np.array([-1, -1, 0, -1, -1, -1,   3, -1, -1, 1, -1, -1], dtype=np.int32)
    stage = np.array([-1, -1, -1, -1, -1, -1,  -1, 2, -1, -1, -1, 0], dtype=np.int32)
    slot, src = layer.lookup(np.array([0, 1, 3, 5]), 1, E, resid, stage)
    assert slot.tolist() == [3, 2, 1, 0]
    assert src.tolist() == [0, 1, 0, 1]
    slot, src = layer.lookup(np.array([2, 4]), 1, E, resid, stage)
    assert slot.tolist() == [-1, -1] and src.tolist() == [-1, -1]


# ---------------------------------------------------------------- expert FFN / combine

def _torch_dense(ex, H, I):
    g, u, d = (torch.from_numpy(formats.dequantize(m, c)) for m, c in ((ex.gate, H), (ex.up, H), (ex.down, I)))
    return g, u, d


def test_lone_expert_is_dense_swiglu():
    """E = k = 1, no shared expert: the layer is one dense SwiGLU FFN with routing weight 1."""
    H, I = 64, 32
    ex = inputs.expert_weights(0, 0, 0, H, I)
    x = inputs.activations(0, 0, 7, H)
    wr = inputs.router_weights(0, 0, 1, H, 0.02)
    res = layer.moe_layer(x, wr, None, 1, lambda e: ex, H, I)
    g, u, d = _torch_dense(ex, H, I)
    tx = torch.from_numpy(formats.bf16_value(x))
    ref = (torch.nn.functional.silu(tx @ g.T) * (tx @ u.T)) @ d.T
    assert np.allclose(res.y, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert np.all(res.w == 1.0)


def test_shared_expert_only_is_gated_dense_ffn():
    """Routed experts with all-zero codes contribute nothing: y = sigmoid(x.w_sg) * S(x)."""
    H, I, Is, E, k = 64, 32, 80, 5, 2
    zero = inputs.expert_weights(0, 0, 0, H, I)
    zero.gate[:, : H // 2] = 0
    zero.up[:, : H // 2] = 0
    zero.down[:, : I // 2] = 0
    sh = inputs.shared_expert_weights(0, 0, H, Is)
    x = inputs.activations(0, 1, 6, H)
    wr = inputs.router_weights(0, 0, E, H, 0.02)
    wsg = inputs.shared_gate_weights(0, 0, H)
    res = layer.moe_layer(x, wr, None, k, lambda e: zero, H, I, shared=sh, I_shared=Is, w_shared_gate_bits=wsg)
    g, u, d = _torch_dense(sh, H, Is)
    tx = torch.from_numpy(formats.bf16_value(x))
    gate = torch.sigmoid(tx @ torch.from_numpy(formats.bf16_value(wsg)))
    ref = gate[:, None] * ((torch.nn.functional.silu(tx @ g.T) * (tx @ u.T)) @ d.T)
    assert np.allclose(res.y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_layer_equals_per_token_brute_force():
    """Grouped evaluation with scatter by position equals evaluating each token's
    chosen experts one by one."""
    w = inputs.small_workload(T=7, H=64, I=32, E=9, k=3, I_shared=32, zipf_s=0.7)
    s = w.shape
    li = inputs.layer_inputs(w)
    experts = {e: ex for e, ex in inputs.experts_of_layer(w, 0)}
    res = layer.moe_layer(li.x, li.w_router, li.bias, s.k, experts.__getitem__, s.H, s.I,
                          shared=li.shared, I_shared=s.I_shared, w_shared_gate_bits=li.w_shared_gate)
    x = formats.bf16_value(li.x)
    for t in range(w.T):
        acc = np.zeros(s.H)
        for r in range(s.k):
            e = int(res.ids[t, r])
            de = layer.dequantize_expert(experts[e], s.H, s.I)
            acc += res.w[t, r] * layer.swiglu_expert(x[t:t + 1], de)[0]
        ds = layer.dequantize_expert(li.shared, s.H, s.I_shared)
        gam = 1 / (1 + np.exp(-(x[t] @ formats.bf16_value(li.w_shared_gate))))
        acc += gam * layer.swiglu_expert(x[t:t + 1], ds)[0]
        assert np.allclose(res.y[t], acc, rtol=1e-12, atol=1e-12)


def test_combine_linear_in_down_scale():
    """Doubling every routed down matrix's global scale doubles the routed part only."""
    w = inputs.small_workload(T=4, H=64, I=32, E=6, k=2, I_shared=32)
    s = w.shape
    li = inputs.layer_inputs(w)
    base = {e: ex for e, ex in inputs.experts_of_layer(w, 0)}
    dbl = {e: inputs.Expert(ex.gate, ex.up, ex.down, (1.0, 1.0, 2.0)) for e, ex in base.items()}
    kw = dict(shared=li.shared, I_shared=s.I_shared, w_shared_gate_bits=li.w_shared_gate)
    r1 = layer.moe_layer(li.x, li.w_router, li.bias, s.k, base.__getitem__, s.H, s.I, **kw)
    r2 = layer.moe_layer(li.x, li.w_router, li.bias, s.k, dbl.__getitem__, s.H, s.I, **kw)
    shared_part = r1.gamma[:, None] * r1.shared
    assert np.allclose(r2.y - shared_part, 2 * (r1.y - shared_part), rtol=1e-12, atol=1e-12)


def test_rmsnorm_against_torch():
    x = np.random.default_rng(0).standard_normal((5, 33))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (33,), eps=1e-6).numpy()
    assert np.allclose(layer.rmsnorm(x), ref, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- policy

def test_swap_worked_example():
    g = {r[0]: float(r[1]) for r in read_golden("swap_example.txt")}
    E = 4
    heat = np.zeros(E, dtype=F32)
    heat[0] = g["heat_A_nonresident"]
    heat[1] = g["heat_B_resident"]
    resid = np.array([-1, 5, -1, -1], dtype=np.int32)
    plan = policy.plan_round(heat, resid, 1, E, threshold=g["threshold"], max_swaps=int(g["max_swaps"]),
                             factor=g["decay"])
    assert len(plan) == int(g["swap"])
    assert (plan[0].hot_expert, plan[0].cold_expert, plan[0].slot) == (0, 1, 5)
    assert plan[0].diff == g["difference"]
    # after the round every heat is scaled by 0.7: 10 -> 7, 8 -> 5.6 (nearest fp32)
    assert heat[0] == F32(7.0) and heat[1] == F32(5.6)
    policy.apply_swaps(resid, plan, E)
    assert resid.tolist() == [5, -1, -1, -1]


def test_threshold_is_inclusive():
    heat = np.array([10.0, 8.5, 0, 0], dtype=F32)    # fl32(10 - 8.5) == 1.5 exactly
    assert len(policy.plan_swaps(heat, np.array([-1, 0, -1, -1]), 1, 4)) == 1
    heat = np.array([10.0, np.nextafter(F32(8.5), F32(9)), 0, 0], dtype=F32)
    assert len(policy.plan_swaps(heat, np.array([-1, 0, -1, -1]), 1, 4)) == 0


def test_cap_keeps_largest_differences():
    L, E = 4, 64
    g = np.random.default_rng(1)
    heat = np.zeros(L * E, dtype=F32)
    resid = np.full(L * E, -1, dtype=np.int32)
    slot = 0
    for l in range(L):
        for e in range(25):                      # 25 non-resident hot experts per layer
            heat[l * E + e] = F32(2 + g.integers(0, 1000))
        for e in range(32, 57):                  # 25 resident cold experts at heat 0
            resid[l * E + e] = slot
            slot += 1
    plan = policy.plan_swaps(heat, resid, L, E)
    assert len(plan) == 96                       # 100 candidates, capped
    all_d = sorted((float(heat[l * E + e]) for l in range(L) for e in range(25)), reverse=True)
    assert [p.diff for p in plan] == all_d[:96]
    assert len({(p.layer, p.slot) for p in plan}) == 96


def test_pairs_stay_within_layer_and_decay_only_round():
    heat = np.array([0, 0, 5, 0,   9, 0, 0, 0], dtype=F32)
    resid = np.array([0, 1, 2, 3,  -1, -1, -1, -1], dtype=np.int32)
    # layer 1 has a hot expert but no resident partner; layer 0 has no non-resident expert
    assert policy.plan_round(heat, resid, 2, 4) == []
    assert heat.tolist() == [0, 0, F32(5) * F32(0.7), 0, F32(9) * F32(0.7), 0, 0, 0]


def test_pairing_hot_desc_with_cold_asc():
    heat = np.array([3, 9, 6, 1, 4, 2], dtype=F32)
    resid = np.array([-1, -1, -1, 10, 11, 12], dtype=np.int32)
    plan = policy.plan_swaps(heat, resid, 1, 6)
    # hot by heat desc: 1(9), 2(6), 0(3); cold by heat asc: 3(1), 5(2), 4(4)
    assert [(p.hot_expert, p.cold_expert, p.diff) for p in plan] == [(1, 3, 8.0), (2, 5, 4.0)]


def test_heat_counts_each_selection_once():
    heat = np.zeros(2 * 5, dtype=F32)
    ids = np.array([[0, 3], [3, 4], [3, 0]])
    policy.heat_update(heat, ids, 1, 5)
    assert heat.tolist() == [0] * 5 + [2, 0, 0, 3, 1]


# ---------------------------------------------------------------- the pages' side arithmetic

def test_initial_share_matches_log():
    g = {r[0]: float(r[1]) for r in read_golden("share.txt")}
    s = side.initial_share(g["probe_gbs"], g["base"], g["reference_gbs"])
    assert abs(s - 0.49225) < 1e-12 and round(s, 2) == g["initial_share_printed"]


def test_share_update_printed_value_is_unpinned():
    """Parity unpinned: the printed rule with the printed rates gives 0.62, the log says 0.60."""
    g = {r[0]: float(r[1]) for r in read_golden("share.txt")}
    s = side.candidate_share(g["probe_gbs"], g["cpu_equiv_gbs"], g["coef"])
    assert round(s, 2) == 0.62 and round(s, 2) != g["updated_share_printed"]


def test_qstar_ratios_match_table():
    for name, bp, bh, printed in read_golden("qstar_table.txt"):
        bp, bh, printed = float(bp), float(bh), float(printed)
        assert round(side.q_star_fraction(bp, bh), 2) == printed, name
        # the balance point: fill time == cpu time at q = m*B_P/B_H (equation (2))
        m, S = 1000, 1.0
        q = m * bp / bh
        assert abs(q * S / bp - (m - q) * S / side.residual_bandwidth(bh, bp)) < 1e-9


def test_qstar_rounding_and_minimum_fill():
    assert side.q_star(0, 10, 20) == 0
    assert side.q_star(1, 1, 100) == 1
    assert side.q_star(10, 25.3, 56.7) == 4


def test_hit_rate_arithmetic():
    g = {r[0]: float(r[1]) for r in read_golden("hit_rate.txt")}
    assert round(100 * g["hits"] / g["lookups"], 1) == g["printed_percent"]


# ---------------------------------------------------------------- tail skip (Strata page, "跳过尾部专家")

def test_tail_skip_rules_worked_by_hand():
    """Threshold 7 on zero-based ranks, k = 10.  Expert 7: ranks {7, 9}, resident -> kept.
    Expert 8: rank {8}, staged -> dropped.  Expert 9: ranks {9, 7}, missing -> dropped
    (and not an error).  Expert 3: ranks {3, 8}, staged -> kept (one token ranks it in
    the top seven).  Everything else ranks below 7 somewhere or is resident."""
    E, k = 20, 10
    ids = np.array([[0, 1, 2, 3, 4, 5, 6, 7, 8, 9],
                    [10, 11, 12, 13, 14, 15, 16, 9, 3, 7]], dtype=np.int32)
    resid = np.full(E, -1, dtype=np.int32)
    stage = np.full(E, -1, dtype=np.int32)
    for e in (0, 1, 2, 4, 5, 6, 7, 10, 11, 12, 13, 14, 15, 16):
        resid[e] = e
    stage[3], stage[8] = 0, 1           # expert 9: neither table
    g = layer.expert_groups(ids)
    slot, src = layer.lookup(g.experts, 0, E, resid, stage)
    drop = layer.tail_skip_mask(g, src, k, 7)
    assert sorted(int(e) for e in g.experts[drop]) == [8, 9]
    assert not layer.tail_skip_mask(g, src, k, 0).any()
    assert not layer.tail_skip_mask(g, src, k, k).any()
    # threshold 9: only an expert every chooser ranks last -- none here (9 is 7th for token 1)
    assert not layer.tail_skip_mask(g, src, k, 9).any()
    assert sorted(int(e) for e in g.experts[layer.tail_skip_mask(g, src, k, 8)]) == [8]


def _skip_workload():
    w = inputs.small_workload(T=3, H=64, I=32, E=24, k=6, I_shared=32, zipf_s=0.5)
    s = w.shape
    li = inputs.layer_inputs(w)
    experts = {e: ex for e, ex in inputs.experts_of_layer(w, 0)}
    # every odd expert staged, every even one resident
    resid = np.array([e if e % 2 == 0 else -1 for e in range(s.E)], dtype=np.int32)
    stage = np.array([-1 if e % 2 == 0 else e for e in range(s.E)], dtype=np.int32)
    return w, s, li, experts, resid, stage


def test_tail_skip_output_moves_by_minus_skipped_terms():
    """The page's identity: y_skip - y_full = -sum over skipped (t, r) of w[t,r] * E_ids[t,r](x_t),
    with the skipped terms evaluated token by token (no grouping, no scatter)."""
    w, s, li, experts, resid, stage = _skip_workload()
    kw = dict(resid=resid, stage=stage, shared=li.shared, I_shared=s.I_shared,
              w_shared_gate_bits=li.w_shared_gate)
    full = layer.moe_layer(li.x, li.w_router, li.bias, s.k, experts.__getitem__, s.H, s.I, **kw)
    R = 3
    skip = layer.moe_layer(li.x, li.w_router, li.bias, s.k, experts.__getitem__, s.H, s.I, tail_skip=R, **kw)
    assert np.array_equal(skip.ids, full.ids) and np.array_equal(skip.w, full.w)   # no renormalisation
    # the skipped experts by the rule, straight from the ids: odd (staged) and never ranked below R
    chosen = {}
    for t in range(w.T):
        for r in range(s.k):
            chosen.setdefault(int(full.ids[t, r]), []).append(r)
    skipped = {e for e, rs in chosen.items() if e % 2 == 1 and min(rs) >= R}
    assert skipped, "the seeded window should skip at least one expert"
    assert {int(e) for e, sr in zip(skip.groups.experts, skip.src) if sr == layer.SRC_SKIPPED} == skipped
    x = formats.bf16_value(li.x)
    for t in range(w.T):
        delta = np.zeros(s.H)
        for r in range(s.k):
            e = int(full.ids[t, r])
            if e in skipped:
                de = layer.dequantize_expert(experts[e], s.H, s.I)
                delta -= full.w[t, r] * layer.swiglu_expert(x[t:t + 1], de)[0]
        assert np.allclose(skip.y[t] - full.y[t], delta, rtol=1e-12, atol=1e-12)


def test_tail_skip_missing_expert_is_dropped_not_an_error():
    """A missing expert is fine when the rule drops it, an error when a token ranks it high."""
    w, s, li, experts, resid, stage = _skip_workload()
    full = layer.moe_layer(li.x, li.w_router, li.bias, s.k, experts.__getitem__, s.H, s.I, resid=resid, stage=stage)
    R = 3
    ranks = {}
    for t in range(w.T):
        for r in range(s.k):
            ranks.setdefault(int(full.ids[t, r]), []).append(r)
    low = [e for e, rs in ranks.items() if e % 2 == 1 and min(rs) >= R]
    high = [e for e, rs in ranks.items() if e % 2 == 1 and min(rs) < R]
    assert low and high
    st2 = stage.copy()
    st2[low[0]] = -1                      # now missing, but dropped by the rule
    res = layer.moe_layer(li.x, li.w_router, li.bias, s.k, experts.__getitem__, s.H, s.I, resid=resid, stage=st2,
                          tail_skip=R)
    g = int(np.nonzero(res.groups.experts == low[0])[0][0])
    assert res.src[g] == layer.SRC_SKIPPED and res.slot[g] == layer.MISSING
    st3 = stage.copy()
    st3[high[0]] = -1                     # missing and kept: the layer cannot run
    with pytest.raises(layer.OracleError):
        layer.moe_layer(li.x, li.w_router, li.bias, s.k, experts.__getitem__, s.H, s.I, resid=resid, stage=st3,
                        tail_skip=R)


def test_tail_skip_all_resident_changes_nothing():
    w, s, li, experts, resid, stage = _skip_workload()
    a = layer.moe_layer(li.x, li.w_router, li.bias, s.k, experts.__getitem__, s.H, s.I)
    b = layer.moe_layer(li.x, li.w_router, li.bias, s.k, experts.__getitem__, s.H, s.I, tail_skip=1)
    assert np.array_equal(a.y, b.y) and (b.src == layer.SRC_RESIDENT).all()


# ---------------------------------------------------------------- global LRU (FreeToken notes, 3.3 and 4)

def _lru_run(calls, nslots, K, E, resid=None, owner=None):
    """Drive the oracle LRU through calls of (layer, [experts]); returns the hit/miss flags per
    call and the final tables.  The lookup is the oracle's (resident or not)."""
    from oracle import lru
    L = 1 + max(l for l, _ in calls)
    resid = np.full(L * E, -1, dtype=np.int32) if resid is None else resid
    owner = np.full(nslots, -1, dtype=np.int32) if owner is None else owner
    st = lru.new_state(nslots)
    flags = []
    for layer, exps in calls:
        exps = sorted(set(exps))
        slot, src = layer_mod.lookup(np.array(exps), layer, E, resid)
        src = np.where(src == layer_mod.SRC_MISSING, layer_mod.SRC_STAGED, src)   # misses come from staging
        flags.append([bool(s == layer_mod.SRC_RESIDENT) for s in src])
        plan = lru.plan_call(st, owner, layer, exps, src, slot, K, E)
        lru.apply(resid, owner, plan, E)
    return flags, resid, owner


layer_mod = layer


def test_lru_single_accesses_match_textbook_lru():
    """One expert per call: the hit sequence is that of a textbook LRU of the same capacity
    (an ordered dict: a hit moves the key to the back, a miss evicts the front when full)."""
    import collections
    g = np.random.default_rng(3)
    E, L, C = 20, 2, 6
    calls = [(int(g.integers(L)), [int(min(E - 1, g.zipf(1.3) - 1))]) for _ in range(400)]
    flags, _, _ = _lru_run(calls, C, K=4, E=E)
    od = collections.OrderedDict()
    ref = []
    for layer, (e,) in calls:
        key = (layer, e)
        if key in od:
            od.move_to_end(key)
            ref.append(True)
        else:
            ref.append(False)
            if len(od) == C:
                od.popitem(last=False)
            od[key] = True
    assert [f[0] for f in flags] == ref


def test_lru_batch_worked_by_hand():
    """Three slots, one layer, E = 8.  Call 1 {1,2}: both miss, fill empty slots 0, 1.
    Call 2 {2,3}: 2 hits; 3 fills empty slot 2.  Call 3 {4,5}: the victims are slots the call
    did not use, oldest first: slot 0 (expert 1, last used in call 1) then slot 1 (expert 2,
    call 2); 4 takes slot 0, 5 takes slot 1.  Call 4 {1}: slot 2 (expert 3, call 2) is the
    oldest; 1 takes it."""
    flags, resid, owner = _lru_run([(0, [1, 2]), (0, [2, 3]), (0, [4, 5]), (0, [1])], 3, K=4, E=8)
    assert flags == [[False, False], [True, False], [False, False], [False]]
    assert owner.tolist() == [4, 5, 1]
    assert [int(resid[e]) for e in range(8)] == [-1, 2, -1, -1, 0, 1, -1, -1]


def test_lru_admits_at_most_k_and_keeps_the_call_hits():
    """Five misses with K = 2: only the first two (ascending expert id) are admitted; a
    slot the call hit is never a victim."""
    from oracle import lru
    E, nslots = 16, 4
    resid = np.full(E, -1, dtype=np.int32)
    owner = np.array([0, 1, 2, 3], dtype=np.int32)
    resid[:4] = [0, 1, 2, 3]
    st = lru.new_state(nslots)
    exps = [0, 9, 10, 11, 12, 13]
    slot, src = layer_mod.lookup(np.array(exps), 0, E, resid)
    src = np.where(src == layer_mod.SRC_MISSING, layer_mod.SRC_STAGED, src)
    plan = lru.plan_call(st, owner, 0, exps, src, slot, 2, E)
    assert [(p.hot_expert, p.cold_flat, p.slot) for p in plan] == [(9, 1, 1), (10, 2, 2)]
    assert st.tick.tolist() == [1, 1, 1, 0]
