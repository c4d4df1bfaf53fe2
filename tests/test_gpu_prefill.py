"""GPU parity of the prefill path (tcgen05 grouped GEMMs) against the oracle, through the C ABI.

Every token is compared, at small ragged shapes and at the full-size chunks,
routed on the GPU's fp32 logits; those logits are held against the oracle's
within the fp32 accumulation bound."""
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


def run_prefill(st, x_bits, T, bf16_out=False):
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    y = torch.zeros((T, st.H), dtype=torch.int16 if bf16_out else torch.float32, device="cuda")
    st.forward(0, x, y, T, y_is_fp32=not bf16_out, mode=moe.MOE_MODE_PREFILL)
    rc = moe.moe_sync_status(st.ws)
    assert rc == moe.MOE_OK, moe.strerror(rc)
    return U.y_to_numpy(y, bf16_out)


def check_router(st, x_bits, logits, ids, tokens):
    """The prefill router GEMM's logits against the oracle's fp64 logits, within the fp32
    accumulation bound; ids chosen on the GPU logits against the oracle's top-k of the
    oracle's own logits, where they may differ only at a near-tie within that bound."""
    li = st.layers[0].host
    ref_logits = olayer.router_logits(x_bits[tokens], li.w_router, li.bias)
    bound = U.logits_bound(x_bits[tokens], li.w_router, li.bias)
    err = np.abs(logits[tokens].astype(np.float64) - ref_logits)
    assert np.all(err <= bound), f"router logits: {int((err > bound).sum())} beyond the bound, max {err.max():.3g}"
    o_ids, _ = olayer.top_k(ref_logits, st.k)
    for i in np.flatnonzero((o_ids != ids[tokens]).any(axis=1)):
        srt = np.sort(ref_logits[i].astype(np.float64))[::-1]
        gaps = np.abs(np.diff(srt[: st.k + 1]))
        assert gaps.min() <= 2 * bound[i].max(), tokens[i]


def check_tokens(st, x_bits, y, tokens, tail_skip=0):
    logits, ids, _ = st.ws.routing(x_bits.shape[0])
    logits = logits.cpu().numpy()
    ids = ids.cpu().numpy()
    li = st.layers[0].host
    check_router(st, x_bits, logits, ids, tokens)
    # routing on the GPU's own logits matches the oracle's top-k bit for bit
    ref_ids, _ = olayer.top_k(logits[tokens], st.k)
    assert np.array_equal(ids[tokens], ref_ids)
    ref = olayer.moe_layer(x_bits[tokens], li.w_router, li.bias, st.k, lambda e: st.expert_host(0, e), st.H, st.I,
                           resid=st.resid_table(), stage=st.stage_table(), shared=li.shared, I_shared=st.I_shared,
                           w_shared_gate_bits=li.w_shared_gate, logits=logits[tokens], tail_skip=tail_skip)
    return ref


@pytest.mark.parametrize("T,H,I_,E,k,Is,zipf", [
    (300, 256, 128, 16, 2, 128, 0.8),   # ragged token count, groups of many sizes
    (160, 2048, 512, 64, 4, 512, 1.1),  # the chunk's row widths, router K = 2048
    (200, 512, 128, 300, 5, 128, 0.0),  # router N of 300 experts (a ragged last N tile)
    (1024, 128, 64, 8, 2, 64, 0.0),     # narrowest rows; groups above 256 tokens (several N tiles)
    (129, 512, 256, 40, 7, 0, 1.2),     # no shared expert, small groups
])
def test_prefill_small_shapes_full(T, H, I_, E, k, Is, zipf):
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=H, I=I_, E=E, k=k, I_shared=Is, zipf_s=zipf, resident_frac=0.5, seed=T + E)
    st = ModelState(w)
    x_bits = I.activations(w.seed, 0, T, H)
    y = run_prefill(st, x_bits, T)
    ref = check_tokens(st, x_bits, y, np.arange(T))
    U.assert_close_layer(y, ref.y)
    yb = run_prefill(st, x_bits, T, bf16_out=True)
    U.assert_close_layer(yb, ref.y, bf16_out=True)


@pytest.mark.parametrize("T,H,I_,E,k,Is,zipf,R", [
    (300, 256, 128, 64, 4, 128, 1.2, 2),    # one-CTA grouping
    (1100, 128, 64, 128, 4, 64, 1.5, 2),    # the multi-CTA grouping passes (T*k > 4096)
])
def test_prefill_tail_skip_full(T, H, I_, E, k, Is, zipf, R):
    """Tail skip (Strata page, "跳过尾部专家") on the prefill path: the dropped groups load no
    weights and add nothing; y against the oracle's layer with the same drops, whole window."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=H, I=I_, E=E, k=k, I_shared=Is, zipf_s=zipf, resident_frac=0.5, seed=T + E)
    st = ModelState(w)
    st.ws.set_tail_skip(R)
    x_bits = I.activations(w.seed, 0, T, H)
    y = run_prefill(st, x_bits, T)
    ref = check_tokens(st, x_bits, y, np.arange(T), tail_skip=R)
    assert (ref.src == olayer.SRC_SKIPPED).any()
    _, _, slot, src, _, _ = st.ws.groups(T)
    assert np.array_equal(src, ref.src) and np.array_equal(slot, ref.slot)
    U.assert_close_layer(y, ref.y)


def test_prefill_chunk_t8192_h2048_e512_k10_all_tokens():
    """The 8192-token chunk: every token of y against the oracle (512 groups of about 160
    tokens, so every work item, tile and split point of the persistent GEMMs is compared)."""
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["prefill_t8192_h2048_e512_k10"]
    st = ModelState(w)
    x_bits = I.activations(w.seed, 0, w.T, w.shape.H)
    y = run_prefill(st, x_bits, w.T)
    tokens = np.arange(w.T)
    ref = check_tokens(st, x_bits, y, tokens)
    U.assert_close_layer(y, ref.y, what="y, all tokens")
    # decode and prefill paths agree on a window both can run
    yd = torch.zeros((64, w.shape.H), dtype=torch.float32, device="cuda")
    st.forward(0, torch.from_numpy(x_bits[:64].view(np.int16)).cuda(), yd, 64, mode=moe.MOE_MODE_DECODE)
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK
    yd = yd.cpu().numpy().astype(np.float64)
    ref64 = check_tokens(st, x_bits[:64], yd, np.arange(64))
    U.assert_close_layer(yd, ref64.y, what="decode window")


def test_prefill_large_expert_layer_all_tokens():
    """One layer of the 4096-hidden, 256-expert top-6 model (I = I_shared = 2048), 4096-token
    chunk, every token against the oracle."""
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["large_h4096_e256_k6"]
    st = ModelState(w, layers=1)
    x_bits = I.activations(w.seed, 0, w.T, w.shape.H)
    y = run_prefill(st, x_bits, w.T)
    ref = check_tokens(st, x_bits, y, np.arange(w.T))
    U.assert_close_layer(y, ref.y, what="y, all tokens")


@pytest.mark.parametrize("T", [300, 1100])   # one-CTA grouping; the multi-CTA grouping passes
def test_prefill_edge_format(T):
    """Zero, subnormal and 448 block scales and global scales 0.375 / 2.0 / 1.25 (gate, up,
    down) through the prefill GEMMs, resident and streamed, every token."""
    from serving_router_top_gb300.model import ModelState
    w = I.edge_workload(T=T, resident_frac=0.5)
    st = ModelState(w)
    x_bits = I.activations(w.seed, 0, T, w.shape.H)
    y = run_prefill(st, x_bits, T)
    ref = check_tokens(st, x_bits, y, np.arange(T))
    U.assert_close_layer(y, ref.y)
    st2 = ModelState(w, stage_rest=False, nstaging=16)
    y2 = run_streamed(st2, x_bits, T, 8)
    ref2 = check_tokens_streamed(st2, x_bits, np.arange(T))
    U.assert_close_layer(y2, ref2.y, what="streamed y")


def run_streamed(st, x_bits, T, U_, bf16_out=False, buffers=2):
    x = torch.from_numpy(x_bits.view(np.int16)).cuda()
    y = torch.zeros((T, st.H), dtype=torch.int16 if bf16_out else torch.float32, device="cuda")
    st.forward_streamed(0, x, y, T, U_, y_is_fp32=not bf16_out, buffers=buffers)
    torch.cuda.synchronize()
    rc = moe.moe_sync_status(st.ws)
    assert rc == moe.MOE_OK, moe.strerror(rc)
    return U.y_to_numpy(y, bf16_out)


def check_tokens_streamed(st, x_bits, tokens):
    """Reference for a streamed call: every expert of the layer is available (no residency tables)."""
    logits, ids, _ = st.ws.routing(x_bits.shape[0])
    logits = logits.cpu().numpy()
    ids = ids.cpu().numpy()
    li = st.layers[0].host
    check_router(st, x_bits, logits, ids, tokens)
    ref_ids, _ = olayer.top_k(logits[tokens], st.k)
    assert np.array_equal(ids[tokens], ref_ids)
    return olayer.moe_layer(x_bits[tokens], li.w_router, li.bias, st.k, lambda e: st.expert_host(0, e), st.H, st.I,
                            shared=li.shared, I_shared=st.I_shared, w_shared_gate_bits=li.w_shared_gate,
                            logits=logits[tokens])


@pytest.mark.parametrize("T,H,I_,E,k,Is,U_", [
    (300, 256, 128, 16, 2, 128, 3),   # six units, the last of one expert; each staging half reused three times
    (129, 512, 256, 40, 7, 0, 8),     # no shared expert
    (1024, 128, 64, 8, 2, 64, 8),     # one unit holding every expert
])
def test_prefill_streamed_small_shapes_full(T, H, I_, E, k, Is, U_):
    """Experts streamed from the backing pool through two halves of the staging pool (copy
    stream: copied; compute stream: used) give the layer with every expert available, although
    half of them are neither resident nor staged in the cache's tables."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=H, I=I_, E=E, k=k, I_shared=Is, zipf_s=0.8, resident_frac=0.5, seed=T + E)
    st = ModelState(w, stage_rest=False, nstaging=2 * U_)
    x_bits = I.activations(w.seed, 1, T, H)
    y = run_streamed(st, x_bits, T, U_)
    ref = check_tokens_streamed(st, x_bits, np.arange(T))
    U.assert_close_layer(y, ref.y)
    yb = run_streamed(st, x_bits, T, U_, bf16_out=True)
    U.assert_close_layer(yb, ref.y, bf16_out=True)
    y1 = run_streamed(st, x_bits, T, U_, buffers=1)   # one staging half: each copy waits for the GEMMs before it
    U.assert_close_layer(y1, ref.y)


def test_prefill_streamed_chunk_t8192_all_tokens():
    """The 8192-token chunk with all 512 experts streamed in eight units of 64 (113 MB each),
    every token against the oracle."""
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["prefill_t8192_h2048_e512_k10"]
    st = ModelState(w, resident=np.zeros((1, w.shape.E), dtype=bool), stage_rest=False, nslots=1, nstaging=128)
    x_bits = I.activations(w.seed, 2, w.T, w.shape.H)
    y = run_streamed(st, x_bits, w.T, 64)
    ref = check_tokens_streamed(st, x_bits, np.arange(w.T))
    U.assert_close_layer(y, ref.y, what="y, all tokens")


def test_prefill_streamed_rejects_bad_units():
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=64, H=128, I=64, E=8, k=2, I_shared=0, zipf_s=0.0, resident_frac=1.0, seed=3)
    st = ModelState(w, nstaging=4)
    x = torch.zeros((64, 128), dtype=torch.int16, device="cuda")
    y = torch.zeros((64, 128), dtype=torch.float32, device="cuda")
    for bad in (0, 3):  # 2*U must fit the four staging slots
        with pytest.raises(moe.MoeError):
            st.forward_streamed(0, x, y, 64, bad)
    for bad_buffers in (0, 3):
        with pytest.raises(moe.MoeError):
            st.forward_streamed(0, x, y, 64, 2, buffers=bad_buffers)
    with pytest.raises(moe.MoeError):  # one buffer of 5 does not fit four slots either
        st.forward_streamed(0, x, y, 64, 5, buffers=1)


def _stack_ref_gpu(st, x_res0, T, L):
    """The same layers through moe_layer_forward in prefill mode, experts from the cache's
    slots; every layer's input rows, logits and output are kept for teacher-forced checks."""
    x_res = x_res0.clone()
    xn = torch.zeros((T, st.H), dtype=torch.int16, device="cuda")
    y = torch.zeros((T, st.H), dtype=torch.int16, device="cuda")
    prev, seen = None, []
    for l in range(L):
        moe.moe_residual_rmsnorm(x_res, prev, xn, T, st.H)
        st.forward(l, xn, y, T, y_is_fp32=False, mode=moe.MOE_MODE_PREFILL)
        torch.cuda.synchronize()
        seen.append(dict(xn=xn.cpu().numpy().view(np.uint16).copy(), y=y.cpu().numpy().view(np.uint16).copy(),
                         logits=st.ws.routing(T)[0].cpu().numpy().copy()))
        prev = y
    moe.moe_residual_rmsnorm(x_res, prev, xn, T, st.H)
    torch.cuda.synchronize()
    return x_res, seen


@pytest.mark.parametrize("backing_on_device", [True, False])
def test_layers_streamed_double_buffer(backing_on_device):
    """Three layers of a prefill chunk with each layer's experts streamed into one half of the
    staging pool one layer ahead (two buffers), and with the second buffer off (each copy
    waits for the previous layer), against the same layers run one call each from resident
    slots -- whose every layer is held against the oracle on that layer's own input rows and
    logits.  The two runs may route a token differently where a layer's bf16 input differs in
    its last bit at a near-tie (the fp32 atomic adds of the prefill combine vary in order), so
    all but at most 2% of the token rows must agree within the layer tolerance."""
    from oracle import formats
    from serving_router_top_gb300.model import ModelState
    L, T = 3, 300
    w = I.small_workload(T=T, H=256, I=128, E=16, k=2, I_shared=128, zipf_s=0.0, resident_frac=1.0, seed=31,
                         layers=L)
    st = ModelState(w, nstaging=32, backing_on_device=backing_on_device, stage_rest=False)
    x0 = torch.from_numpy(formats.bf16_value(I.activations(w.seed, 5, T, st.H)).astype(np.float32)).cuda()
    ref, seen = _stack_ref_gpu(st, x0, T, L)
    for l, d in enumerate(seen):
        li = st.layers[l].host
        o = olayer.moe_layer(d["xn"], li.w_router, li.bias, st.k, lambda e, l=l: st.expert_host(l, e), st.H, st.I,
                             layer=l, shared=li.shared, I_shared=st.I_shared, w_shared_gate_bits=li.w_shared_gate,
                             logits=d["logits"])
        U.assert_close_layer(formats.bf16_value(d["y"]), o.y, bf16_out=True, what=f"layer {l}")
    copy = torch.cuda.Stream()
    r = ref.cpu().numpy().astype(np.float64)
    tol = U.TOL_REL * np.sqrt(np.mean(r * r)) + U.TOL_ABS
    for buffers in (2, 1):
        x_res = x0.clone()
        xn = torch.zeros((T, st.H), dtype=torch.int16, device="cuda")
        y = torch.zeros((T, st.H), dtype=torch.int16, device="cuda")
        moe.moe_layers_forward_streamed([st.layers[l].desc for l in range(L)], x_res, xn, y, T, st.cache, st.ws,
                                        buffers=buffers, copy_stream=copy)
        torch.cuda.synchronize()
        assert moe.moe_sync_status(st.ws) == moe.MOE_OK
        rows_ok = (np.abs(x_res.cpu().numpy() - r) <= tol).all(axis=1)
        assert rows_ok.mean() >= 0.98, (buffers, int((~rows_ok).sum()))
