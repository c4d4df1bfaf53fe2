"""GPU parity of the single-kernel decode forward (router -> top-k -> groups -> lookup ->
gate/up -> down -> combine in one cooperative launch) against the oracle, through the C ABI,
and its agreement with the chain of kernels on the same windows."""
import numpy as np
import pytest
import torch

from oracle import layer as olayer
from oracle import policy as opol
from serving_router_top_gb300 import inputs as I
from serving_router_top_gb300 import moe
from tests import gpu_util as U
from tests.test_gpu_layer import check_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def ran_fused(st, T, x_bits=None):
    """One forward with per-kernel events: the single kernel ran (and nothing else did)."""
    x_bits = I.activations(st.w.seed, 99, T, st.H) if x_bits is None else x_bits
    st.ws.set_profiling(True)
    run_layer(st, x_bits, T)
    names = [n for n, _ in st.ws.kernel_times()]
    st.ws.set_profiling(False)
    return names == ["decode_fused"]


@pytest.mark.parametrize("T,H,I_,E,k,Is,frac,zipf", [
    (4, 2048, 512, 512, 10, 512, 0.5, 1.1),    # the decode verify window's shapes
    (1, 2048, 512, 512, 10, 512, 0.5, 1.1),
    (8, 2048, 512, 512, 10, 512, 0.3, 1.1),    # the widest window, 70% of the groups staged
    (3, 512, 256, 40, 7, 256, 0.5, 0.8),       # narrowest rows: one router slice, one down chunk
    (4, 1024, 1024, 1000, 6, 0, 1.0, 0.0),     # no shared expert, E not a power of two, I of four chunks
    (7, 1024, 256, 64, 9, 256, 0.25, 0.5),     # ragged token count, 9 of 64 experts per token
    (2, 512, 512, 1, 1, 512, 1.0, 0.0),        # a single routed expert (weight 1) and the shared one
    (8, 2048, 256, 256, 32, 256, 0.5, 0.6),    # 256 selections, many shared groups
    (16, 2048, 512, 512, 10, 512, 0.5, 1.1),   # two 8-row tiles of B per unit, the shared expert on both
    (12, 1024, 256, 64, 9, 256, 0.25, 0.5),    # ragged second tile, groups above 8 tokens
    (9, 512, 512, 40, 7, 0, 1.0, 0.0),         # one token past a tile, no shared expert
    (13, 2048, 1024, 200, 16, 1024, 0.5, 0.8),  # 208 selections, I of four chunks, second tile
])
def test_fused_decode_layer(T, H, I_, E, k, Is, frac, zipf):
    """Logits within the fp32 bound of the oracle's, ids bit-exact on the same logits (near-ties
    only on the oracle's own), groups, slots and sources bit-exact, y within tolerance in fp32
    and bf16 output; and the call ran as the single kernel."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=T, H=H, I=I_, E=E, k=k, I_shared=Is, zipf_s=zipf, resident_frac=frac, seed=3 * T + E)
    st = ModelState(w)
    assert ran_fused(st, T)
    check_layer(st, T)
    check_layer(st, max(1, T // 2), step=1, bf16_out=True)


def test_fused_decode_window_all_steps_and_stats():
    """The decode verify window: several windows, statistics and the fused heat update bit-exact
    against the oracle's heat update on the kernel's own ids."""
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["decode_t4_h2048_e512_k10"]
    st = ModelState(w)
    st.ws.set_fused_heat(True)
    heat = np.zeros(w.shape.E, dtype=np.float32)
    groups = 0
    for step in range(4):
        _, ref = check_layer(st, w.T, step=step)
        opol.heat_update(heat, ref.ids, 0, w.shape.E)
        groups += ref.groups.num_groups
    assert np.array_equal(st.cache.tables()[2].cpu().numpy()[:w.shape.E], heat)
    stats = st.cache.stats()
    assert stats[0, 0] == groups and stats[0, 0] == stats[0, 1] + stats[0, 2] and stats[0, 3] == 0
    assert ran_fused(st, w.T)


def test_fused_and_chain_agree():
    """The same windows through both decode paths: each within tolerance of the oracle, and the
    two outputs within the same tolerance of each other."""
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["decode_t4_h2048_e512_k10"]
    st = ModelState(w)
    for step in range(3):
        x_bits = I.activations(w.seed, 40 + step, w.T, st.H)
        st.ws.set_decode_path(moe.MOE_DECODE_CHAIN)
        y_chain = run_layer(st, x_bits, w.T)
        st.ws.set_decode_path(moe.MOE_DECODE_FUSED)
        y_fused = run_layer(st, x_bits, w.T)
        U.assert_close_layer(y_fused, y_chain, what="fused vs chain")


def test_fused_decode_edge_format():
    """Zero, subnormal and 448 block scales and global scales 0.375 / 2.0 / 1.25 on the single kernel."""
    from serving_router_top_gb300.model import ModelState
    w = I.edge_workload(T=6, H=512, I=256, E=24, k=4, I_shared=256)
    st = ModelState(w)
    assert ran_fused(st, 6)
    check_layer(st, 6)
    check_layer(st, 6, bf16_out=True, step=2)


def test_fused_decode_tail_skip():
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["decode_t4_h2048_e512_k10"]
    st = ModelState(w)
    st.ws.set_tail_skip(7)
    n_skip = 0
    for step in range(4):
        _, ref = check_layer(st, w.T, step=step, tail_skip=7)
        n_skip += int((ref.src == olayer.SRC_SKIPPED).sum())
    assert n_skip > 0
    assert st.cache.stats()[0, 4] == n_skip


def test_fused_decode_missing_expert():
    """An expert neither resident nor staged: MOE_EMISSING, recorded once, then cleared."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=6, H=512, I=256, E=12, k=3, I_shared=0, resident_frac=0.25, seed=3)
    st = ModelState(w, stage_rest=False)
    x = torch.from_numpy(I.activations(w.seed, 0, 6, 512).view(np.int16)).cuda()
    y = torch.zeros((6, 512), dtype=torch.float32, device="cuda")
    st.forward(0, x, y, 6)
    assert moe.moe_sync_status(st.ws) == moe.MOE_EMISSING
    assert moe.moe_sync_status(st.ws) == moe.MOE_OK


def test_fused_decode_bounded_wait_expires_and_recovers():
    """Fault injection on the host side of a flag: the grid barrier waits for one arrival beyond
    the grid, which nothing makes; after the 20 ms bound the kernel records MOE_ETIMEOUT and
    returns, the context stays usable, and the next call (hook off) is correct again."""
    from serving_router_top_gb300.model import ModelState
    w = I.small_workload(T=4, H=512, I=256, E=32, k=4, I_shared=256, zipf_s=0.5, resident_frac=1.0, seed=8)
    st = ModelState(w)
    st.ws.set_wait_test(20_000_000, 1)
    x = torch.from_numpy(I.activations(w.seed, 0, 4, 512).view(np.int16)).cuda()
    y = torch.zeros((4, 512), dtype=torch.float32, device="cuda")
    st.forward(0, x, y, 4)
    assert moe.moe_sync_status(st.ws) == moe.MOE_ETIMEOUT
    st.ws.set_wait_test(1_000_000_000, 0)
    for step in range(2):
        check_layer(st, 4, step=step)
    assert ran_fused(st, 4)


def test_fused_decode_rejects_bad_settings():
    from serving_router_top_gb300.model import ModelState
    st = ModelState(I.small_workload(T=2, H=512, I=256, E=8, k=2, I_shared=0))
    with pytest.raises(moe.MoeError):
        st.ws.set_decode_path(2)
    with pytest.raises(moe.MoeError):
        st.ws.set_wait_test(0, 0)
    with pytest.raises(moe.MoeError):
        st.ws.set_wait_test(1000, -1)


def test_fused_decode_in_graph_replays():
    """The single kernel captured in a CUDA graph and replayed on fresh windows."""
    from serving_router_top_gb300.model import ModelState
    w = I.WORKLOADS["decode_t4_h2048_e512_k10"]
    st = ModelState(w)
    T = w.T
    x_in = torch.zeros((T, st.H), dtype=torch.int16, device="cuda")
    y = torch.zeros((T, st.H), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        st.forward(0, x_in, y, T, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            st.forward(0, x_in, y, T, stream=s)
    for step in range(3):
        x_bits = I.activations(w.seed, 70 + step, T, st.H)
        x_in.copy_(torch.from_numpy(x_bits.view(np.int16)).cuda())
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert moe.moe_sync_status(st.ws) == moe.MOE_OK
        logits = st.ws.routing(T)[0].cpu().numpy()
        ref = U.oracle_layer_from_state(st, 0, x_bits, logits)
        U.assert_close_layer(y.cpu().numpy(), ref.y)
