"""Pins of the oracle's NVFP4 activation split (the quantiser behind the FP4 prefill path) and
the measurement that sets its number of terms R.  The quantiser reads the format's decoding
(PLE offload page, "NVFP4 code 和 scale 如何反量化": E2M1 code x E4M3 scale per 16 x FP32 global)."""
import numpy as np
import pytest

from oracle import formats, layer as olayer, nvfp4_split as S
from serving_router_top_gb300 import inputs as I


def test_e2m1_rounding_grid_and_ties():
    grid = formats.E2M1_MAGNITUDES
    assert np.array_equal(S.e2m1_round(grid), grid)
    assert np.array_equal(S.e2m1_round(-grid), -grid)
    # ties go to the even code: 0.25->0 (code 0), 0.75->1 (code 2), 1.25->1 (code 2), 1.75->2 (code 4),
    # 2.5->2 (code 4), 3.5->4 (code 6), 5->4 (code 6)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    assert S.e2m1_round(ties).tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]
    assert S.e2m1_round(np.array([0.26, 2.51, 5.01, 5.99])).tolist() == [0.5, 3.0, 6.0, 6.0]


def test_e4m3_ceil_is_the_smallest_not_below():
    allv = formats.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    assert np.array_equal(S.e4m3_ceil(allv), allv)
    g = np.random.default_rng(1)
    v = g.uniform(0, 448, 1000)
    c = S.e4m3_ceil(v)
    assert (c >= v).all()
    below = allv[np.searchsorted(allv, c) - 1]
    assert (below < v).all()


def test_representable_rows_are_one_exact_term():
    """A row whose blocks are E2M1 values times an E4M3 scale times the row's own power of two,
    each block holding a 6, quantises to itself: one term, zero residual."""
    g = np.random.default_rng(2)
    codes = formats.e2m1_value(g.integers(0, 16, size=(8, 16)))
    codes[:, 0] = 6.0
    sc = formats.e4m3_value(g.integers(0x20, 0x78, size=8))
    G = 2.0 ** -5
    # the row's G must come out as the given one: put one block's scale at the top of its octave range
    sc[0] = 448.0
    row = (codes * sc[:, None] * G).reshape(-1)
    c, sb, Gq = S.encode_nvfp4(row)
    assert Gq == G
    assert np.array_equal(S.quantize_nvfp4(row), row)
    assert np.array_equal(S.split_sum(row, 3)[0], row)


def test_terms_shrink_the_residual():
    g = np.random.default_rng(3)
    v = g.standard_normal((4, 512))
    prev = np.inf
    for R in (1, 2, 3, 4):
        err = np.abs(S.split_sum(v, R) - v).max() / np.abs(v).max()
        assert err < prev
        prev = err
    assert prev < 2.0 ** -9


@pytest.mark.parametrize("R,ok", [(2, False), (4, True)])
def test_layer_error_per_R(R, ok):
    """The evidence for R: the layer with x and h split into R terms, against the exact layer,
    under the parity tolerance 1e-2 rms + 1e-3 (a small layer of the chunk's kind; the committed
    study at the chunk's full shape measured max|dy|/rms 1.36, 0.092, 0.0094, 0.00055 for
    R = 1..4)."""
    w = I.small_workload(T=12, H=512, I=256, E=16, k=4, I_shared=256, zipf_s=0.5, seed=4)
    s = w.shape
    li = I.layer_inputs(w)
    logits = olayer.router_logits(li.x, li.w_router, li.bias)
    ex = lambda e: I.expert_of(w, 0, e)
    ref = olayer.moe_layer(li.x, li.w_router, li.bias, s.k, ex, s.H, s.I, shared=li.shared, I_shared=s.I_shared,
                           w_shared_gate_bits=li.w_shared_gate, logits=logits).y
    y = S.layer_with_split(li.x, li, ex, s.H, s.I, s.k, R, logits)
    rms = np.sqrt(np.mean(ref ** 2))
    within = np.abs(y - ref).max() <= 1e-2 * rms + 1e-3
    assert within == ok
