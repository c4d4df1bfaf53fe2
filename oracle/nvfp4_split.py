"""Activations as a sum of NVFP4 terms (oracle side; test infrastructure only).

A block-scaled FP4 tensor-core product needs both operands in the 4-bit format.
The weights already are; an activation vector v (bf16 x, or the fp32
intermediate h) is not.  The split writes v as R NVFP4 terms,
q_1 = Q(v), q_2 = Q(v - q_1), ..., so that sum_r q_r approaches v, and each
term enters the product as its own operand.  This module states the quantiser
Q and measures, on the layer, how far the R-term product is from the exact one
-- the evidence for choosing R.  The layer oracle itself (oracle/layer.py)
stays exact.

The format (PLE offload page, "NVFP4 code 和 scale 如何反量化"): a value is an
E2M1 code value times the FP8-E4M3 scale of its block of 16 times an FP32
global scale.  The pages give the decoding only; the quantiser is the plain
reading of it:
  * one FP32 global scale G per term: the power of two that puts the term's
    largest block scale at most at 448 (the largest E4M3 value) -- the smallest
    G with max|v| / (6 G) <= 448;
  * the block scale s of each 16 values: the smallest non-negative E4M3 value
    with 6 s G >= max|v| of the block (rounded up, so no code saturates);
  * each code: the E2M1 value nearest to v / (s G), ties to the even code
    (the one whose lowest mantissa bit is 0).
"""
from __future__ import annotations

import numpy as np

from .formats import E2M1_MAGNITUDES, e4m3_value

# every non-negative E4M3 value below NaN, ascending (bytes 0x00..0x7E)
_E4M3_POS = e4m3_value(np.arange(0, 0x7F, dtype=np.uint8))


def e4m3_ceil(v: np.ndarray) -> np.ndarray:
    """The smallest non-negative E4M3 value >= v (v >= 0, at most 448)."""
    v = np.asarray(v, dtype=np.float64)
    idx = np.searchsorted(_E4M3_POS, v, side="left")
    return _E4M3_POS[np.minimum(idx, _E4M3_POS.size - 1)]


def e2m1_round(u: np.ndarray) -> np.ndarray:
    """|u| <= 6 to the nearest E2M1 value, ties to the even code; the sign is kept."""
    u = np.asarray(u, dtype=np.float64)
    a = np.abs(u)
    grid = E2M1_MAGNITUDES                       # codes 0..7 by magnitude
    i = np.clip(np.searchsorted(grid, a, side="left"), 1, grid.size - 1)
    lo, hi = grid[i - 1], grid[i]
    take_hi = (a - lo > hi - a) | ((a - lo == hi - a) & ((i % 2) == 0))   # tie: the even code
    mag = np.where(take_hi, hi, lo)
    return np.where(u < 0, -mag, mag)


def quantize_nvfp4(v: np.ndarray) -> np.ndarray:
    """Q(v) for rows of v (last axis a multiple of 16): the dequantised NVFP4 value of v."""
    v = np.asarray(v, dtype=np.float64)
    amax = float(np.max(np.abs(v))) if v.size else 0.0
    if amax == 0.0:
        return np.zeros_like(v)
    G = 2.0 ** np.ceil(np.log2(amax / (6.0 * 448.0)))
    blocks = v.reshape(v.shape[:-1] + (v.shape[-1] // 16, 16))
    bmax = np.max(np.abs(blocks), axis=-1, keepdims=True)
    s = e4m3_ceil(bmax / (6.0 * G))
    safe = np.where(s > 0, s, 1.0)
    q = np.where(s > 0, e2m1_round(blocks / (safe * G)), 0.0) * s * G
    return q.reshape(v.shape)


def encode_nvfp4(row: np.ndarray):
    """Q of one row as stored: (code values [K] (E2M1 values, fp64), E4M3 scale bytes [K/16],
    global scale G).  The dequantised term is codes * scale(byte) * G, per block of 16."""
    row = np.asarray(row, dtype=np.float64)
    K = row.size
    amax = float(np.max(np.abs(row))) if K else 0.0
    if amax == 0.0:
        return np.zeros(K), np.zeros(K // 16, dtype=np.uint8), 1.0
    G = float(2.0 ** np.ceil(np.log2(amax / (6.0 * 448.0))))
    blocks = row.reshape(K // 16, 16)
    bmax = np.max(np.abs(blocks), axis=-1)
    sbyte = np.minimum(np.searchsorted(_E4M3_POS, bmax / (6.0 * G), side="left"), _E4M3_POS.size - 1)
    s = _E4M3_POS[sbyte]
    safe = np.where(s > 0, s, 1.0)
    codes = np.where(s[:, None] > 0, e2m1_round(blocks / (safe[:, None] * G)), 0.0)
    return codes.reshape(K), sbyte.astype(np.uint8), G


def split_terms(v: np.ndarray, R: int):
    """The R terms q_1 .. q_R of each row of v (each a dequantised NVFP4 array; every row of
    every term has its own global scale)."""
    v = np.atleast_2d(np.asarray(v, dtype=np.float64))
    terms, rest = [], v
    for _ in range(R):
        q = np.stack([quantize_nvfp4(row) for row in rest])
        terms.append(q)
        rest = rest - q
    return terms


def split_sum(v: np.ndarray, R: int) -> np.ndarray:
    return np.sum(split_terms(v, R), axis=0)


def layer_with_split(x_bits, li, experts, H: int, I: int, k: int, R: int, logits):
    """The layer of oracle/layer.py with the activations of every expert product replaced by
    their R-term splits (x for gate/up, h for down); routing as given.  Returns y (fp64)."""
    from . import layer as L
    from .formats import bf16_value
    x = bf16_value(x_bits)
    ids, w = L.top_k(logits, k)
    T = x.shape[0]
    y = np.zeros((T, H))
    xs = split_sum(x, R)

    def ffn(xq, de):
        hq = L.silu(xq @ de.gate.T) * (xq @ de.up.T)
        return split_sum(hq, R) @ de.down.T

    for t in range(T):
        for r in range(k):
            de = L.dequantize_expert(experts(int(ids[t, r])), H, I)
            y[t] += w[t, r] * ffn(xs[t:t + 1], de)[0]
    if li.shared is not None:
        de = L.dequantize_expert(li.shared, H, I)
        gamma = L.sigmoid(x @ bf16_value(li.w_shared_gate))
        y += gamma[:, None] * ffn(xs, de)
    return y
