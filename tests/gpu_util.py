"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and the
oracle on the same seeded inputs, and compare."""
import numpy as np
import pytest
import torch

from oracle import formats, layer as olayer

TOL_REL = 1e-2   # max|dy| <= 1e-2 * rms(ref) + 1e-3 (fp32 accumulate, fp32 output)
TOL_ABS = 1e-3


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from serving_router_top_gb300 import build
    build.build()


def bf16_half_ulp(a: np.ndarray) -> np.ndarray:
    """Half a bf16 unit in the last place at |a| (normal range)."""
    a = np.abs(np.asarray(a, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-38)))
    return np.exp2(e - 8)


def assert_close_layer(y_gpu: np.ndarray, y_ref: np.ndarray, bf16_out: bool = False, what: str = "y"):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    d = np.abs(y_gpu - y_ref)
    rms = float(np.sqrt(np.mean(y_ref * y_ref)))
    tol = TOL_REL * rms + TOL_ABS
    if bf16_out:
        tol = tol + bf16_half_ulp(y_ref)
    bad = d > tol
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {d.size} elements out of tolerance; max|d|={d.max():.4g}, "
                           f"rms(ref)={rms:.4g}, max|d|/rms={d.max() / max(rms, 1e-30):.3g}")
    return float(d.max() / max(rms, 1e-30))


def logits_bound(x_bits, wr_bits, bias) -> np.ndarray:
    """Error bound for an fp32-accumulated dot product of H exact products, plus the bias add:
    H * 2^-24 * sum|x_i w_i| + 2^-24 |l|."""
    x = np.abs(formats.bf16_value(x_bits))
    w = np.abs(formats.bf16_value(wr_bits))
    s = x @ w.T
    H = x.shape[1]
    mag = s + (np.abs(bias)[None, :] if bias is not None else 0)
    return H * 2.0 ** -24 * s + 2.0 ** -23 * mag + 1e-30


def bf16_to_f32_tensor(bits: np.ndarray) -> np.ndarray:
    return formats.bf16_value(bits)


def y_to_numpy(y: torch.Tensor, bf16: bool) -> np.ndarray:
    if bf16:
        return y.view(torch.bfloat16).float().cpu().numpy().astype(np.float64)
    return y.cpu().numpy().astype(np.float64)


def oracle_layer_from_state(st, layer: int, x_bits: np.ndarray, logits: np.ndarray, tail_skip: int = 0):
    """Oracle forward of one layer of a ModelState, routed on the given fp32 logits."""
    lw = st.layers[layer]
    li = lw.host
    resid = st.resid_table()
    stage = st.stage_table()
    return olayer.moe_layer(x_bits, li.w_router, li.bias, st.k, lambda e: st.expert_host(layer, e), st.H, st.I,
                            layer=layer, resid=resid, stage=stage, shared=li.shared, I_shared=st.I_shared,
                            w_shared_gate_bits=li.w_shared_gate, logits=logits, tail_skip=tail_skip)
