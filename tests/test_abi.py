"""The C-ABI library builds, loads without a GPU and exports every symbol include/moe.h declares;
host-only entry points (blob sizing and packing, error strings) checked on the CPU."""
import os
import re

import numpy as np
import pytest

from oracle import formats
from serving_router_top_gb300 import build, inputs, moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return moe.load()


def test_header_declares_the_five_path_calls():
    names = header_functions()
    for n in ("moe_route", "moe_group", "moe_layer_forward", "cache_heat_update", "cache_plan_swaps"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    assert set(names) == set(moe.EXPORTED), set(names) ^ set(moe.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror(lib):
    assert moe.strerror(moe.MOE_OK) == "ok"
    assert "resident" in moe.strerror(moe.MOE_EMISSING)


@pytest.mark.parametrize("H,I", [(256, 128), (2048, 512), (128, 64), (4096, 2048)])
def test_blob_pack_layout(lib, H, I):
    ex = inputs.expert_weights(0, 0, 7, H, I)
    ex.gscale = (0.5, 2.0, 1.25)
    blob = moe.moe_pack_expert(ex.gate, ex.up, ex.down, H, I, ex.gscale)
    assert blob.size == moe.moe_blob_bytes(H, I)
    hdr = blob[:32].view(np.uint32)
    assert hdr[0] == 0x42454F4D and hdr[2] == H and hdr[3] == I
    assert blob[16:28].view(np.float32).tolist() == [0.5, 2.0, 1.25]
    # every region holds the canonical codes / scales, 256-byte aligned, in gate, up, down order
    off = 256
    regions = []
    for rows, cols in ((I, H), (I, H), (H, I)):
        regions.append((off, rows, cols))
        off += -(-rows * cols // 2 // 256) * 256
    for (coff, rows, cols), m in zip(regions, (ex.gate, ex.up, ex.down)):
        assert np.array_equal(blob[coff:coff + rows * cols // 2].reshape(rows, cols // 2), m[:, :cols // 2])
    for (_, rows, cols), m in zip(regions, (ex.gate, ex.up, ex.down)):
        assert np.array_equal(blob[off:off + rows * cols // 16].reshape(rows, cols // 16), m[:, cols // 2:])
        off += -(-rows * cols // 16 // 256) * 256
    assert off + 256 == blob.size  # 256-byte tail guard


def test_pack_rejects_bad_shapes(lib):
    with pytest.raises(moe.MoeError):
        moe.moe_pack_expert(np.zeros((4, 9), np.uint8), np.zeros((4, 9), np.uint8), np.zeros((16, 2), np.uint8),
                            16, 4)
    assert moe.moe_blob_bytes(100, 64) == 0


def test_blob_roundtrip_dequantises_like_canonical(lib):
    """Reading a blob region back as canonical rows gives the same oracle values."""
    H, I = 128, 64
    ex = inputs.expert_weights(3, 1, 2, H, I)
    blob = moe.moe_pack_expert(ex.gate, ex.up, ex.down, H, I)
    codes = blob[256:256 + I * H // 2].reshape(I, H // 2)
    sc_off = 256 + 2 * (I * H // 2) + (H * I // 2)
    scales = blob[sc_off:sc_off + I * H // 16].reshape(I, H // 16)
    rows = np.concatenate([codes, scales], axis=1)
    assert np.array_equal(formats.dequantize(rows, H), formats.dequantize(ex.gate, H))


def test_null_handles_are_rejected_without_a_device(lib):
    """Every entry point that takes a cache or workspace handle checks it before any CUDA call,
    so these run on a machine without a GPU."""
    P = None
    assert lib.moe_ws_set_tail_skip(P, 7) == moe.MOE_EINVAL
    assert lib.moe_ws_set_fused_heat(P, 1) == moe.MOE_EINVAL
    assert lib.moe_ws_set_profiling(P, 1) == moe.MOE_EINVAL
    assert lib.cache_lru_plan(P, P, 0, 8, P, P, P) == moe.MOE_EINVAL
    assert lib.moe_cache_apply_lru(P, P, P, P, P) == moe.MOE_EINVAL
    assert lib.moe_cache_apply_swaps(P, P, P, P, P) == moe.MOE_EINVAL
    assert lib.moe_group(P, 4, 2, 8, 0, P, P, P) == moe.MOE_EINVAL
    assert lib.moe_cache_destroy(P) == moe.MOE_OK
    assert lib.moe_ws_destroy(P) == moe.MOE_OK


def test_shape_limits_stated_in_the_header_are_enforced(lib):
    """moe_ws_create rejects rows outside powers of two in [64, 4096] and k outside [1, min(E, 32)]
    before allocating (MOE_EINVAL, no CUDA call)."""
    import ctypes as C
    h = C.c_void_p()
    for H, I, E, k in ((96, 64, 8, 2), (64, 8192, 8, 2), (64, 64, 8, 9), (64, 64, 2048, 2), (64, 64, 64, 33),
                       (64, 64, 8, 0)):
        assert lib.moe_ws_create(C.byref(h), 4, moe.moe_layer_shape(H, I, E, k, 0)) == moe.MOE_EINVAL
    assert lib.moe_ws_create(C.byref(h), 0, moe.moe_layer_shape(64, 64, 8, 2, 0)) == moe.MOE_EINVAL


def test_edge_recipe_reaches_the_ends_of_the_format(lib):
    """The edge-case workload's weights hold zero, subnormal and 448 block scales, keep the scale
    sign bit clear, and carry their non-unit global scales into the blob header; the oracle's
    values then reach 6 * 448 = 2688 and 0.5 * 2^-9 = 2^-10 (times the global scale)."""
    w = inputs.edge_workload()
    ex = inputs.expert_of(w, 0, 3)
    sc = np.concatenate([m[:, c // 2:].ravel() for m, c in ((ex.gate, w.shape.H), (ex.up, w.shape.H),
                                                              (ex.down, w.shape.I))])
    assert (sc == 0).any() and ((sc >= 1) & (sc <= 7)).any() and (sc == 0x7E).any()
    assert (sc < 0x7F).all()   # no NaN scale, sign bit clear
    vals = np.abs(formats.dequantize(ex.gate, w.shape.H, ex.gscale[0]))
    nz = vals[vals > 0]
    assert vals.max() == 2688.0 * 0.375
    assert nz.min() == 2.0 ** -10 * 0.375
    blob = moe.moe_pack_expert(ex.gate, ex.up, ex.down, w.shape.H, w.shape.I, ex.gscale)
    assert blob[16:28].view(np.float32).tolist() == [0.375, 2.0, 1.25]
    # the default recipe is unchanged by the edge option: exponent fields 3..6 only
    d = inputs.expert_weights(0, 0, 1, 128, 64)
    e = (d.gate[:, 64:] >> 3) & 15
    assert e.min() == 3 and e.max() == 6
