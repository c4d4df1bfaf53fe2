"""ctypes binding of libmoe (``include/moe.h``): same names, argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module only
turns torch tensors into device pointers and streams into handles.  If the
library has not been built (``python -m serving_router_top_gb300.build``) the
first call raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libmoe.so")

MOE_OK, MOE_EINVAL, MOE_ENOMEM, MOE_ECUDA, MOE_EMISSING, MOE_ERANGE, MOE_ENAN, MOE_ETIMEOUT = range(8)
MOE_SRC_MISSING, MOE_SRC_RESIDENT, MOE_SRC_STAGED, MOE_SRC_SKIPPED = -1, 0, 1, 2
MOE_MODE_AUTO, MOE_MODE_DECODE, MOE_MODE_PREFILL = 0, 1, 2
MOE_DECODE_FUSED, MOE_DECODE_CHAIN = 0, 1

# Every symbol include/moe.h declares.
EXPORTED = (
    "moe_blob_bytes", "moe_pack_expert", "moe_cache_create", "moe_cache_destroy", "moe_cache_admit",
    "moe_cache_fill", "moe_cache_get_view", "moe_get_stats", "moe_ws_create", "moe_ws_destroy", "moe_ws_get_view",
    "moe_sync_status", "moe_strerror", "moe_route", "moe_group", "moe_layer_forward", "cache_heat_update",
    "cache_plan_swaps", "moe_cache_apply_swaps", "moe_ws_set_profiling", "moe_ws_kernel_times",
    "cache_plan_swaps_noalloc", "moe_residual_rmsnorm", "moe_layer_forward_streamed", "moe_ws_set_tail_skip",
    "moe_ws_set_fused_heat", "cache_lru_plan", "moe_cache_apply_lru", "moe_ws_set_decode_path",
    "moe_ws_set_wait_test", "moe_nvfp4_split", "moe_layers_forward_streamed",
)


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})" if what else f"{strerror(code)} ({code})")


class moe_layer_shape(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("k", C.c_int), ("I_shared", C.c_int)]


class moe_layer_desc(C.Structure):
    _fields_ = [("w_router", C.c_void_p), ("bias", C.c_void_p), ("w_shared_gate", C.c_void_p),
                ("shared_blob", C.c_void_p), ("layer", C.c_int), ("s", moe_layer_shape)]


class moe_cache_view(C.Structure):
    _fields_ = [("resid", C.c_void_p), ("stage", C.c_void_p), ("heat", C.c_void_p), ("slot_owner", C.c_void_p),
                ("slots", C.c_void_p), ("staging", C.c_void_p), ("blob_bytes", C.c_size_t), ("L", C.c_int),
                ("E", C.c_int), ("nslots", C.c_int), ("nstaging", C.c_int), ("lru_tick", C.c_void_p),
                ("lru_clock", C.c_void_p)]


class moe_ws_view(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("num_groups", "grp_expert", "grp_off", "grp_slot", "grp_src", "ent_tok",
                                           "ent_pos", "logits", "topk_ids", "topk_w", "error")]


class moe_swap(C.Structure):
    _fields_ = [("layer", C.c_int), ("hot_expert", C.c_int), ("cold_expert", C.c_int), ("slot", C.c_int),
                ("diff", C.c_float)]


class moe_policy_cfg(C.Structure):
    _fields_ = [("threshold", C.c_float), ("max_swaps", C.c_int), ("decay", C.c_float)]


SWAP_DTYPE = np.dtype([("layer", "<i4"), ("hot_expert", "<i4"), ("cold_expert", "<i4"), ("slot", "<i4"),
                       ("diff", "<f4")])

_lib = None


def load() -> C.CDLL:
    """Load libmoe.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libmoe.so not built ({LIB_PATH}); run python -m serving_router_top_gb300.build")
    lib = C.CDLL(LIB_PATH)
    P, I, Z, F = C.c_void_p, C.c_int, C.c_size_t, C.c_float
    sig = {
        "moe_blob_bytes": (Z, [I, I]),
        "moe_pack_expert": (I, [P, P, P, I, I, F, F, F, P]),
        "moe_cache_create": (I, [C.POINTER(P), I, I, I, I, I, I, P, I]),
        "moe_cache_destroy": (I, [P]),
        "moe_cache_admit": (I, [P, I, I, C.POINTER(C.c_int32)]),
        "moe_cache_fill": (I, [P, P, I]),
        "moe_cache_get_view": (I, [P, C.POINTER(moe_cache_view)]),
        "moe_get_stats": (I, [P, P]),
        "moe_ws_create": (I, [C.POINTER(P), I, moe_layer_shape]),
        "moe_ws_destroy": (I, [P]),
        "moe_ws_get_view": (I, [P, C.POINTER(moe_ws_view)]),
        "moe_sync_status": (I, [P, P]),
        "moe_strerror": (C.c_char_p, [I]),
        "moe_route": (I, [P, P, P, P, I, I, I, I, P, P, P, P]),
        "moe_group": (I, [P, I, I, I, I, P, P, P]),
        "moe_layer_forward": (I, [C.POINTER(moe_layer_desc), P, P, I, I, P, P, I, P]),
        "moe_layer_forward_streamed": (I, [C.POINTER(moe_layer_desc), P, P, I, I, P, P, I, I, P, P]),
        "cache_heat_update": (I, [P, P, I, I, I, P, P]),
        "cache_plan_swaps": (I, [P, C.POINTER(moe_policy_cfg), P, P, P]),
        "cache_plan_swaps_noalloc": (I, [P, P, I, I, C.POINTER(moe_policy_cfg), P, P, P]),
        "moe_residual_rmsnorm": (I, [P, P, P, I, I, F, P]),
        "moe_cache_apply_swaps": (I, [P, P, P, P, P]),
        "moe_ws_set_profiling": (I, [P, I]),
        "moe_ws_set_tail_skip": (I, [P, I]),
        "moe_ws_set_fused_heat": (I, [P, I]),
        "moe_ws_set_decode_path": (I, [P, I]),
        "moe_ws_set_wait_test": (I, [P, C.c_ulonglong, I]),
        "moe_nvfp4_split": (I, [P, I, I, I, I, I, P, P, P, P]),
        "moe_layers_forward_streamed": (I, [P, I, P, P, P, I, P, P, I, F, P, P]),
        "cache_lru_plan": (I, [P, P, I, I, P, P, P]),
        "moe_cache_apply_lru": (I, [P, P, P, P, P]),
        "moe_ws_kernel_times": (I, [P, I, P, P, C.POINTER(C.c_int)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().moe_strerror(int(code)).decode()
    except RuntimeError:
        return f"error {code}"


def _check(rc: int, what: str) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


class _CudaArray:
    """Minimal __cuda_array_interface__ holder so torch can view library-owned memory."""

    def __init__(self, ptr: int, shape, typestr: str, owner):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}
        self._owner = owner


def device_view(ptr: int, shape, dtype: str, owner=None):
    """A torch tensor aliasing library device memory (no copy)."""
    import torch
    typestr = {"int32": "<i4", "float32": "<f4", "uint8": "|u1"}[dtype]
    return torch.as_tensor(_CudaArray(ptr, shape, typestr, owner), device="cuda")


# ------------------------------------------------------------------ blobs

def moe_blob_bytes(H: int, I: int) -> int:
    return int(load().moe_blob_bytes(H, I))


def moe_pack_expert(gate_rows: np.ndarray, up_rows: np.ndarray, down_rows: np.ndarray, H: int, I: int,
                    gscale=(1.0, 1.0, 1.0), out: Optional[np.ndarray] = None) -> np.ndarray:
    """Canonical packed rows (host numpy uint8) -> one slot blob (host numpy uint8)."""
    nb = moe_blob_bytes(H, I)
    if out is None:
        out = np.empty(nb, dtype=np.uint8)
    g, u, d = (np.ascontiguousarray(a, dtype=np.uint8) for a in (gate_rows, up_rows, down_rows))
    _check(load().moe_pack_expert(g.ctypes.data, u.ctypes.data, d.ctypes.data, H, I, float(gscale[0]),
                                  float(gscale[1]), float(gscale[2]), out.ctypes.data), "moe_pack_expert")
    return out


# ------------------------------------------------------------------ cache

class Cache:
    """Owner of a moe_cache handle and (a reference to) its backing store tensor."""

    def __init__(self, L: int, E: int, H: int, I: int, nslots: int, nstaging: int, backing, backing_on_device: bool):
        h = C.c_void_p()
        _check(load().moe_cache_create(C.byref(h), L, E, H, I, nslots, nstaging, _ptr(backing),
                                       1 if backing_on_device else 0), "moe_cache_create")
        self.handle = h
        self.backing = backing
        self.L, self.E, self.H, self.I, self.nslots, self.nstaging = L, E, H, I, nslots, nstaging
        v = moe_cache_view()
        _check(load().moe_cache_get_view(h, C.byref(v)), "moe_cache_get_view")
        self.view = v

    def close(self):
        if self.handle:
            load().moe_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def admit(self, layer: int, expert: int) -> int:
        s = C.c_int32()
        _check(load().moe_cache_admit(self.handle, layer, expert, C.byref(s)), "moe_cache_admit")
        return int(s.value)

    def fill(self, mask: np.ndarray, staging: bool = False) -> None:
        m = np.ascontiguousarray(mask, dtype=np.uint8).ravel()
        assert m.size == self.L * self.E
        _check(load().moe_cache_fill(self.handle, m.ctypes.data, 1 if staging else 0), "moe_cache_fill")

    def tables(self):
        """Torch views of resid, stage, heat (device, aliasing the library's memory)."""
        LE = self.L * self.E
        return (device_view(self.view.resid, (LE,), "int32", self), device_view(self.view.stage, (LE,), "int32", self),
                device_view(self.view.heat, (LE,), "float32", self))

    def lru_tables(self):
        """Torch views of the global LRU's slot ticks (uint32 as int32 [nslots]) and clock (int32 [1])."""
        return (device_view(self.view.lru_tick, (max(1, self.view.nslots),), "int32", self),
                device_view(self.view.lru_clock, (1,), "int32", self))

    def stats(self) -> np.ndarray:
        """int64 [L, 5]: groups looked up, resident hits, staged, missing, skipped by the tail skip."""
        out = np.zeros((self.L, 5), dtype=np.int64)
        _check(load().moe_get_stats(self.handle, out.ctypes.data), "moe_get_stats")
        return out


# -------------------------------------------------------------- workspace

class Workspace:
    def __init__(self, maxT: int, H: int, I: int, E: int, k: int, I_shared: int):
        h = C.c_void_p()
        self.shape = moe_layer_shape(H, I, E, k, I_shared)
        _check(load().moe_ws_create(C.byref(h), maxT, self.shape), "moe_ws_create")
        self.handle = h
        self.maxT = maxT
        v = moe_ws_view()
        _check(load().moe_ws_get_view(h, C.byref(v)), "moe_ws_get_view")
        self.view = v

    def close(self):
        if self.handle:
            load().moe_ws_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def groups(self, T: int):
        """Copy the last grouping to host numpy: (experts, off, slot, src, ent_tok, ent_pos)."""
        import torch
        torch.cuda.synchronize()
        k = self.shape.k
        G = int(device_view(self.view.num_groups, (1,), "int32", self).cpu()[0])
        n = T * k
        get = lambda p, m: device_view(p, (m,), "int32", self).cpu().numpy().copy()
        return (get(self.view.grp_expert, G), get(self.view.grp_off, G + 1), get(self.view.grp_slot, G),
                get(self.view.grp_src, G), get(self.view.ent_tok, n), get(self.view.ent_pos, n))

    def routing(self, T: int):
        """(logits [T,E], ids [T,k], w [T,k]) of the last forward (device tensors)."""
        E, k = self.shape.E, self.shape.k
        return (device_view(self.view.logits, (T, E), "float32", self),
                device_view(self.view.topk_ids, (T, k), "int32", self),
                device_view(self.view.topk_w, (T, k), "float32", self))

    def set_tail_skip(self, min_rank: int) -> None:
        """Drop non-resident experts that every choosing token ranks at or past min_rank (0: off)."""
        _check(load().moe_ws_set_tail_skip(self.handle, int(min_rank)), "moe_ws_set_tail_skip")

    def set_fused_heat(self, enable: bool) -> None:
        """Let the grouping of later calls with a cache also add the window's counts to the layer's heat."""
        _check(load().moe_ws_set_fused_heat(self.handle, 1 if enable else 0), "moe_ws_set_fused_heat")

    def set_decode_path(self, path: int) -> None:
        """MOE_DECODE_FUSED (one cooperative kernel where the shapes fit) or MOE_DECODE_CHAIN."""
        _check(load().moe_ws_set_decode_path(self.handle, int(path)), "moe_ws_set_decode_path")

    def set_wait_test(self, wait_ns: int, phantom_arrivals: int) -> None:
        """Bound of the decode kernel's grid-barrier waits, and arrivals they wait for that never come."""
        _check(load().moe_ws_set_wait_test(self.handle, int(wait_ns), int(phantom_arrivals)), "moe_ws_set_wait_test")

    def set_profiling(self, enable: bool) -> None:
        _check(load().moe_ws_set_profiling(self.handle, 1 if enable else 0), "moe_ws_set_profiling")

    def kernel_times(self):
        """[(name, ms)] of the kernels of the most recent call (profiling must be on)."""
        ms = (C.c_float * 16)()
        names = (C.c_char_p * 16)()
        n = C.c_int()
        _check(load().moe_ws_kernel_times(self.handle, 16, ms, names, C.byref(n)), "moe_ws_kernel_times")
        return [(names[i].decode(), float(ms[i])) for i in range(n.value)]

    @property
    def error_ptr(self) -> int:
        return self.view.error


# ------------------------------------------------------------- hot path

def moe_sync_status(ws: Workspace, stream=None) -> int:
    return int(load().moe_sync_status(ws.handle, _stream(stream)))


def moe_route(x, w_router, bias, logits_io, T: int, H: int, E: int, k: int, topk_ids, topk_w, err=None,
              stream=None) -> None:
    _check(load().moe_route(_ptr(x), _ptr(w_router), _ptr(bias), _ptr(logits_io), T, H, E, k, _ptr(topk_ids),
                            _ptr(topk_w), _ptr(err), _stream(stream)), "moe_route")


def moe_group(topk_ids, T: int, k: int, E: int, layer: int, cache: Cache, ws: Workspace, stream=None) -> None:
    _check(load().moe_group(_ptr(topk_ids), T, k, E, layer, cache.handle, ws.handle, _stream(stream)), "moe_group")


def layer_desc(w_router, bias, w_shared_gate, shared_blob, layer: int, H: int, I: int, E: int, k: int,
               I_shared: int) -> moe_layer_desc:
    return moe_layer_desc(_ptr(w_router), _ptr(bias), _ptr(w_shared_gate), _ptr(shared_blob), layer,
                          moe_layer_shape(H, I, E, k, I_shared))


def moe_layer_forward(desc: moe_layer_desc, x, y, y_is_fp32: bool, T: int, cache: Cache, ws: Workspace,
                      mode: int = MOE_MODE_AUTO, stream=None) -> None:
    _check(load().moe_layer_forward(C.byref(desc), _ptr(x), _ptr(y), 1 if y_is_fp32 else 0, T, cache.handle,
                                    ws.handle, mode, _stream(stream)), "moe_layer_forward")


def moe_layer_forward_streamed(desc: moe_layer_desc, x, y, y_is_fp32: bool, T: int, cache: Cache, ws: Workspace,
                               U: int, stream=None, copy_stream=None, buffers: int = 2) -> None:
    _check(load().moe_layer_forward_streamed(C.byref(desc), _ptr(x), _ptr(y), 1 if y_is_fp32 else 0, T, cache.handle,
                                             ws.handle, U, buffers, _stream(stream), _stream(copy_stream)),
           "moe_layer_forward_streamed")


def moe_layers_forward_streamed(descs, x_res, xn, y, T: int, cache: Cache, ws: Workspace, buffers: int = 2,
                                eps: float = 1e-6, stream=None, copy_stream=None) -> None:
    """Layers of a prefill chunk on a residual stream, each layer's experts streamed one layer ahead."""
    arr = (moe_layer_desc * len(descs))(*descs)
    _check(load().moe_layers_forward_streamed(arr, len(descs), _ptr(x_res), _ptr(xn), _ptr(y), T, cache.handle,
                                              ws.handle, buffers, eps, _stream(stream), _stream(copy_stream)),
           "moe_layers_forward_streamed")


def moe_nvfp4_split(src, src_is_fp32: bool, rows: int, K: int, ld: int, R: int, codes, scales, gscale,
                    stream=None) -> None:
    """Rows of activations -> R NVFP4 terms each (codes, block scales, global scales)."""
    _check(load().moe_nvfp4_split(_ptr(src), 1 if src_is_fp32 else 0, rows, K, ld, R, _ptr(codes), _ptr(scales),
                                  _ptr(gscale), _stream(stream)), "moe_nvfp4_split")


def cache_heat_update(cache: Cache, topk_ids, T: int, k: int, layer: int, err=None, stream=None) -> None:
    _check(load().cache_heat_update(cache.handle, _ptr(topk_ids), T, k, layer, _ptr(err), _stream(stream)),
           "cache_heat_update")


def cache_plan_swaps(cache: Cache, threshold: float, max_swaps: int, decay: float, plan_dev, n_dev,
                     stream=None) -> None:
    cfg = moe_policy_cfg(threshold, max_swaps, decay)
    _check(load().cache_plan_swaps(cache.handle, C.byref(cfg), _ptr(plan_dev), _ptr(n_dev), _stream(stream)),
           "cache_plan_swaps")


def moe_residual_rmsnorm(x_res, y_prev, xn_out, T: int, H: int, eps: float = 1e-6, stream=None) -> None:
    """x_res (fp32 [T,H]) += y_prev (bf16 bits, or None); xn_out (bf16 bits) = RMSNorm(x_res)."""
    _check(load().moe_residual_rmsnorm(_ptr(x_res), _ptr(y_prev), _ptr(xn_out), T, H, eps, _stream(stream)),
           "moe_residual_rmsnorm")


# Capacity of the static scratch behind cache_plan_swaps_noalloc.
NOALLOC_MAX_L, NOALLOC_MAX_E, NOALLOC_MAX_LE, NOALLOC_MAX_KEYS = 1024, 1024, 32768, 16384


def cache_plan_swaps_noalloc(heat_dev, resid_dev, L: int, E: int, threshold: float, max_swaps: int, decay: float,
                             plan_dev, n_dev, stream=None) -> None:
    """Swap planning on caller-owned heat [L, E] (decayed in place) and residency [L, E] tables; allocates nothing."""
    if not (1 <= L <= NOALLOC_MAX_L and 1 <= E <= NOALLOC_MAX_E and L * E <= NOALLOC_MAX_LE
            and L * ((E + 1) // 2) <= NOALLOC_MAX_KEYS):
        raise ValueError(f"cache_plan_swaps_noalloc: L={L}, E={E} exceed the static scratch (L <= {NOALLOC_MAX_L}, "
                         f"E <= {NOALLOC_MAX_E}, L*E <= {NOALLOC_MAX_LE}, L*ceil(E/2) <= {NOALLOC_MAX_KEYS})")
    cfg = moe_policy_cfg(threshold, max_swaps, decay)
    _check(load().cache_plan_swaps_noalloc(_ptr(heat_dev), _ptr(resid_dev), L, E, C.byref(cfg), _ptr(plan_dev),
                                           _ptr(n_dev), _stream(stream)), "cache_plan_swaps_noalloc")


def cache_lru_plan(cache: Cache, ws: Workspace, layer: int, K: int, plan_dev, n_dev, stream=None) -> None:
    """After a layer call's grouping on ws: refresh its hits, plan its admissions into the K LRU victims."""
    _check(load().cache_lru_plan(cache.handle, ws.handle, layer, K, _ptr(plan_dev), _ptr(n_dev), _stream(stream)),
           "cache_lru_plan")


def moe_cache_apply_lru(cache: Cache, plan_dev, n_dev, compute=None, copy=None) -> None:
    _check(load().moe_cache_apply_lru(cache.handle, _ptr(plan_dev), _ptr(n_dev), _stream(compute), _stream(copy)),
           "moe_cache_apply_lru")


def moe_cache_apply_swaps(cache: Cache, plan_dev, n_dev, compute=None, copy=None) -> None:
    _check(load().moe_cache_apply_swaps(cache.handle, _ptr(plan_dev), _ptr(n_dev), _stream(compute),
                                        _stream(copy)), "moe_cache_apply_swaps")
