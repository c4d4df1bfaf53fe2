"""Slot-addressed expert-cache MoE layer for GB300 (sm_103a).

The compute path lives in ``libmoe.so`` (hand-written CUDA behind a C ABI,
``include/moe.h``); :mod:`serving_router_top_gb300.moe` is the thin ctypes
binding with the same names.  Importing this package does not load the
library; the binding loads it on first use and raises if it is missing.
"""
__all__ = ["inputs"]
