"""bounded_expert_cache_gb300 — a routed MoE FFN layer over a bounded,
page-table-addressed cache of quantised expert slots, for one GB300 (sm_103a).

The compute path is the in-tree CUDA library ``libmoecache.so`` (C ABI in
``include/moecache.h``); this package only marshals arguments to it. Importing
it fails if the library has not been built.
"""
from . import _native
from ._native import (Q8_0, Q4_0, I4_G64, LRU, RANDOM, FARTHEST_NEXT_USE, STATIC_SET, F32, BF16, MODE_AUTO, MODE_DECODE,
                      MODE_PREFILL, PREFETCH_OFF, PREFETCH_REFRESH, PREFETCH_PRESERVE)
from .api import Context, Plan, Slots, Misses, MoeError, splitmix64, static_budget, replay

__all__ = ["Context", "Plan", "Slots", "Misses", "MoeError", "splitmix64", "static_budget", "replay",
           "FARTHEST_NEXT_USE", "STATIC_SET", "Q8_0", "Q4_0", "I4_G64", "LRU",
           "RANDOM", "F32", "BF16", "MODE_AUTO", "MODE_DECODE", "MODE_PREFILL", "PREFETCH_OFF",
           "PREFETCH_REFRESH", "PREFETCH_PRESERVE"]
