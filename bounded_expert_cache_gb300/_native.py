"""ctypes declarations of the libmoecache C ABI (include/moecache.h).

Argument marshalling only. Importing this module loads the in-tree
``libmoecache.so`` and raises ImportError if it is missing: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoecache.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_ARG", 2: "MOE_ERR_CUDA", 3: "MOE_ERR_CAPACITY",
                4: "MOE_ERR_STALE", 5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_UNCERTIFIED",
                7: "MOE_ERR_STATE"}
Q8_0, Q4_0, I4_G64 = 0, 1, 2
LRU, RANDOM, FARTHEST_NEXT_USE, STATIC_SET = 0, 1, 2, 3
F32, BF16 = 0, 1
MODE_AUTO, MODE_DECODE, MODE_PREFILL = 0, 1, 2
PREFETCH_OFF, PREFETCH_REFRESH, PREFETCH_PRESERVE = 0, 1, 2
PREFETCH_ACTIONS = ("probe", "refresh", "load")
KERNEL_KINDS = ("route", "plan", "ffn_gateup", "ffn_down", "stage_copy", "ffn_decode")


class Config(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("n_experts", C.c_int32), ("top_k", C.c_int32),
                ("hidden", C.c_int32), ("inter", C.c_int32), ("shared_inter", C.c_int32),
                ("quant", C.c_int32), ("slots_per_layer", C.c_int32), ("policy", C.c_int32),
                ("n_streams", C.c_int32), ("seed", C.c_uint64), ("tile_bytes", C.c_int64),
                ("max_tokens", C.c_int32), ("admit_on_device", C.c_int32), ("decode_ffn", C.c_int32)]


class PlanT(C.Structure):
    _fields_ = [("counts", C.c_void_p), ("offsets", C.c_void_p), ("uniq", C.c_void_p),
                ("n_uniq", C.c_void_p), ("perm_tok", C.c_void_p), ("perm_rank", C.c_void_p),
                ("perm_w", C.c_void_p), ("inv", C.c_void_p), ("capacity", C.c_int32)]


class MissList(C.Structure):
    _fields_ = [("n", C.c_int32), ("expert", C.POINTER(C.c_int32)), ("slot", C.POINTER(C.c_int32)),
                ("victim", C.POINTER(C.c_int32)), ("wave", C.POINTER(C.c_int32)),
                ("n_waves", C.c_int32), ("hits", C.c_int32), ("misses", C.c_int32),
                ("layer", C.c_int32)]


class Stats(C.Structure):
    _fields_ = [("steps", C.c_int64), ("hits", C.c_int64), ("misses", C.c_int64),
                ("evictions", C.c_int64), ("materialized_bytes", C.c_int64),
                ("tiles_staged", C.c_int64), ("bytes_staged", C.c_int64),
                ("uncertified_repairs", C.c_int64), ("prefetch_loads", C.c_int64),
                ("prefetch_useful", C.c_int64), ("prefetch_wasted", C.c_int64),
                ("prefetch_refreshes", C.c_int64), ("prefetch_probes", C.c_int64),
                ("prefetch_bytes", C.c_int64), ("route_filter_fallbacks", C.c_int64)]


class Budget(C.Structure):
    _fields_ = [("common_bytes", C.c_int64), ("expert_bytes", C.c_int64), ("kv_bytes", C.c_int64),
                ("overhead_bytes", C.c_int64), ("lower_bound", C.c_int64), ("footprint", C.c_int64),
                ("slots_per_layer", C.c_int32), ("accepted", C.c_int32)]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; "
            "g.build()' or python bounded_expert_cache_gb300/build.py). There is no fallback.")
    return C.CDLL(_LIB_PATH)


lib = _load()

_vp, _i32, _i64, _u64, _sz = C.c_void_p, C.c_int32, C.c_int64, C.c_uint64, C.c_size_t
_st = C.c_int  # moe_status_t

# (name, restype, argtypes) for every symbol of include/moecache.h
SIGNATURES = [
    ("moe_create", _st, [C.POINTER(Config), C.POINTER(_vp)]),
    ("moe_destroy", None, [_vp]),
    ("moe_last_error", C.c_char_p, [_vp]),
    ("moe_payload_bytes", _i64, [_vp]),
    ("moe_shared_payload_bytes", _i64, [_vp]),
    ("moe_bind_store", _st, [_vp, _vp, _sz]),
    ("moe_bind_shared", _st, [_vp, _i32, _vp]),
    ("moe_route", _st, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    ("moe_route_noalloc", _st, [_vp, _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    ("moe_plan_union", _st, [_vp, _vp, _vp, _i32, C.POINTER(PlanT), _vp]),
    ("moe_cache_admit", _st, [_vp, _i32, C.POINTER(PlanT), C.POINTER(MissList), _vp]),
    ("moe_cache_evict", _st, [_vp, _i32, _i32]),
    ("moe_cache_preload", _st, [_vp, _i32, C.POINTER(_i32), _i32]),
    ("moe_stage_tiles", _st, [_vp, _i32, C.POINTER(MissList), _vp]),
    ("moe_expert_ffn", _st, [_vp, _i32, _vp, _i32, _i32, C.POINTER(PlanT), _vp, _i32, _vp]),
    ("moe_layer_forward", _st, [_vp, _i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, C.POINTER(PlanT),
                                _vp, C.POINTER(MissList), _vp]),
    ("moe_set_prefetch", _st, [_vp, _i32, C.c_float]),
    ("moe_check_device_errors", _st, [_vp, _vp]),
    ("moe_get_stats", _st, [_vp, _i32, C.POINTER(Stats)]),
    ("moe_read_page_table", _st, [_vp, _i32, C.POINTER(_i32), C.POINTER(C.c_uint32)]),
    ("moe_read_slot", _st, [_vp, _i32, _i32, _vp, _sz]),
    ("moe_set_kernel_timing", _st, [_vp, _i32]),
    ("moe_get_kernel_times", _st, [_vp, C.POINTER(C.c_double), C.POINTER(_i64)]),
    ("moe_debug_fail_staging_after", _st, [_vp, _i32]),
    ("moe_debug_corrupt_generation", _st, [_vp, _i32, _i32]),
    ("moe_debug_prefill_wait_timeout", _st, [_vp, _i64, _i32]),
    ("moe_slots_create", _st, [_i32, _i32, _i32, _u64, _i32, _i64, C.POINTER(_vp)]),
    ("moe_slots_destroy", None, [_vp]),
    ("moe_slots_step", _st, [_vp, C.POINTER(_i32), _i32, C.POINTER(_i32), C.POINTER(MissList)]),
    ("moe_slots_prefetch", _st, [_vp, _i32, _i32, C.POINTER(_i32), C.POINTER(MissList)]),
    ("moe_slots_preload", _st, [_vp, C.POINTER(_i32), _i32]),
    ("moe_slots_evict", _st, [_vp, _i32]),
    ("moe_slots_read", _st, [_vp, C.POINTER(_i32), C.POINTER(C.c_uint32)]),
    ("moe_slots_stats", _st, [_vp, C.POINTER(Stats)]),
    ("moe_splitmix64_next", _u64, [C.POINTER(_u64)]),
    ("moe_replay", _st, [_i32, _i32, _i32, _u64, _i32, C.c_int64, _i32, _i32, _i32, C.POINTER(_i32),
                         C.POINTER(_i32), C.POINTER(_i32), C.POINTER(Stats)]),
    ("moe_static_budget", _st, [_i32, _i32, C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_int64, C.c_int64,
                                C.c_int64, C.POINTER(Budget)]),
]

for _name, _res, _args in SIGNATURES:
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args
