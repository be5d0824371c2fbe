"""Thin Python binding over the libmoecache C ABI.

Marshals torch tensors into pointers and raises MoeError on a non-OK status.
PyTorch supplies device memory, pinned host memory and streams; every step of
the path runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass
from typing import List, Optional

import torch

from . import _native as N
from ._native import lib


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{N.STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(st: int, ctx_ptr=None):
    if st != N.MOE_OK:
        m = lib.moe_last_error(ctx_ptr)
        raise MoeError(st, (m or b"").decode(errors="replace"))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _xt(x: torch.Tensor) -> int:
    if x.dtype == torch.float32:
        return N.F32
    if x.dtype in (torch.bfloat16, torch.int16, torch.uint16):
        return N.BF16
    raise TypeError(f"activations must be float32 or bfloat16 (got {x.dtype})")


@dataclass
class Misses:
    """Host copy of one cache resolve's fill list."""
    expert: List[int]
    slot: List[int]
    victim: List[int]
    wave: List[int]
    n_waves: int
    hits: int
    misses: int
    layer: int
    raw: N.MissList


class Plan:
    """Device arrays of an expert-major plan for up to ``max_tokens`` tokens."""

    def __init__(self, n_experts: int, top_k: int, max_tokens: int, device=None):
        dev = device or torch.device("cuda")
        A = max_tokens * top_k
        i32 = dict(dtype=torch.int32, device=dev)
        self.counts = torch.zeros(n_experts, **i32)
        self.offsets = torch.zeros(n_experts + 1, **i32)
        self.uniq = torch.zeros(n_experts, **i32)
        self.n_uniq = torch.zeros(1, **i32)
        self.perm_tok = torch.zeros(A, **i32)
        self.perm_rank = torch.zeros(A, **i32)
        self.perm_w = torch.zeros(A, dtype=torch.float32, device=dev)
        self.inv = torch.zeros(A, **i32)
        self.raw = N.PlanT(self.counts.data_ptr(), self.offsets.data_ptr(), self.uniq.data_ptr(),
                           self.n_uniq.data_ptr(), self.perm_tok.data_ptr(),
                           self.perm_rank.data_ptr(), self.perm_w.data_ptr(), self.inv.data_ptr(),
                           A)


class Context:
    """One moe_ctx_t on the current CUDA device."""

    def __init__(self, n_layers, n_experts, top_k, hidden, inter, shared_inter=0, quant=N.Q8_0,
                 slots_per_layer=None, policy=N.LRU, n_streams=3, seed=0, tile_bytes=262144,
                 max_tokens=8, admit_on_device=0, decode_ffn=0):
        self.cfg = N.Config(n_layers, n_experts, top_k, hidden, inter, shared_inter, quant,
                            slots_per_layer or n_experts, policy, n_streams, seed, tile_bytes,
                            max_tokens, int(admit_on_device), int(decode_ffn))
        h = C.c_void_p()
        _check(lib.moe_create(C.byref(self.cfg), C.byref(h)), None)
        self.h = h
        self._keep = []

    def close(self):
        if self.h:
            lib.moe_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _ck(self, st):
        _check(st, self.h)

    @property
    def payload_bytes(self) -> int:
        return lib.moe_payload_bytes(self.h)

    @property
    def shared_payload_bytes(self) -> int:
        return lib.moe_shared_payload_bytes(self.h)

    def bind_store(self, store: torch.Tensor):
        assert store.dtype == torch.uint8 and store.is_pinned() and store.is_contiguous()
        self._ck(lib.moe_bind_store(self.h, _ptr(store), store.numel()))
        self._keep.append(store)

    def bind_shared(self, layer: int, payload: torch.Tensor):
        assert payload.is_cuda and payload.dtype == torch.uint8
        self._ck(lib.moe_bind_shared(self.h, layer, _ptr(payload)))
        self._keep.append(payload)

    def route(self, layer, x, w_router, bias, topk_idx, topk_w, stream=None):
        self._ck(lib.moe_route(self.h, layer, _ptr(x), _xt(x), x.shape[0], _ptr(w_router),
                               _ptr(bias), _ptr(topk_idx), _ptr(topk_w), _stream(stream)))

    def plan_union(self, topk_idx, topk_w, T, plan: Plan, stream=None):
        self._ck(lib.moe_plan_union(self.h, _ptr(topk_idx), _ptr(topk_w), T, C.byref(plan.raw),
                                    _stream(stream)))

    def cache_admit(self, layer, plan: Plan, stream=None) -> Misses:
        ml = N.MissList()
        self._ck(lib.moe_cache_admit(self.h, layer, C.byref(plan.raw), C.byref(ml), _stream(stream)))
        return _misses(ml)

    def stage_tiles(self, layer, misses: Misses, stream=None):
        self._ck(lib.moe_stage_tiles(self.h, layer, C.byref(misses.raw), _stream(stream)))

    def expert_ffn(self, layer, x, plan: Plan, y, mode=N.MODE_AUTO, stream=None):
        self._ck(lib.moe_expert_ffn(self.h, layer, _ptr(x), _xt(x), x.shape[0], C.byref(plan.raw),
                                    _ptr(y), mode, _stream(stream)))

    def layer_forward(self, layer, x, w_router, bias, topk_idx, topk_w, plan: Plan, y,
                      stream=None) -> Misses:
        ml = N.MissList()
        self._ck(lib.moe_layer_forward(self.h, layer, _ptr(x), _xt(x), x.shape[0], _ptr(w_router),
                                       _ptr(bias), _ptr(topk_idx), _ptr(topk_w), C.byref(plan.raw),
                                       _ptr(y), C.byref(ml), _stream(stream)))
        return _misses(ml)

    def check_device_errors(self, stream=None):
        self._ck(lib.moe_check_device_errors(self.h, _stream(stream)))

    def evict(self, layer, expert):
        self._ck(lib.moe_cache_evict(self.h, layer, expert))

    def preload(self, layer, experts):
        arr = (C.c_int32 * len(experts))(*experts)
        self._ck(lib.moe_cache_preload(self.h, layer, arr, len(experts)))

    def stats(self, layer=-1) -> dict:
        s = N.Stats()
        self._ck(lib.moe_get_stats(self.h, layer, C.byref(s)))
        return {f: getattr(s, f) for f, _ in N.Stats._fields_}

    def read_page_table(self, layer):
        E, S = self.cfg.n_experts, self.cfg.slots_per_layer
        pt = (C.c_int32 * E)()
        gen = (C.c_uint32 * S)()
        self._ck(lib.moe_read_page_table(self.h, layer, pt, gen))
        return list(pt), list(gen)

    def read_slot(self, layer, slot, nbytes=None) -> bytes:
        n = nbytes or self.payload_bytes
        buf = (C.c_uint8 * n)()
        self._ck(lib.moe_read_slot(self.h, layer, slot, buf, n))
        return bytes(buf)

    def set_kernel_timing(self, enable: bool):
        self._ck(lib.moe_set_kernel_timing(self.h, 1 if enable else 0))

    def kernel_times(self) -> dict:
        """{kind: (total_ms, launches)} since the last call; synchronises."""
        ms = (C.c_double * len(N.KERNEL_KINDS))()
        n = (C.c_int64 * len(N.KERNEL_KINDS))()
        self._ck(lib.moe_get_kernel_times(self.h, ms, n))
        return {k: (ms[i], n[i]) for i, k in enumerate(N.KERNEL_KINDS)}

    def set_prefetch(self, mode: int, threshold: float = 0.2):
        """Confidence-gated prefetch before every layer step (host admission)."""
        self._ck(lib.moe_set_prefetch(self.h, mode, threshold))

    def debug_fail_staging_after(self, n_tiles: int):
        self._ck(lib.moe_debug_fail_staging_after(self.h, n_tiles))

    def debug_corrupt_generation(self, layer, expert):
        self._ck(lib.moe_debug_corrupt_generation(self.h, layer, expert))

    def debug_prefill_wait_timeout(self, wait_cycles: int, skip_ring: int):
        self._ck(lib.moe_debug_prefill_wait_timeout(self.h, wait_cycles, skip_ring))


def _misses(ml: N.MissList) -> Misses:
    n = ml.n
    return Misses([ml.expert[i] for i in range(n)], [ml.slot[i] for i in range(n)],
                  [ml.victim[i] for i in range(n)], [ml.wave[i] for i in range(n)], ml.n_waves,
                  ml.hits, ml.misses, ml.layer, ml)


class Slots:
    """The host slot manager alone (no CUDA calls)."""

    def __init__(self, n_experts, n_slots, policy=N.LRU, seed=0, layer=0, payload_bytes=0):
        h = C.c_void_p()
        _check(lib.moe_slots_create(n_experts, n_slots, policy, seed, layer, payload_bytes,
                                    C.byref(h)))
        self.h = h
        self.E, self.S = n_experts, n_slots

    def __del__(self):
        if getattr(self, "h", None):
            lib.moe_slots_destroy(self.h)
            self.h = None

    def step(self, uniq, counts) -> Misses:
        u = (C.c_int32 * max(1, len(uniq)))(*uniq)
        cnt = (C.c_int32 * self.E)(*counts)
        ml = N.MissList()
        _check(lib.moe_slots_step(self.h, u, len(uniq), cnt, C.byref(ml)))
        return _misses(ml)

    def prefetch(self, expert, mode):
        """Speculative access before the next step: returns (action, fill)
        with action "probe", "refresh" or "load" and fill (expert, slot,
        victim) of a load, else None."""
        act = C.c_int32()
        ml = N.MissList()
        _check(lib.moe_slots_prefetch(self.h, expert, mode, C.byref(act), C.byref(ml)))
        fill = (ml.expert[0], ml.slot[0], ml.victim[0]) if ml.n else None
        return N.PREFETCH_ACTIONS[act.value], fill

    def preload(self, experts):
        arr = (C.c_int32 * max(1, len(experts)))(*experts)
        _check(lib.moe_slots_preload(self.h, arr, len(experts)))

    def evict(self, e):
        _check(lib.moe_slots_evict(self.h, e))

    def read(self):
        pt = (C.c_int32 * self.E)()
        gen = (C.c_uint32 * self.S)()
        _check(lib.moe_slots_read(self.h, pt, gen))
        return list(pt), list(gen)

    def stats(self) -> dict:
        s = N.Stats()
        _check(lib.moe_slots_stats(self.h, C.byref(s)))
        return {f: getattr(s, f) for f, _ in N.Stats._fields_}


def replay(policy, n_experts, n_slots, steps, payload=0, seed=0, layer=0, width=0, calib=0) -> dict:
    """Offline replay of one layer's steps (moe_replay); steps: a list of
    (union, counts[E]) as for Slots.step. Returns the counters."""
    offs, ex, cn = [0], [], []
    for uniq, counts in steps:
        for e in uniq:
            ex.append(int(e))
            cn.append(int(counts[int(e)]))
        offs.append(len(ex))
    n = len(steps)
    o = (C.c_int32 * (n + 1))(*offs)
    e_arr = (C.c_int32 * max(1, len(ex)))(*ex)
    c_arr = (C.c_int32 * max(1, len(cn)))(*cn)
    st = N.Stats()
    _check(lib.moe_replay(policy, n_experts, n_slots, seed, layer, payload, width, calib, n, o, e_arr, c_arr,
                          C.byref(st)))
    return {f: getattr(st, f) for f, _ in N.Stats._fields_}


def static_budget(n_layers, n_experts, payload_bytes, cache_ppm, common_bytes=0, kv_bytes_per_token=0,
                  context=0, overhead_bytes=0, target_bytes=0) -> dict:
    """Static budget check before serving (moe_static_budget): the lower
    bound C + E(p) + K(n), the footprint with the overhead, the slots per
    layer and whether the row fits the target."""
    b = N.Budget()
    _check(lib.moe_static_budget(n_layers, n_experts, payload_bytes, cache_ppm, common_bytes,
                                 kv_bytes_per_token, context, overhead_bytes, target_bytes, C.byref(b)))
    return {f: getattr(b, f) for f, _ in N.Budget._fields_}


def splitmix64(state: int, n: int) -> List[int]:
    s = C.c_uint64(state)
    return [lib.moe_splitmix64_next(C.byref(s)) for _ in range(n)]
