"""Shared helpers of the GPU parity tests: seeded inputs from ``workloads``,
expected values from ``oracle`` only."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W


def tolerance_ok(y: np.ndarray, ref: np.ndarray):
    """The output bar: relative L2 <= 5e-3 and max |diff| <= 2e-2 * RMS(ref)."""
    ref = np.asarray(ref, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    rel = float(np.linalg.norm(y - ref) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(y - ref))) if y.size else 0.0
    return rel <= 5e-3 and mx <= 2e-2 * rms, rel, mx / max(rms, 1e-300)


def x_to_f64(w: W.Workload, x: np.ndarray) -> np.ndarray:
    return oracle.bf16_bits_to_f64(x) if w.x_dtype == "bf16" else x.astype(np.float64)


def x_to_torch(w: W.Workload, x: np.ndarray, device="cuda") -> torch.Tensor:
    if w.x_dtype == "bf16":
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).to(device)
    return torch.from_numpy(x.copy()).to(device)


def pinned_store(w: W.Workload, layers: int) -> torch.Tensor:
    t = torch.empty((layers, w.n_experts, w.payload_bytes), dtype=torch.uint8, pin_memory=True)
    W.fill_store(w, t.numpy())
    return t


class ExpertCache:
    """fp64 matrices of experts, dequantised by the oracle from generated payloads."""

    def __init__(self, w: W.Workload):
        self.w = w
        self.cache = {}

    def get(self, layer, e):
        key = (layer, e)
        if key not in self.cache:
            w = self.w
            inter = w.shared_inter if e == w.n_experts else w.inter
            self.cache[key] = oracle.expert_matrices(W.expert_payload(w, layer, e), w.hidden, inter,
                                                     w.quant)
        return self.cache[key]


def make_context(bec, w: W.Workload, layers: int, policy=None, slots=None, seed=0,
                 tile_bytes=262144, max_tokens=None, device_admit=False, decode_ffn=0):
    ctx = bec.Context(layers, w.n_experts, w.top_k, w.hidden, w.inter, w.shared_inter, w.quant,
                      slots or w.slots, w.policy if policy is None else policy, 3, seed,
                      tile_bytes, max_tokens or w.tokens_per_step, admit_on_device=device_admit,
                      decode_ffn=decode_ffn)
    return ctx


def bind_all(ctx, w: W.Workload, layers: int, store: torch.Tensor):
    ctx.bind_store(store)
    shared = []
    if w.shared_inter:
        for l in range(layers):
            p = torch.from_numpy(W.expert_payload(w, l, w.n_experts)).cuda()
            ctx.bind_shared(l, p)
            shared.append(p)
    return shared


def _route_rows(args):
    x64, wr, bias, k = args
    idx, w, _ = oracle.route(x64, wr, bias, k)
    return idx, w


def oracle_route_rows(x64: np.ndarray, wr: np.ndarray, bias, k: int, rows, workers: int = 0):
    """Oracle routing of the given token rows, split over a pool of worker
    processes started with ``spawn`` (a forked child of a process that has
    used the GPU can hang). Returns (idx [n,k], weights [n,k]) in row order."""
    import multiprocessing as mp
    import os
    rows = list(rows)
    n = len(rows)
    workers = workers or max(1, min(16, (os.cpu_count() or 1), n // 32))
    if workers <= 1 or n < 64:
        return _route_rows((x64[rows], wr, bias, k))
    parts = np.array_split(np.asarray(rows), workers)
    with mp.get_context("spawn").Pool(workers) as pool:
        res = pool.map(_route_rows, [(x64[p], wr, bias, k) for p in parts])
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])
