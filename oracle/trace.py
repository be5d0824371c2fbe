"""Step-by-step replay of one layer over a trace (oracle; test infrastructure only).

Per layer and step, in the order of the path: the optional confidence-gated
prefetch of the previous step's prediction ("Paging the Experts" §3.3) ->
route (authoritative, "Nanite for Experts" §3.1) -> expert-major union
(§5.3) -> cache resolve with admission of misses into slots (MawForge §IV-C,
Routide §3.2/§4.1) -> FFN and combine (fp64, optional). Layers keep separate
caches (per-layer slot tensors, MawForge §IV-C), so a layer can be replayed
on its own.
"""
from __future__ import annotations

from typing import Callable, List, Optional

import numpy as np

from .cache import SlotCache
from .ffn import moe_layer
from .plan import plan_union
from .prefetch import THRESHOLD, prediction
from .route import route


def replay_layer(x_steps: List[np.ndarray], w_router: np.ndarray,
                 bias: Optional[np.ndarray], k: int, cache: SlotCache,
                 expert: Optional[Callable] = None, shared=None,
                 ffn_steps: Optional[set] = None, prefetch: int = 0,
                 threshold: float = THRESHOLD) -> List[dict]:
    """x_steps: fp64 [T, H] per step. Returns one record per step with idx,
    weights, plan, the cache record, the prefetch taken before the step
    (None, or the cache's prefetch record with the expert) and (for steps in
    ffn_steps, or all steps when ffn_steps is None and ``expert`` is given)
    the fp64 output y. prefetch: 0 off, else PREFETCH_REFRESH or
    PREFETCH_PRESERVE with the previous step's prediction."""
    out = []
    E = w_router.shape[0]
    pred = None
    for s, x in enumerate(x_steps):
        pf = None
        if prefetch and pred is not None:
            pf = dict(cache.prefetch(pred, prefetch), expert=pred)
        idx, w, _ = route(x, w_router, bias, k)
        plan = plan_union(idx, w, E)
        rec = cache.step(plan["uniq"], plan["counts"])
        pred = prediction(idx, w, threshold)
        r = dict(idx=idx, w=w, plan=plan, cache=rec, prefetch=pf)
        if expert is not None and (ffn_steps is None or s in ffn_steps):
            r["y"] = moe_layer(x, idx, w, expert, shared)
        out.append(r)
    return out
