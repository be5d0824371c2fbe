"""Step-by-step replay of one layer over a trace (oracle; test infrastructure only).

Per layer and step, in the order of the path: route (authoritative, "Nanite
for Experts" §3.1) -> expert-major union (§5.3) -> cache resolve with
admission of misses into slots (MawForge §IV-C, Routide §3.2/§4.1) -> FFN and
combine (fp64, optional). Layers keep separate caches (per-layer slot tensors,
MawForge §IV-C), so a layer can be replayed on its own.
"""
from __future__ import annotations

from typing import Callable, List, Optional

import numpy as np

from .cache import SlotCache
from .ffn import moe_layer
from .plan import plan_union
from .route import route


def replay_layer(x_steps: List[np.ndarray], w_router: np.ndarray,
                 bias: Optional[np.ndarray], k: int, cache: SlotCache,
                 expert: Optional[Callable] = None, shared=None,
                 ffn_steps: Optional[set] = None) -> List[dict]:
    """x_steps: fp64 [T, H] per step. Returns one record per step with idx,
    weights, plan, the cache record and (for steps in ffn_steps, or all steps
    when ffn_steps is None and ``expert`` is given) the fp64 output y."""
    out = []
    E = w_router.shape[0]
    for s, x in enumerate(x_steps):
        idx, w, _ = route(x, w_router, bias, k)
        plan = plan_union(idx, w, E)
        rec = cache.step(plan["uniq"], plan["counts"])
        r = dict(idx=idx, w=w, plan=plan, cache=rec)
        if expert is not None and (ffn_steps is None or s in ffn_steps):
            r["y"] = moe_layer(x, idx, w, expert, shared)
        out.append(r)
    return out
