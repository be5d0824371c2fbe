"""Router: logits, top-k and combine weights (oracle; test infrastructure only).

Routing is authoritative ("Nanite for Experts" §3.1 and §9: native route ids
decide which experts execute; prediction may move data but never changes the
selection). Each token selects top-k of E routed experts (eight of 256 in
"Nanite for Experts" §1; top-eight in Routide §3.1).

The pages give no router formula, so this takes the plainest exact reading:

* logit l[t, e] is the correctly rounded fp64 value of the exact sum
  sum_i x[t, i] * W_r[e, i] (+ b[e]). Each product of a bf16/fp32 activation
  and an fp32 weight is exact in fp64, and ``math.fsum`` rounds the exact sum
  correctly;
* the k largest logits win; equal logits go to the lower expert id; the
  selection is listed by descending logit, then ascending id;
* combine weights are the softmax over the k selected logits, i.e. the softmax
  over all E renormalised to the selection, so they sum to one.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np


def router_logits(x: np.ndarray, w_router: np.ndarray,
                  bias: Optional[np.ndarray] = None) -> np.ndarray:
    """x fp64 [T, H] (exact activation values), w_router fp32 [E, H],
    bias fp32 [E] or None -> fp64 [T, E], each entry an fsum."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w_router, dtype=np.float32).astype(np.float64)
    T, H = x.shape
    E = w.shape[0]
    out = np.empty((T, E), dtype=np.float64)
    b = None if bias is None else np.asarray(bias, dtype=np.float32).astype(np.float64)
    for t in range(T):
        prods = (w * x[t][None, :]).tolist()  # exact products
        for e in range(E):
            terms = prods[e]
            if b is not None:
                terms = terms + [float(b[e])]
            out[t, e] = math.fsum(terms)
    return out


def topk_select(logits: np.ndarray, k: int) -> np.ndarray:
    """int32 [T, k]: per token the k largest logits, ties to the lower id,
    ordered by descending logit then ascending id."""
    T, E = logits.shape
    idx = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))
        idx[t] = order[:k]
    return idx


def combine_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """fp64 [T, k]: softmax over each token's selected logits."""
    T, k = idx.shape
    w = np.empty((T, k), dtype=np.float64)
    for t in range(T):
        sel = logits[t, idx[t]]
        z = np.exp(sel - sel.max())
        w[t] = z / z.sum()
    return w


def route(x: np.ndarray, w_router: np.ndarray, bias: Optional[np.ndarray], k: int):
    """(idx [T,k] int32, weights [T,k] fp64, logits [T,E] fp64)."""
    l = router_logits(x, w_router, bias)
    idx = topk_select(l, k)
    return idx, combine_weights(l, idx), l
