"""SwiGLU expert FFN, shared expert and weighted combine (oracle; test
infrastructure only).

* Routide §3.1: each expert has gate, up and down projections; MawForge §IV-C
  allows them separate or fused (here: separate).
* "Nanite for Experts" §1: eight routed experts plus one shared expert per
  token. The shared expert is added with weight one (no gate; the pages give
  none).
* "Nanite for Experts" §5.5: per-expert results merge back into their
  original output positions.

SwiGLU: h = silu(Wg x) * (Wu x), silu(z) = z / (1 + exp(-z)); y_e = Wd h.
Layer output: y[t] = sum_j w[t, j] * y_{idx[t, j]}(x[t]) + shared(x[t]).
All arithmetic is fp64.
"""
from __future__ import annotations

from typing import Callable, Optional, Tuple

import numpy as np

Mats = Tuple[np.ndarray, np.ndarray, np.ndarray]


def silu(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_ffn(mats: Mats, x: np.ndarray) -> np.ndarray:
    """mats = (Wg [I,H], Wu [I,H], Wd [H,I]) fp64; x [M, H] -> [M, H]."""
    wg, wu, wd = mats
    g = x @ wg.T
    u = x @ wu.T
    h = silu(g) * u
    return h @ wd.T


def moe_layer(x: np.ndarray, idx: np.ndarray, weights: np.ndarray,
              expert: Callable[[int], Mats], shared: Optional[Mats]) -> np.ndarray:
    """x fp64 [T, H]; idx [T, k]; weights [T, k]; expert(e) -> fp64 matrices."""
    T, H = x.shape
    y = np.zeros((T, H), dtype=np.float64)
    k = idx.shape[1]
    for e in sorted(set(int(v) for v in idx.ravel())):
        toks = [t for t in range(T) if e in set(int(v) for v in idx[t])]
        ye = expert_ffn(expert(e), x[toks])
        for r, t in enumerate(toks):
            j = [jj for jj in range(k) if int(idx[t, jj]) == e][0]
            y[t] += weights[t, j] * ye[r]
    if shared is not None:
        y += expert_ffn(shared, x)
    return y
