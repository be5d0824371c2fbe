"""Expert-major union and permutation (oracle; test infrastructure only).

"Nanite for Experts" §5.3 and §11.3: instead of moving an expert once per
token position, union the expert ids across the window and schedule each
unique expert once. §5.5: results merge back into their original output
positions.

Reading of the order, which the page leaves open: the union is listed by
ascending expert id; each expert's assignments are listed by ascending token
(a token selects an expert at most once).
"""
from __future__ import annotations

import numpy as np


def plan_union(idx: np.ndarray, weights: np.ndarray, n_experts: int) -> dict:
    """idx int [T, k], weights [T, k] -> expert-major plan.

    Returns counts[E], offsets[E+1] (exclusive scan of counts), uniq (experts
    with a non-zero count, ascending), perm_tok/perm_rank/perm_w [T*k]
    (assignment p is token perm_tok[p]'s perm_rank[p]-th choice, with weight
    perm_w[p]) and inv [T*k] (inv[t*k + j] = p for that assignment).
    """
    T, k = idx.shape
    lists = {e: [] for e in range(n_experts)}
    for t in range(T):
        for j in range(k):
            lists[int(idx[t, j])].append((t, j))
    counts = np.array([len(lists[e]) for e in range(n_experts)], dtype=np.int32)
    offsets = np.zeros(n_experts + 1, dtype=np.int32)
    offsets[1:] = np.cumsum(counts)
    uniq = np.array([e for e in range(n_experts) if counts[e] > 0], dtype=np.int32)
    perm_tok = np.empty(T * k, dtype=np.int32)
    perm_rank = np.empty(T * k, dtype=np.int32)
    perm_w = np.empty(T * k, dtype=np.float64)
    inv = np.empty(T * k, dtype=np.int32)
    p = 0
    for e in range(n_experts):
        for (t, j) in sorted(lists[e]):
            perm_tok[p] = t
            perm_rank[p] = j
            perm_w[p] = weights[t, j]
            inv[t * k + j] = p
            p += 1
    return dict(counts=counts, offsets=offsets, uniq=uniq, perm_tok=perm_tok,
                perm_rank=perm_rank, perm_w=perm_w, inv=inv)
