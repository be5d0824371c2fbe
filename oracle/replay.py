"""Offline replays of one layer's step sequence under other cache policies —
test infrastructure only.

"Paging the Experts" (Routide) §2 treats farthest-next-use as an offline
paging reference (it needs future routing), and §5.1 compares policies on
fixed route replays; "Nanite for Experts" §5.6/§7.4 serve from a learned,
static working set of 16 (or 20) experts per layer instead of rolling
replacement.

Readings: a step is one layer evaluation with union U (all of it pinned, as
in the slot cache's step); hits = assignments - missing experts.
* farthest next use: resident experts are touched first, then the missing
  experts of U are admitted in ascending id; a miss takes the lowest free
  slot, else evicts the resident expert outside U whose next step of use is
  the farthest (never again counts as infinitely far; ties to the lower
  slot index).
* static working set of width W: the W experts with the most assignments
  over the first `calib` steps (ties to the lower id) are resident before
  the first step (not counted) and never evicted; any other expert of a
  step is a miss, materialised for that step and not admitted.
LRU and seeded random replay through SlotCache.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

from .cache import LRU, RANDOM, CapacityError, SlotCache

FARTHEST_NEXT_USE = 2
STATIC_SET = 3

Step = Tuple[Sequence[int], Sequence[int]]  # (union, counts[E])


def static_set(steps: List[Step], n_experts: int, width: int, calib: int) -> List[int]:
    total = [0] * n_experts
    for uniq, counts in steps[:calib]:
        for e in uniq:
            total[int(e)] += int(counts[int(e)])
    order = sorted(range(n_experts), key=lambda e: (-total[e], e))
    return sorted(order[:width])


def replay(policy: int, n_experts: int, n_slots: int, steps: List[Step], payload: int = 0, seed: int = 0,
           layer: int = 0, width: int = 0, calib: int = 0) -> dict:
    if policy in (LRU, RANDOM):
        c = SlotCache(n_experts, n_slots, policy, seed=seed, layer=layer, payload_bytes=payload)
        for uniq, counts in steps:
            c.step(uniq, counts)
        return c.stats()
    hits = misses = evictions = 0
    if policy == STATIC_SET:
        if width > n_slots:
            raise CapacityError("static set wider than the slots")
        keep = set(static_set(steps, n_experts, width, calib))
        for uniq, counts in steps:
            m = sum(1 for e in uniq if int(e) not in keep)
            misses += m
            hits += sum(int(counts[int(e)]) for e in uniq) - m
        return dict(hits=hits, misses=misses, evictions=0, materialized_bytes=misses * payload)
    if policy != FARTHEST_NEXT_USE:
        raise ValueError("unknown policy")
    sets = [set(int(e) for e in uniq) for uniq, _ in steps]
    owner = [-1] * n_slots
    where = [-1] * n_experts

    def next_use(e: int, t: int) -> float:
        for u in range(t + 1, len(steps)):
            if e in sets[u]:
                return u
        return float("inf")

    for t, (uniq, counts) in enumerate(steps):
        U = sorted(sets[t])
        if len(U) > n_slots:
            raise CapacityError("union larger than the slots")
        missing = [e for e in U if where[e] < 0]
        for e in missing:
            free = [s for s in range(n_slots) if owner[s] < 0]
            if free:
                s = free[0]
            else:
                cand = [s for s in range(n_slots) if owner[s] not in sets[t]]
                s = max(cand, key=lambda q: (next_use(owner[q], t), -q))
                where[owner[s]] = -1
                evictions += 1
            owner[s] = e
            where[e] = s
        misses += len(missing)
        hits += sum(int(counts[e]) for e in U) - len(missing)
    return dict(hits=hits, misses=misses, evictions=evictions, materialized_bytes=misses * payload)
