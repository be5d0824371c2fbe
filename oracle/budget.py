"""Static budget check (MawForge §IV-D) — test infrastructure only.

L(p, n) = C + E(p) + K(n) is the static lower bound of the serving footprint
F(p, n) = L(p, n) + O, with C the resident common tensor bytes, E(p) the
expert-cache budget at cache fraction p, K(n) the KV-cache bytes at context
length n and O the runtime overhead; a row whose lower bound already exceeds
the serving target is rejected.

Readings: p is given in parts per million, so every quantity is an integer
number of bytes; E(p) = floor(p * layers * experts * payload) (the pages'
static minima differ by exactly 15% of the total expert bytes between their
50% and 65% rows); the slots of one layer are floor(p * experts) (the slot
counts 38, 89 and 44 of the workloads); K(n) = bytes per token * n.
"""
from __future__ import annotations

PPM = 1_000_000


def static_budget(layers: int, experts: int, payload: int, cache_ppm: int, common: int,
                  kv_per_token: int, context: int, overhead: int, target: int) -> dict:
    if min(layers, experts, payload, cache_ppm, common, kv_per_token, context, overhead, target) < 0:
        raise ValueError("negative input")
    if cache_ppm > PPM:
        raise ValueError("cache fraction above 1")
    expert_bytes = layers * experts * payload * cache_ppm // PPM
    kv = kv_per_token * context
    lower = common + expert_bytes + kv
    return dict(common_bytes=common, expert_bytes=expert_bytes, kv_bytes=kv, overhead_bytes=overhead,
                lower_bound=lower, footprint=lower + overhead,
                slots_per_layer=experts * cache_ppm // PPM, accepted=int(lower <= target))
