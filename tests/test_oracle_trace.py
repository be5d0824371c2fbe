"""Pin of the oracle's per-step layer replay (route -> union -> cache -> FFN).

The trace is built so that every value is known by hand: router rows are unit
vectors, so a token x = 2 e_a + e_b has logits 2 (expert a), 1 (expert b) and
0 elsewhere; top-2 is [a, b] with weights e/(e+1) and 1/(e+1). The cache
records follow the rules of the slot cache worked by hand below (LRU, 3
slots); the FFN uses experts with closed-form outputs.
"""
import math

import numpy as np

from oracle.cache import LRU, SlotCache
from oracle.trace import replay_layer

E, H, K, S = 6, 8, 2, 3
PAIRS = [(0, 1), (2, 1), (4, 3), (5, 1)]  # (top expert, second expert) per step


def _inputs():
    wr = np.zeros((E, H), dtype=np.float32)
    for e in range(E):
        wr[e, e] = 1.0
    xs = []
    for a, b in PAIRS:
        x = np.zeros((1, H))
        x[0, a], x[0, b] = 2.0, 1.0
        xs.append(x)
    return wr, xs


# Hand-worked LRU replay (access order: resident experts ascending, then
# missing ones ascending; a miss takes the lowest free slot, else the slot
# with the oldest access):
#   step 0, union {0,1}: 0 -> slot 0 (tick 1), 1 -> slot 1 (tick 2)
#   step 1, union {1,2}: hit 1 (tick 3); 2 -> free slot 2 (tick 4)
#   step 2, union {3,4}: 3 evicts 0 from slot 0 (oldest, tick 1) at tick 5;
#                        4 evicts 1 from slot 1 (tick 3) at tick 6
#   step 3, union {1,5}: 1 evicts 2 from slot 2 (tick 4) at tick 7;
#                        5 evicts 3 from slot 0 (tick 5) at tick 8
HAND = [
    dict(hits=0, misses=2, fills=[(0, 0, -1), (1, 1, -1)], pt=[0, 1, -1, -1, -1, -1], gen=[1, 1, 0]),
    dict(hits=1, misses=1, fills=[(2, 2, -1)], pt=[0, 1, 2, -1, -1, -1], gen=[1, 1, 1]),
    dict(hits=0, misses=2, fills=[(3, 0, 0), (4, 1, 1)], pt=[-1, -1, 2, 0, 1, -1], gen=[2, 2, 1]),
    dict(hits=0, misses=2, fills=[(1, 2, 2), (5, 0, 3)], pt=[-1, 2, -1, -1, 1, 0], gen=[3, 2, 2]),
]

C = math.log(3.0)


def _expert(e):
    # gate = C * identity, up = identity, down = (e + 1) * identity:
    # y_e(x) = (e + 1) * silu(C x) * x elementwise
    eye = np.eye(H)
    return C * eye, eye, (e + 1) * eye


def test_replay_layer_matches_hand_worked_trace():
    wr, xs = _inputs()
    cache = SlotCache(E, S, LRU, payload_bytes=100)
    recs = replay_layer(xs, wr, None, K, cache, expert=_expert)
    wa, wb = math.e / (math.e + 1.0), 1.0 / (math.e + 1.0)
    # silu(2C) * 2 at the top expert's coordinate, silu(C) * 1 at the second's:
    # silu(ln 3) = (3/4) ln 3 and silu(2 ln 3) = (9/10) 2 ln 3
    top_val, second_val = 2.0 * 1.8 * C, 0.75 * C
    for s, ((a, b), rec, hand) in enumerate(zip(PAIRS, recs, HAND)):
        assert rec["idx"].tolist() == [[a, b]], s
        assert np.allclose(rec["w"], [[wa, wb]], rtol=0, atol=1e-15), s
        assert rec["plan"]["uniq"].tolist() == sorted((a, b)), s
        for key in ("hits", "misses", "pt", "gen"):
            assert rec["cache"][key] == hand[key], (s, key)
        assert [tuple(f) for f in rec["cache"]["fills"]] == hand["fills"], s
        factor = wa * (a + 1) + wb * (b + 1)
        want = np.zeros((1, H))
        want[0, a], want[0, b] = factor * top_val, factor * second_val
        assert np.allclose(rec["y"], want, rtol=1e-14, atol=0), s
    assert cache.stats() == dict(hits=1, misses=7, evictions=4, materialized_bytes=700)


def test_replay_layer_ffn_only_on_requested_steps():
    wr, xs = _inputs()
    recs = replay_layer(xs, wr, None, K, SlotCache(E, S, LRU), expert=_expert, ffn_steps={1, 3})
    assert ["y" in r for r in recs] == [False, True, False, True]
    recs = replay_layer(xs, wr, None, K, SlotCache(E, S, LRU))
    assert not any("y" in r for r in recs)


# Confidence-gated prefetch ("Paging the Experts" §3.3) in the resident-refresh
# mode: before each step the previous step's top expert (weight e/(e+1) >= 0.20
# here) is touched if resident. Hand-worked LRU replay on 3 slots:
#   step 0, union {0,1}: 0 -> slot 0 (tick 1), 1 -> slot 1 (tick 2); predict 0
#   step 1: refresh 0 (tick 3); union {2,3}: 2 -> free slot 2 (tick 4),
#           3 evicts 1 from slot 1 (oldest, tick 2) at tick 5; predict 2
#   step 2: refresh 2 (tick 6); union {0,4}: hit 0 (tick 7), 4 evicts 3 from
#           slot 1 (tick 5) at tick 8; predict 0
#   step 3: refresh 0 (tick 9); union {1,5}: 1 evicts 2 from slot 2 (tick 6)
#           at tick 10, 5 evicts 4 from slot 1 (tick 8) at tick 11
# Without the refreshes step 1 would evict 0 (tick 1) instead of 1, and step 2
# would miss twice.
PAIRS_PF = [(0, 1), (2, 3), (0, 4), (1, 5)]
HAND_PF = [
    dict(hits=0, misses=2, fills=[(0, 0, -1), (1, 1, -1)], pt=[0, 1, -1, -1, -1, -1], gen=[1, 1, 0]),
    dict(hits=0, misses=2, fills=[(2, 2, -1), (3, 1, 1)], pt=[0, -1, 2, 1, -1, -1], gen=[1, 2, 1]),
    dict(hits=1, misses=1, fills=[(4, 1, 3)], pt=[0, -1, 2, -1, 1, -1], gen=[1, 3, 1]),
    dict(hits=0, misses=2, fills=[(1, 2, 2), (5, 1, 4)], pt=[0, 2, -1, -1, -1, 1], gen=[1, 4, 2]),
]


def _inputs_pf():
    wr, _ = _inputs()
    xs = []
    for a, b in PAIRS_PF:
        x = np.zeros((1, H))
        x[0, a], x[0, b] = 2.0, 1.0
        xs.append(x)
    return wr, xs


def test_replay_layer_with_resident_refresh_prefetch():
    from oracle.cache import PREFETCH_PRESERVE, PREFETCH_REFRESH
    wr, xs = _inputs_pf()
    cache = SlotCache(E, S, LRU, payload_bytes=100)
    recs = replay_layer(xs, wr, None, K, cache, prefetch=PREFETCH_REFRESH)
    assert [r["prefetch"] and (r["prefetch"]["action"], r["prefetch"]["expert"]) for r in recs] == \
        [None, ("refresh", 0), ("refresh", 2), ("refresh", 0)]
    for s, (rec, hand) in enumerate(zip(recs, HAND_PF)):
        for key in ("hits", "misses", "pt", "gen"):
            assert rec["cache"][key] == hand[key], (s, key)
        assert [tuple(f) for f in rec["cache"]["fills"]] == hand["fills"], s
    assert cache.stats() == dict(hits=1, misses=7, evictions=4, materialized_bytes=700)
    assert cache.prefetch_stats() == dict(loads=0, useful=0, wasted=0, refreshes=3, probes=0, bytes=0)
    # preserve-resident probes leave the cache exactly as demand-only replay
    plain = replay_layer(xs, wr, None, K, SlotCache(E, S, LRU))
    kept = SlotCache(E, S, LRU)
    pres = replay_layer(xs, wr, None, K, kept, prefetch=PREFETCH_PRESERVE)
    assert [r["cache"] for r in pres] == [r["cache"] for r in plain]
    assert kept.prefetch_stats()["probes"] == 3
    # the rule's threshold: top weight e/(e+1) = 0.731 fires at 0.73, not at 0.74
    assert replay_layer(xs, wr, None, K, SlotCache(E, S, LRU), prefetch=PREFETCH_REFRESH,
                        threshold=0.74)[1]["prefetch"] is None
    assert replay_layer(xs, wr, None, K, SlotCache(E, S, LRU), prefetch=PREFETCH_REFRESH,
                        threshold=0.73)[1]["prefetch"] is not None
