"""Pins for the oracle's slot cache, SplitMix64 and tile partition (CPU only)."""
import collections
import os

import numpy as np
import pytest

import oracle
from oracle.cache import SlotCache, LRU, RANDOM, CapacityError


def _read_worked(golden_dir):
    steps, want, totals = [], {"lru": [], "random": []}, {}
    for line in open(os.path.join(golden_dir, "cache_worked_example.txt")):
        if line.startswith("#") or not line.strip():
            continue
        f = line.split()
        if f[0] == "step":
            steps.append({int(a.split(":")[0]): int(a.split(":")[1]) for a in f[2:]})
        elif f[1] == "totals":
            totals[f[0]] = [int(v) for v in f[2:]]
        else:
            pt = [int(v) for v in f[7:13]]
            gen = [int(v) for v in f[14:17]]
            want[f[0]].append((int(f[3]), int(f[5]), pt, gen))
    return steps, want, totals


@pytest.mark.parametrize("policy,name", [(LRU, "lru"), (RANDOM, "random")])
def test_worked_example(golden_dir, policy, name):
    steps, want, totals = _read_worked(golden_dir)
    c = SlotCache(6, 3, policy, seed=0, layer=0, payload_bytes=100)
    for s, counts in enumerate(steps):
        cnt = [counts.get(e, 0) for e in range(6)]
        r = c.step(sorted(counts), cnt)
        h, m, pt, gen = want[name][s]
        assert (r["hits"], r["misses"], r["pt"], r["gen"]) == (h, m, pt, gen), (name, s)
    st = c.stats()
    assert [st["hits"], st["misses"], st["evictions"], st["materialized_bytes"]] == totals[name]


def _textbook_lru(trace, S):
    """Independent LRU: an OrderedDict in recency order over the same access
    sequence (resident experts ascending, then missing ones ascending)."""
    od = collections.OrderedDict()
    rec = []
    for uniq, counts in trace:
        hits_e = [e for e in sorted(uniq) if e in od]
        miss_e = [e for e in sorted(uniq) if e not in od]
        ev = 0
        for e in hits_e:
            od.move_to_end(e)
        for e in miss_e:
            if len(od) == S:
                od.popitem(last=False)
                ev += 1
            od[e] = True
        rec.append((sum(counts[e] for e in uniq) - len(miss_e), len(miss_e), ev, set(od)))
    return rec


def _random_trace(rng, E, steps, width):
    out = []
    for _ in range(steps):
        uniq = sorted(rng.choice(E, size=width, replace=False).tolist())
        counts = [0] * E
        for e in uniq:
            counts[e] = int(rng.integers(1, 4))
        out.append((uniq, counts))
    return out


def test_lru_matches_textbook_lru():
    rng = np.random.default_rng(0)
    for (E, S, width) in ((16, 8, 2), (64, 10, 7), (256, 38, 8), (40, 12, 12)):
        trace = _random_trace(rng, E, 200, width)
        c = SlotCache(E, S, LRU)
        ref = _textbook_lru(trace, S)
        evs = 0
        for (uniq, counts), (h, m, ev, resident) in zip(trace, ref):
            r = c.step(uniq, counts)
            evs += ev
            assert (r["hits"], r["misses"]) == (h, m)
            assert {e for e in range(E) if r["pt"][e] >= 0} == resident
            assert c.evictions == evs
            # page table is injective, consistent with the slot owners
            slots = [s for s in r["pt"] if s >= 0]
            assert len(slots) == len(set(slots)) <= S
            for e in range(E):
                if r["pt"][e] >= 0:
                    assert c.owner[r["pt"][e]] == e


def test_hits_plus_misses_equal_assignments_and_bytes():
    rng = np.random.default_rng(1)
    E, S, k, T = 32, 13, 4, 3  # S >= T*k so the random policy always has a victim
    for policy in (LRU, RANDOM):
        c = SlotCache(E, S, policy, seed=3, payload_bytes=1234)
        n = 0
        for _ in range(100):
            idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
            p = oracle.plan_union(idx, np.ones((T, k)), E)
            r = c.step(p["uniq"], p["counts"])
            assert r["hits"] + r["misses"] == k * T
            n += k * T
        st = c.stats()
        assert st["hits"] + st["misses"] == n
        assert st["materialized_bytes"] == st["misses"] * 1234


def test_cyclic_reuse_distance_cliff(golden_dir):
    # Routide §5.1: 303 fitting payloads below a 313-entry reuse cycle give
    # 0.00% LRU hits; seeded random eviction keeps some hits on the same trace.
    vals = {}
    for line in open(os.path.join(golden_dir, "page_numbers.txt")):
        if not line.startswith("#") and line.strip():
            a, b = line.split()[:2]
            vals[a] = float(b)
    cycle = int(vals["routide_reuse_threshold"])
    S = int(vals["routide_fitting_payloads"])
    E = 400
    trace = [([e % cycle], [1 if i == e % cycle else 0 for i in range(E)]) for e in range(5 * cycle)]
    lru = SlotCache(E, S, LRU)
    for u, cnt in trace:
        lru.step(u, cnt)
    assert lru.hits == 0 and lru.misses == 5 * cycle
    big = SlotCache(E, cycle, LRU)
    for u, cnt in trace:
        big.step(u, cnt)
    assert big.misses == cycle and big.hits == 4 * cycle
    rnd = SlotCache(E, S, RANDOM, seed=0)
    for u, cnt in trace:
        rnd.step(u, cnt)
    assert 0 < rnd.hits < 4 * cycle


def test_random_capacity_and_pinning():
    c = SlotCache(10, 3, RANDOM, seed=1)
    c.step([0, 1, 2], [1, 1, 1] + [0] * 7)
    with pytest.raises(CapacityError):
        c.step([3, 4, 5, 6], [0, 0, 0, 1, 1, 1, 1, 0, 0, 0])
    # the random victim is never an expert of the current step
    rng = np.random.default_rng(4)
    c = SlotCache(20, 6, RANDOM, seed=2)
    for _ in range(300):
        u = sorted(rng.choice(20, size=4, replace=False).tolist())
        before = {e for e in range(20) if c.pt[e] >= 0}
        r = c.step(u, [1 if e in u else 0 for e in range(20)])
        for (e, s, victim) in r["fills"]:
            assert victim not in u
            assert victim == -1 or victim in before


def test_lru_waves_when_union_exceeds_slots():
    # |U| > S: textbook LRU over the access sequence, so access i reuses the
    # slot of access i - S once the slots are full.
    E, S = 12, 4
    c = SlotCache(E, S, LRU)
    r = c.step(list(range(10)), [1] * 10 + [0, 0])
    slots = [s for (_, s, _) in r["fills"]]
    assert slots[:S] == [0, 1, 2, 3]
    for i in range(S, 10):
        assert slots[i] == slots[i - S]
    assert [e for e in range(E) if c.pt[e] >= 0] == [6, 7, 8, 9]


def test_preload_and_evict():
    c = SlotCache(8, 8, LRU, payload_bytes=10)
    c.preload(range(8))
    assert c.pt == list(range(8)) and c.misses == 0 and c.materialized_bytes == 0
    r = c.step([1, 5], [0, 2, 0, 0, 0, 1, 0, 0])
    assert r["hits"] == 3 and r["misses"] == 0
    c.evict(5)
    assert c.pt[5] == -1 and c.owner[5] == -1 and c.evictions == 1
    r = c.step([5], [0, 0, 0, 0, 0, 1, 0, 0])
    assert r["misses"] == 1 and c.pt[5] == 5 and c.gen[5] == 2


def test_splitmix64_published_vectors(golden_dir):
    for line in open(os.path.join(golden_dir, "splitmix64.txt")):
        if line.startswith("#") or not line.strip():
            continue
        seed, vals = line.split(":")
        g = oracle.SplitMix64(int(seed))
        assert [g.next() for _ in vals.split()] == [int(v) for v in vals.split()]


def test_tile_partition(golden_dir):
    from workloads import WORKLOADS
    for w in WORKLOADS.values():
        tiles = oracle.tile_partition(w.hidden, w.inter, w.quant)
        assert tiles[0][0] == 0
        for (o1, l1), (o2, _) in zip(tiles, tiles[1:]):
            assert o1 + l1 == o2
        assert sum(l for _, l in tiles) == w.payload_bytes
        assert max(l for _, l in tiles) <= 262144
    d = WORKLOADS["decode"]
    t = oracle.tile_partition(d.hidden, d.inter, d.quant)
    assert len(t) == 15 and t[4][1] == 65536  # 5 tiles per matrix, last 64 KiB
    wp = WORKLOADS["wide_prefill"]
    t = oracle.tile_partition(wp.hidden, wp.inter, wp.quant)
    assert len(t) == 27 and t[8][1] == 9216
    # Nanite §5.4: 1.61 GB over 7,504 tiles is below 256 KiB a tile on
    # average, so partial tiles occur
    vals = {}
    for line in open(os.path.join(golden_dir, "page_numbers.txt")):
        if not line.startswith("#") and line.strip():
            a, b = line.split()[:2]
            vals[a] = float(b)
    assert vals["nanite_tile_gb"] * 1e9 / vals["nanite_tiles"] < vals["nanite_tile_bytes"]


def test_prefetch_loads_useful_wasted_hand_worked():
    # "Paging the Experts" §3.3/§5.2: speculative loads, counted apart from
    # demand misses (§4.2) as useful when the next step uses them. Hand-worked
    # LRU replay, 2 slots, payload 100 B:
    #   step {0,1,2} (larger than the slots): 0 -> s0 (t1), 1 -> s1 (t2),
    #        2 evicts 0 from s0 (t3)
    #   prefetch 0: absent -> load, evicts 1 from s1 (oldest, t2) at t4
    #   step {0,3}: 0 was the load -> useful; hit 0 (t5); 3 evicts 2 from s0 (t3) at t6
    #   prefetch 4: absent -> load, evicts 0 from s1 (t5) at t7
    #   step {3,5}: 4 unused -> wasted; hit 3 (t8); 5 evicts 4 from s1 (t7) at t9
    #   prefetch 5 (preserve): resident -> probe; prefetch 3 (refresh): touch s0 at t10
    from oracle.cache import PREFETCH_PRESERVE, PREFETCH_REFRESH
    c = SlotCache(6, 2, LRU, payload_bytes=100)
    c.step([0, 1, 2], [1, 1, 1, 0, 0, 0])
    assert c.prefetch(0, PREFETCH_REFRESH) == dict(action="load", slot=1, victim=1)
    r = c.step([0, 3], [1, 0, 0, 1, 0, 0])
    assert (r["hits"], r["misses"], r["fills"]) == (1, 1, [(3, 0, 2)])
    assert c.prefetch(4, PREFETCH_PRESERVE) == dict(action="load", slot=1, victim=0)
    r = c.step([3, 5], [0, 0, 0, 1, 0, 1])
    assert (r["hits"], r["misses"], r["fills"]) == (1, 1, [(5, 1, 4)])
    assert c.prefetch(5, PREFETCH_PRESERVE) == dict(action="probe", slot=1, victim=-1)
    assert c.prefetch(3, PREFETCH_REFRESH) == dict(action="refresh", slot=0, victim=-1)
    assert c.last == [10, 9] and c.tick == 10
    assert c.pt == [-1, -1, -1, 0, -1, 1] and c.gen == [3, 4]
    assert c.stats() == dict(hits=2, misses=5, evictions=5, materialized_bytes=500)
    assert c.prefetch_stats() == dict(loads=2, useful=1, wasted=1, refreshes=1, probes=1, bytes=200)


def test_prefetch_random_policy_draws_over_every_slot():
    # nothing is pinned before a step: the random victim of a speculative
    # load is cand[next() mod n] over all slots; SplitMix64 (seed 0, layer 0)
    # first output 0xE220A8397B1DCDAF is odd -> slot 1 of 2
    from oracle.cache import PREFETCH_PRESERVE
    c = SlotCache(6, 2, RANDOM, seed=0, layer=0)
    c.step([0, 1], [1, 1, 0, 0, 0, 0])
    assert c.prefetch(5, PREFETCH_PRESERVE) == dict(action="load", slot=1, victim=1)
    assert c.pt == [0, -1, -1, -1, -1, 1]
