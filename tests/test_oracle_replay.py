"""Pins of the offline policy replays (farthest next use, static working set)
against brute force and hand examples, all on the CPU; and the C ABI's
replay against the oracle."""
import functools

import numpy as np
import pytest

import oracle
from oracle.cache import LRU, RANDOM
from oracle.replay import FARTHEST_NEXT_USE, STATIC_SET


def _trace(rng, E, S, n, max_u=None):
    steps = []
    for _ in range(n):
        w = int(rng.integers(1, (max_u or S) + 1))
        u = sorted(rng.choice(E, size=w, replace=False).tolist())
        counts = [0] * E
        for e in u:
            counts[e] = int(rng.integers(1, 4))
        steps.append((u, counts))
    return steps


def _min_misses(steps, S):
    """Fewest misses of any eviction schedule that keeps each step's union
    resident (exhaustive search over the resident set)."""
    sets = [frozenset(u) for u, _ in steps]

    @functools.lru_cache(maxsize=None)
    def best(t, resident):
        if t == len(sets):
            return 0
        U = sets[t]
        miss = len(U - resident)
        others = sorted(resident - U)
        keep_max = S - len(U)
        out = None
        # keep any subset of the other residents that fits
        for mask in range(1 << len(others)):
            kept = frozenset(o for i, o in enumerate(others) if mask >> i & 1)
            if len(kept) > keep_max:
                continue
            v = best(t + 1, U | kept)
            out = v if out is None else min(out, v)
        return miss + out

    return best(0, frozenset())


def test_farthest_next_use_is_optimal_on_tiny_traces():
    rng = np.random.default_rng(3)
    for _ in range(60):
        E, S = int(rng.integers(4, 7)), int(rng.integers(1, 4))
        steps = _trace(rng, E, S, int(rng.integers(4, 9)))
        r = oracle.replay(FARTHEST_NEXT_USE, E, S, steps)
        assert r["misses"] == _min_misses(steps, S), steps


def test_farthest_next_use_bounds_lru_and_random():
    rng = np.random.default_rng(4)
    for _ in range(10):
        E, S = 40, 10
        steps = _trace(rng, E, S, 80, max_u=6)
        f = oracle.replay(FARTHEST_NEXT_USE, E, S, steps)
        assert f["misses"] <= oracle.replay(LRU, E, S, steps)["misses"]
        for seed in range(3):
            assert f["misses"] <= oracle.replay(RANDOM, E, S, steps, seed=seed)["misses"]
        assert f["hits"] + f["misses"] == sum(sum(c) for _, c in steps)


def test_static_working_set_hand_example():
    E = 5
    steps = [([0, 1], [3, 1, 0, 0, 0]), ([1, 2], [0, 2, 2, 0, 0]), ([3], [0, 0, 0, 1, 0]),
             ([0, 4], [1, 0, 0, 0, 2])]
    # calibration over the first two steps: totals 0:3 1:3 2:2 -> width 2 keeps {0, 1}
    assert oracle.static_set(steps, E, 2, 2) == [0, 1]
    r = oracle.replay(STATIC_SET, E, 3, steps, payload=10, width=2, calib=2)
    # misses: step 1 {2}, step 2 {3}, step 3 {4} -> 3; hits = 12 assignments - 3
    assert r == dict(hits=9, misses=3, evictions=0, materialized_bytes=30)
    # everything resident: no misses
    assert oracle.replay(STATIC_SET, E, E, steps, width=E, calib=4)["misses"] == 0


@pytest.fixture(scope="module")
def bec():
    import __graft_entry__
    __graft_entry__.build()
    import bounded_expert_cache_gb300 as m
    return m


def test_abi_replay_matches_oracle(bec):
    rng = np.random.default_rng(8)
    for (E, S, n, mu) in ((8, 3, 40, 3), (64, 16, 120, 12), (256, 38, 100, 8)):
        steps = _trace(rng, E, S, n, max_u=mu)
        for policy, kw in ((LRU, {}), (RANDOM, dict(seed=2, layer=5)), (FARTHEST_NEXT_USE, {}),
                           (STATIC_SET, dict(width=min(S, 6), calib=n // 4))):
            want = oracle.replay(policy, E, S, steps, payload=7, **kw)
            got = bec.replay(policy, E, S, steps, payload=7, **kw)
            assert {k: got[k] for k in want} == want, (E, S, policy)
