"""Pins of the static budget check (MawForge §IV-D) and of the C ABI's copy
of it, all on the CPU."""
import os

import numpy as np
import pytest

import oracle
from oracle.formats import Q8_0, payload_bytes


def _golden(golden_dir):
    vals = {}
    for line in open(os.path.join(golden_dir, "page_numbers.txt")):
        if not line.startswith("#") and line.strip():
            a, b = line.split()[:2]
            vals[a] = float(b)
    return vals


def test_static_minima_differ_by_the_expert_cache_share(golden_dir):
    # MawForge §V-C: the same profile and context at 50% and 65% cache; C and
    # K(n) are common to both rows, so the difference is E(0.65) - E(0.50)
    v = _golden(golden_dir)
    L, E = int(v["gemma_layers"]), int(v["gemma_experts"])
    P = payload_bytes(2816, 704, Q8_0)
    a = oracle.static_budget(L, E, P, 500_000, 0, 0, 0, 0, 0)
    b = oracle.static_budget(L, E, P, 650_000, 0, 0, 0, 0, 0)
    gib = (b["lower_bound"] - a["lower_bound"]) / 2**30
    # each printed minimum is rounded to 4 decimals: the difference is good
    # to 1e-4
    assert abs(gib - (v["gemma_static_min_65_gib"] - v["gemma_static_min_50_gib"])) <= 1e-4 + 1e-12
    # and the whole expert cache at 100% is 30 x 128 payloads
    assert oracle.static_budget(L, E, P, 1_000_000, 0, 0, 0, 0, 0)["expert_bytes"] == L * E * P


def test_slot_counts_of_the_workloads():
    # floor(p * E): 15% of 256 -> 38, 35% of 256 -> 89, 35% of 128 -> 44
    assert oracle.static_budget(1, 256, 1, 150_000, 0, 0, 0, 0, 0)["slots_per_layer"] == 38
    assert oracle.static_budget(1, 256, 1, 350_000, 0, 0, 0, 0, 0)["slots_per_layer"] == 89
    assert oracle.static_budget(1, 128, 1, 350_000, 0, 0, 0, 0, 0)["slots_per_layer"] == 44


def test_rejection_rule_and_terms():
    # L = C + E + K; F = L + O; rejected exactly when L exceeds the target
    r = oracle.static_budget(2, 10, 1000, 500_000, 7, 3, 100, 11, 0)
    assert r["expert_bytes"] == 10_000 and r["kv_bytes"] == 300
    assert r["lower_bound"] == 7 + 10_000 + 300 and r["footprint"] == r["lower_bound"] + 11
    L = r["lower_bound"]
    assert oracle.static_budget(2, 10, 1000, 500_000, 7, 3, 100, 11, L)["accepted"] == 1
    assert oracle.static_budget(2, 10, 1000, 500_000, 7, 3, 100, 11, L - 1)["accepted"] == 0
    # the overhead is not part of the static check
    assert oracle.static_budget(2, 10, 1000, 500_000, 7, 3, 100, 10**9, L)["accepted"] == 1
    with pytest.raises(ValueError):
        oracle.static_budget(1, 1, 1, 1_000_001, 0, 0, 0, 0, 0)


@pytest.fixture(scope="module")
def bec():
    import __graft_entry__
    __graft_entry__.build()
    import bounded_expert_cache_gb300 as m
    return m


def test_abi_static_budget_matches_oracle(bec):
    rng = np.random.default_rng(5)
    for _ in range(300):
        args = (int(rng.integers(1, 80)), int(rng.integers(1, 513)), int(rng.integers(1, 20_000_000)),
                int(rng.integers(0, 1_000_001)), int(rng.integers(0, 2**40)), int(rng.integers(0, 2**20)),
                int(rng.integers(0, 2**18)), int(rng.integers(0, 2**36)), int(rng.integers(0, 2**46)))
        assert bec.static_budget(*args) == oracle.static_budget(*args), args
    with pytest.raises(bec.MoeError):
        bec.static_budget(1, 1, 1, 1_000_001)
    with pytest.raises(bec.MoeError):
        bec.static_budget(1, 1, 2**62, 1_000_000, kv_bytes_per_token=2**62, context=4)
