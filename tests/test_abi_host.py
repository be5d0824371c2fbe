"""Host-side tests of the C ABI (no GPU): symbol exports, the slot manager
against the oracle's replay, SplitMix64, argument validation."""
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from oracle.cache import SlotCache

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bec():
    import __graft_entry__
    __graft_entry__.build()
    import bounded_expert_cache_gb300 as m
    return m


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol(bec):
    from bounded_expert_cache_gb300 import _native
    declared = _declared_symbols()
    assert len(declared) >= 25
    out = subprocess.run(["nm", "-D", "--defined-only", _native._LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (moe_\w+)", out))
    assert declared <= exported, declared - exported
    bound = {n for n, _, _ in _native.SIGNATURES}
    assert declared == bound, declared ^ bound


def test_ctypes_structs_match_header(bec, tmp_path):
    # the binding's structures have the header's size and field offsets, as a
    # C compiler lays them out (the header needs no CUDA header of its own)
    import ctypes

    from bounded_expert_cache_gb300 import _native as N
    pairs = {"moe_config_t": N.Config, "moe_plan_t": N.PlanT, "moe_miss_list_t": N.MissList,
             "moe_stats_t": N.Stats, "moe_budget_t": N.Budget}
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "moecache.h"', "int main(void) {"]
    for cname, cls in pairs.items():
        lines.append('  printf("%s %%zu\\n", sizeof(%s));' % (cname, cname))
        for fname, _ in cls._fields_:
            lines.append('  printf("%s.%s %%zu\\n", offsetof(%s, %s));' % (cname, fname, cname, fname))
    lines += ["  return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines) + "\n")
    exe = tmp_path / "layout"
    r = subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    if r.returncode != 0:
        pytest.skip("no C compiler for the header: " + r.stderr[-200:])
    got = dict(line.split() for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                       check=True).stdout.splitlines())
    for cname, cls in pairs.items():
        assert int(got[cname]) == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert int(got[cname + "." + fname]) == getattr(cls, fname).offset, (cname, fname)


def test_splitmix64_published_vectors(bec, golden_dir):
    for line in open(os.path.join(golden_dir, "splitmix64.txt")):
        if line.startswith("#") or not line.strip():
            continue
        seed, vals = line.split(":")
        want = [int(v) for v in vals.split()]
        assert bec.splitmix64(int(seed), len(want)) == want


def _compare_replay(bec, E, S, policy, seed, layer, trace, payload=1000):
    ref = SlotCache(E, S, policy, seed=seed, layer=layer, payload_bytes=payload)
    s = bec.Slots(E, S, policy, seed, layer, payload)
    for uniq, counts in trace:
        r = ref.step(uniq, counts)
        m = s.step(list(uniq), list(counts))
        pt, gen = s.read()
        assert pt == r["pt"] and gen == r["gen"]
        assert (m.hits, m.misses) == (r["hits"], r["misses"])
        assert list(zip(m.expert, m.slot, m.victim)) == [tuple(f) for f in r["fills"]]
    st = s.stats()
    rs = ref.stats()
    for key in ("hits", "misses", "evictions", "materialized_bytes"):
        assert st[key] == rs[key], key


@pytest.mark.parametrize("policy", [0, 1])
def test_slot_manager_matches_oracle_replay(bec, policy):
    rng = np.random.default_rng(10 + policy)
    for (E, S, width, layer, seed) in ((16, 8, 2, 0, 0), (256, 38, 8, 7, 3), (64, 20, 12, 39, 4),
                                       (256, 89, 30, 1, 2)):
        trace = []
        for _ in range(150):
            u = sorted(rng.choice(E, size=width, replace=False).tolist())
            counts = [0] * E
            for e in u:
                counts[e] = int(rng.integers(1, 5))
            trace.append((u, counts))
        _compare_replay(bec, E, S, policy, seed, layer, trace)


def test_slot_manager_worked_example(bec, golden_dir):
    steps = []
    for line in open(os.path.join(golden_dir, "cache_worked_example.txt")):
        f = line.split()
        if f and f[0] == "step":
            steps.append({int(a.split(":")[0]): int(a.split(":")[1]) for a in f[2:]})
    for policy in (0, 1):
        trace = [(sorted(c), [c.get(e, 0) for e in range(6)]) for c in steps]
        _compare_replay(bec, 6, 3, policy, 0, 0, trace, payload=100)


def test_slot_manager_on_routed_trace(bec):
    # a route trace of the tiny workload computed by the oracle, replayed by both
    from workloads import WORKLOADS, router_weights, activations, with_changes
    w = with_changes(WORKLOADS["tiny"], n_steps=24)
    W = router_weights(w, 0)
    x = activations(w, 0).astype(np.float64)
    trace = []
    for s in range(w.n_steps):
        idx, wt, _ = oracle.route(x[s * 4:(s + 1) * 4], W, None, w.top_k)
        p = oracle.plan_union(idx, wt, w.n_experts)
        trace.append((p["uniq"].tolist(), p["counts"].tolist()))
    for policy in (0, 1):
        _compare_replay(bec, w.n_experts, w.slots, policy, 0, 0, trace)


def test_slot_manager_waves_and_capacity(bec):
    s = bec.Slots(12, 4, 0)
    m = s.step(list(range(10)), [1] * 10 + [0, 0])
    assert m.slot[:4] == [0, 1, 2, 3]
    assert all(m.slot[i] == m.slot[i - 4] for i in range(4, 10))
    assert m.wave == [0, 0, 0, 0, 1, 1, 1, 1, 2, 2] and m.n_waves == 3
    r = bec.Slots(10, 3, 1, 1)
    r.step([0, 1, 2], [1, 1, 1] + [0] * 7)
    before = r.read()
    with pytest.raises(bec.MoeError) as ei:
        r.step([3, 4, 5, 6], [0, 0, 0, 1, 1, 1, 1, 0, 0, 0])
    assert ei.value.status == 3
    assert r.read() == before


def test_slot_manager_waves_over_many_steps_match_oracle(bec):
    # LRU steps whose unions are larger than the slots, with residents of the
    # union that a fill of the same step evicts: fills, page table,
    # generations and counters follow the oracle's replay (the misses are
    # the experts absent when the step starts), and the wave of a fill comes
    # after the wave of the in-step expert it evicts
    rng = np.random.default_rng(21)
    for (E, S, lo, hi) in ((12, 4, 3, 11), (128, 44, 30, 128), (64, 20, 15, 64)):
        s = bec.Slots(E, S, 0, 0, 0, 1)
        ref = SlotCache(E, S, 0, seed=0, layer=0, payload_bytes=1)
        for _ in range(40):
            width = int(rng.integers(lo, hi + 1))
            u = sorted(rng.choice(E, size=width, replace=False).tolist())
            counts = [0] * E
            for e in u:
                counts[e] = int(rng.integers(1, 4))
            r = ref.step(u, counts)
            m = s.step(u, counts)
            assert list(zip(m.expert, m.slot, m.victim)) == [tuple(f) for f in r["fills"]]
            assert s.read() == (r["pt"], r["gen"])
            assert (m.hits, m.misses) == (r["hits"], r["misses"])
            wave_of = {e: 0 for e in u}
            for e, v, wv in zip(m.expert, m.victim, m.wave):
                assert wv == (wave_of[v] + 1 if v in wave_of else 0)
                wave_of[e] = wv
            assert m.n_waves == (max(m.wave) + 1 if m.wave else 1)
        st, rs = s.stats(), ref.stats()
        for key in ("hits", "misses", "evictions", "materialized_bytes"):
            assert st[key] == rs[key], key


def test_slot_manager_rejects_bad_union(bec):
    s = bec.Slots(8, 4, 0)
    with pytest.raises(bec.MoeError):
        s.step([1, 1], [0] * 8)
    with pytest.raises(bec.MoeError):
        s.step([9], [0] * 8)


def test_create_validates_config_without_gpu(bec):
    import ctypes as C
    from bounded_expert_cache_gb300 import _native as N
    bad = [dict(hidden=100), dict(top_k=0), dict(slots_per_layer=0), dict(quant=7),
           dict(tile_bytes=10), dict(n_streams=0), dict(n_experts=2000)]
    for b in bad:
        kw = dict(n_layers=1, n_experts=16, top_k=2, hidden=256, inter=128, shared_inter=0,
                  quant=0, slots_per_layer=8, policy=0, n_streams=3, seed=0, tile_bytes=262144,
                  max_tokens=4)
        kw.update(b)
        cfg = N.Config(**kw)
        h = C.c_void_p()
        st = N.lib.moe_create(C.byref(cfg), C.byref(h))
        assert st == 1 and not h.value
        assert b"moe_create" in N.lib.moe_last_error(None)


@pytest.mark.parametrize("policy", [0, 1])
@pytest.mark.parametrize("mode", [1, 2])
def test_slot_manager_prefetch_matches_oracle(bec, policy, mode):
    # speculative accesses between steps ("Paging the Experts" §3.3): the
    # ABI's loads, refreshes, probes, victims and useful/wasted counts equal
    # the oracle's on random traces; a predicted expert is sometimes resident,
    # sometimes absent (also when a union larger than the slots evicted it)
    rng = np.random.default_rng(40 + 2 * policy + mode)
    for (E, S, width) in ((16, 8, 3), (64, 12, 10), (32, 6, 9 if policy == 0 else 4)):
        ref = SlotCache(E, S, policy, seed=5, layer=3, payload_bytes=77)
        s = bec.Slots(E, S, policy, 5, 3, 77)
        for _ in range(120):
            if rng.random() < 0.7:
                e = int(rng.integers(E))
                r = ref.prefetch(e, mode)
                act, fill = s.prefetch(e, mode)
                assert act == r["action"]
                if act == "load":
                    assert fill == (e, r["slot"], r["victim"])
            u = sorted(rng.choice(E, size=width, replace=False).tolist())
            counts = [0] * E
            for e in u:
                counts[e] = int(rng.integers(1, 4))
            r = ref.step(u, counts)
            m = s.step(u, counts)
            assert (m.hits, m.misses) == (r["hits"], r["misses"])
            assert list(zip(m.expert, m.slot, m.victim)) == [tuple(f) for f in r["fills"]]
            assert s.read() == (r["pt"], r["gen"])
        st, rs, pf = s.stats(), ref.stats(), ref.prefetch_stats()
        for key in ("hits", "misses", "evictions", "materialized_bytes"):
            assert st[key] == rs[key], key
        for key in ("loads", "useful", "wasted", "refreshes", "probes", "bytes"):
            assert st["prefetch_" + key] == pf[key], key
        assert pf["loads"] > 0 and pf["refreshes" if mode == 1 else "probes"] > 0
