"""Bounded expert-slot cache with a page table (oracle; test infrastructure only).

What the pages fix:

* MawForge §IV-C: compact per-layer slot tensors; the slot count follows from
  the requested cache bytes and the per-slot expert block size; on a miss the
  requested expert block is materialised into an available slot and the
  route-to-slot metadata is updated.
* Routide §3.2: the budget counts expert-payload bytes, and entries are pinned
  while their layer is evaluated. §4.1/§5.1: LRU and seeded random eviction
  replayed on the same fixed route traces (0.00% LRU hits at 512 MiB is a
  reuse-distance effect: 303 fitting payloads against a 313-entry cycle).
  §4.2: with no speculation, materialised bytes = demand misses x payload.
* "Nanite for Experts" §5.4: persistent page-table entries with sentinel
  values for absent or stale generations.

Readings where the pages are silent (listed with the other readings of the
pages in the design notes):

* per step, hits = (number of assignments) - (number of missing experts): an
  expert that misses costs one miss and its other assignments in the step hit;
* access order within a step: resident experts of the union ascending, then
  missing experts ascending; every access takes the next tick;
* a miss takes the lowest-index free slot, else the victim's slot; the LRU
  victim is the resident expert with the oldest tick (textbook LRU over that
  access sequence); the random victim is drawn among resident experts that are
  not in the current union, listed by slot index, as cand[next() mod n] with
  SplitMix64 seeded by seed XOR (layer * 0x9E3779B97F4A7C15); draws happen in
  miss order; with no candidate the random policy fails with CapacityError;
* each fill of a slot bumps that slot's generation; the page table maps expert
  -> slot (-1 when absent).
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

from .splitmix import SplitMix64, layer_seed

LRU = 0
RANDOM = 1

# Prefetch modes ("Paging the Experts" §3.3): an absent predicted expert is
# loaded in both; a resident one is either touched like a hit
# (resident-refresh: the check updates its recency) or only recorded
# (preserve-resident: the cache state does not change).
PREFETCH_REFRESH = 1
PREFETCH_PRESERVE = 2


class CapacityError(RuntimeError):
    pass


def slot_count(budget_bytes: int, payload_bytes: int) -> int:
    """Slots that fit a byte budget (MawForge §IV-C): floor(budget / payload)."""
    return budget_bytes // payload_bytes


class SlotCache:
    def __init__(self, n_experts: int, n_slots: int, policy: int = LRU,
                 seed: int = 0, layer: int = 0, payload_bytes: int = 0):
        self.E = n_experts
        self.S = n_slots
        self.policy = policy
        self.payload = payload_bytes
        self.pt: List[int] = [-1] * n_experts  # expert -> slot
        self.owner: List[int] = [-1] * n_slots  # slot -> expert
        self.gen: List[int] = [0] * n_slots
        self.last: List[int] = [0] * n_slots  # tick of the slot's last access
        self.tick = 0
        self.rng = SplitMix64(layer_seed(seed, layer))
        self.hits = 0
        self.misses = 0
        self.evictions = 0
        self.materialized_bytes = 0
        # speculative loads are counted apart from demand ("Paging the
        # Experts" §4.2): loads, useful / wasted (the next step's union holds
        # the loaded expert / does not), resident probes that refreshed
        # recency or changed nothing, and the bytes the loads moved
        self.pending = -1
        self.pf = dict(loads=0, useful=0, wasted=0, refreshes=0, probes=0, bytes=0)

    # -- helpers
    def _fill(self, e: int, s: int) -> None:
        self.owner[s] = e
        self.pt[e] = s
        self.gen[s] += 1
        self.last[s] = self.tick

    def _take_slot(self, current: set) -> Tuple[int, int]:
        """Slot for a new fill: the lowest free one, else the policy's
        victim (evicted here). Returns (slot, evicted expert or -1)."""
        free = [s for s in range(self.S) if self.owner[s] < 0]
        if free:
            return free[0], -1
        s = self._victim_slot(current)
        victim = self.owner[s]
        self.pt[victim] = -1
        self.owner[s] = -1
        self.evictions += 1
        return s, victim

    def _victim_slot(self, current: set) -> int:
        if self.policy == LRU:
            return min(range(self.S), key=lambda s: self.last[s])
        cand = [s for s in range(self.S) if self.owner[s] not in current]
        if not cand:
            raise CapacityError("every resident expert is pinned by the current step")
        return cand[self.rng.next() % len(cand)]

    # -- public
    def step(self, uniq: Sequence[int], counts: Sequence[int]) -> dict:
        """One layer evaluation: resolve the union ``uniq`` (any order) whose
        experts have ``counts[e]`` assignments. Returns the step record."""
        U = sorted(int(e) for e in uniq)
        current = set(U)
        if self.pending >= 0:  # the last speculative load meets its step
            self.pf["useful" if self.pending in current else "wasted"] += 1
            self.pending = -1
        hit_e = [e for e in U if self.pt[e] >= 0]
        miss_e = [e for e in U if self.pt[e] < 0]
        for e in hit_e:
            self.tick += 1
            self.last[self.pt[e]] = self.tick
        fills: List[Tuple[int, int, int]] = []  # (expert, slot, evicted expert or -1)
        for e in miss_e:
            self.tick += 1
            s, victim = self._take_slot(current)
            self._fill(e, s)
            fills.append((e, s, victim))
        n_assign = sum(int(counts[e]) for e in U)
        hits = n_assign - len(miss_e)
        self.hits += hits
        self.misses += len(miss_e)
        self.materialized_bytes += len(miss_e) * self.payload
        return dict(hits=hits, misses=len(miss_e), fills=fills,
                    pt=list(self.pt), gen=list(self.gen))

    def prefetch(self, e: int, mode: int) -> dict:
        """Speculative access to expert ``e`` before a step ("Paging the
        Experts" §3.3): routing and arithmetic are unchanged, only the cache
        is. If ``e`` is absent it is loaded like a miss, with nothing pinned
        (the lowest free slot, else the policy's victim), one tick; if it is
        resident, PREFETCH_REFRESH touches it as a hit would (one tick) and
        PREFETCH_PRESERVE records the probe and changes nothing. Returns
        dict(action="load"|"refresh"|"probe", slot, victim)."""
        e = int(e)
        if self.pt[e] >= 0:
            if mode == PREFETCH_REFRESH:
                self.tick += 1
                self.last[self.pt[e]] = self.tick
                self.pf["refreshes"] += 1
                return dict(action="refresh", slot=self.pt[e], victim=-1)
            self.pf["probes"] += 1
            return dict(action="probe", slot=self.pt[e], victim=-1)
        self.tick += 1
        s, victim = self._take_slot(set())
        self._fill(e, s)
        self.pending = e
        self.pf["loads"] += 1
        self.pf["bytes"] += self.payload
        return dict(action="load", slot=s, victim=victim)

    def preload(self, experts: Sequence[int]) -> None:
        """Fill slots with ``experts`` (ascending) before the first step; not
        counted as hits, misses or materialised bytes."""
        for e in sorted(int(x) for x in experts):
            if self.pt[e] >= 0:
                continue
            self.tick += 1
            free = [s for s in range(self.S) if self.owner[s] < 0]
            if not free:
                raise CapacityError("preload exceeds the slot count")
            self._fill(e, free[0])

    def evict(self, e: int) -> None:
        """Explicit eviction: the expert's slot becomes free."""
        s = self.pt[e]
        if s < 0:
            return
        self.pt[e] = -1
        self.owner[s] = -1
        self.evictions += 1

    def stats(self) -> dict:
        return dict(hits=self.hits, misses=self.misses, evictions=self.evictions,
                    materialized_bytes=self.materialized_bytes)

    def prefetch_stats(self) -> dict:
        return dict(self.pf)
