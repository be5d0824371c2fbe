"""CPU oracle for the bounded-expert-cache MoE layer — TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously-correct restatement of what the routed MoE layer over
a bounded, page-table-addressed expert-slot cache computes, written from the
pages:

* "MawForge: Memory-Bounded Expert Materialization for Local MoE Inference"
  (arxiv 2607.09686v1), §IV-B/§IV-C (split packs, per-layer slot tensors,
  materialise a miss into an available slot and update route-to-slot
  metadata) and §IV-D (static budget);
* "Nanite for Experts", §1 (40 layers, 256 routed experts, eight routed plus
  one shared expert per token), §3.1 (authoritative routing), §5.3
  (expert-major union across the multi-token window), §5.4 (256 KiB virtual
  tiles, device page table with sentinel entries), §5.5 (merge into the
  original output positions);
* "Paging the Experts" (Routide, arxiv 2609.29032v1), §3.1 (gate/up/down
  projections), §3.2 (byte-budgeted cache, entries pinned per layer), §3.3
  and §5.2 (confidence-gated prefetch, useful and wasted loads),
  §4.1/§5.1 (LRU versus seeded random eviction on fixed route replays),
  §4.2 (materialised bytes = demand misses x payload).

Floating point is fp64 (numpy) with ``math.fsum`` for the router's exact,
correctly rounded dot products. Library primitives (matmul, sort, fsum) are
used as single steps; nothing is blocked, fused or reordered.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline``
leg may import this package. It shares no code with the CUDA path and never
consumes its outputs.

Pins: every function here is checked in ``tests/test_oracle_formats.py``,
``test_oracle_route.py``, ``test_oracle_ffn.py``, ``test_oracle_cache.py``,
``test_oracle_replay.py``, ``test_oracle_budget.py`` and
``test_oracle_trace.py`` against closed forms, brute force, an independent
implementation of textbook LRU, hand-worked replays and the byte counts
printed on the pages. The routine ``moe_layer`` (fp64 FFN) is
pinned by permutation-matrix closed forms; no page prints a worked output
vector for synthetic inputs.
"""
from .formats import (Q8_0, Q4_0, I4_G64, bf16_bits_to_f64, f16_bits_to_f64, payload_bytes,
                      dequant_q8_0, dequant_q4_0, dequant_i4_g64, expert_matrices)
from .route import router_logits, topk_select, combine_weights, route
from .plan import plan_union
from .splitmix import SplitMix64
from .cache import (SlotCache, CapacityError, LRU, RANDOM, PREFETCH_REFRESH, PREFETCH_PRESERVE,
                    slot_count)
from .prefetch import prediction as prefetch_prediction
from .budget import static_budget
from .replay import replay, static_set, FARTHEST_NEXT_USE, STATIC_SET
from .ffn import silu, expert_ffn, moe_layer
from .tiles import tile_partition

__all__ = [
    "Q8_0", "Q4_0", "bf16_bits_to_f64", "f16_bits_to_f64", "payload_bytes",
    "dequant_q8_0", "dequant_q4_0", "expert_matrices", "router_logits",
    "topk_select", "combine_weights", "route", "plan_union", "SplitMix64",
    "SlotCache", "CapacityError", "LRU", "RANDOM", "slot_count", "silu",
    "expert_ffn", "moe_layer", "tile_partition",
]
