"""SplitMix64 (oracle; test infrastructure only).

The seeded random eviction of Routide (§4.1, §5.1: "seeded random eviction",
five declared seeds) needs a generator that both implementations can run
identically. This is SplitMix64 as published by Steele, Lea and Flood
("Fast splittable pseudorandom number generators", OOPSLA 2014): a Weyl
sequence with increment 0x9E3779B97F4A7C15 passed through a 64-bit mixing
function (Stafford's "Mix13" constants).
"""
from __future__ import annotations

_M64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15


class SplitMix64:
    def __init__(self, seed: int):
        self.state = seed & _M64

    def next(self) -> int:
        self.state = (self.state + GOLDEN_GAMMA) & _M64
        z = self.state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
        return z ^ (z >> 31)


def layer_seed(seed: int, layer: int) -> int:
    """Per-layer stream: seed XOR (layer * golden gamma) modulo 2^64."""
    return (seed ^ ((layer * GOLDEN_GAMMA) & _M64)) & _M64
