"""Seeded synthetic workloads for the bounded-expert-cache MoE layer.

This module only draws inputs and lays them out in memory. It holds none of
the method's arithmetic (no dequantisation, routing, union, caching or FFN);
both the CPU oracle and the CUDA path consume what it produces, and neither
imports the other.

Workloads (sizes and distributions as stated for the five measured
configurations; names describe what each one is):

=============  ======  ====  ==  ====  =====  =====  =====================  ====
name           H       E     k   I     I_s    quant  tokens                 S
=============  ======  ====  ==  ====  =====  =====  =====================  ====
tiny           256     16    2   128   0      Q8_0   4 fp32 N(0,1)          8
decode         2048    256   8   512   512    Q8_0   1/step bf16 AR(1)      38
mtp_decode     2048    256   8   512   512    Q4_0   4/step bf16 AR(1)      89
prefill        2048    256   8   512   512    Q8_0   4096 bf16 N(0,1)+Zipf  256
wide_prefill   2816    128   8   704   2112   Q8_0   32768 bf16 (8x4096)    44
i4_decode      2048    256   8   512   512    I4_G64 1/step bf16 AR(1)      38
=============  ======  ====  ==  ====  =====  =====  =====================  ====

Router weights are fp32 N(0, 0.02). Q8_0 quants are uniform on [-127, 127];
Q4_0 nibbles are uniform on [0, 15]; every 32-weight block carries an fp16
scale drawn U[1e-3, 2e-2] and rounded to fp16. I4_G64 (affine INT4, groups
of 64) nibbles are uniform on [0, 15]; each group's bf16 scale s is drawn
U[1e-3, 2e-2] and its bf16 bias -s*U[7, 8], both rounded to bf16. bf16 activations are drawn in
fp64 and rounded (fp64 -> fp32 -> bf16, round-to-nearest-even at each step).

Expert payload layout ("split-plane"): for each matrix in the order gate
[I, H], up [I, H], down [H, I] (row-major, 32-weight blocks consecutive along
the input dimension K), a quant plane followed by a scale plane:

* Q8_0 quant plane: int8 [rows][K]; Q4_0 quant plane: uint8 [rows][K/2], where
  byte j of each 32-block holds element j in its low nibble and element j+16
  in its high nibble (the GGUF convention);
* scale plane: fp16 [rows][K/32], little-endian; for I4_G64 (quant plane as
  uint8 [rows][K/2] with element 2j in the low nibble of byte j and element
  2j+1 in its high nibble) the plane holds (scale, bias) bf16 pairs
  [rows][K/64][2], the same number of bytes.

The bytes per expert equal the interleaved GGUF size (34 B per 32 weights for
Q8_0, 18 B for Q4_0); only the order of the bytes differs.

Random streams are keyed by ``SeedSequence([seed, layer, expert, field])`` so
any single expert can be regenerated on its own. The shared expert uses the
expert id ``E``.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Optional

import numpy as np

Q8_0 = 0
Q4_0 = 1
I4_G64 = 2

LRU = 0
RANDOM = 1

# field ids of the keyed random streams
_F_ROUTER = 1
_F_BIAS = 2
_F_X = 3
_F_QUANT = 10  # + matrix id (0 gate, 1 up, 2 down)
_F_SCALE = 20  # + matrix id


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int  # 0: no shared expert
    quant: int
    x_dtype: str  # "f32" or "bf16"
    x_recipe: str  # "normal", "ar1"
    tokens_per_step: int
    n_layers: int
    n_steps: int
    slots: int
    policy: int
    seed: int
    rho: float = 0.0
    zipf_s: float = 0.0  # > 0: router bias b_e = -s * ln(1 + pi(e))
    preload: bool = False  # every expert resident before the first step

    @property
    def block_bytes(self) -> int:
        return 34 if self.quant == Q8_0 else 18

    def matrix_bytes(self, rows: int, k: int) -> int:
        return rows * (k // 32) * self.block_bytes

    @property
    def payload_bytes(self) -> int:
        """Bytes of one routed expert (gate + up + down)."""
        return 3 * self.matrix_bytes(self.inter, self.hidden)

    @property
    def shared_payload_bytes(self) -> int:
        if self.shared_inter == 0:
            return 0
        return 3 * self.matrix_bytes(self.shared_inter, self.hidden)

    @property
    def n_tokens(self) -> int:
        """Tokens per layer over the whole trace."""
        return self.tokens_per_step * self.n_steps


WORKLOADS = {
    "tiny": Workload("tiny", 256, 16, 2, 128, 0, Q8_0, "f32", "normal", 4, 1, 1,
                     8, LRU, seed=0),
    "decode": Workload("decode", 2048, 256, 8, 512, 512, Q8_0, "bf16", "ar1", 1,
                       40, 128, 38, LRU, seed=1, rho=0.9),
    "mtp_decode": Workload("mtp_decode", 2048, 256, 8, 512, 512, Q4_0, "bf16",
                           "ar1", 4, 40, 128, 89, LRU, seed=2, rho=0.9),
    "prefill": Workload("prefill", 2048, 256, 8, 512, 512, Q8_0, "bf16",
                        "normal", 4096, 1, 1, 256, LRU, seed=3, zipf_s=1.1,
                        preload=True),
    "wide_prefill": Workload("wide_prefill", 2816, 128, 8, 704, 2112, Q8_0,
                             "bf16", "normal", 4096, 1, 8, 44, LRU, seed=4),
    "i4_decode": Workload("i4_decode", 2048, 256, 8, 512, 512, I4_G64, "bf16",
                          "ar1", 1, 4, 24, 38, LRU, seed=5, rho=0.9),
}


def with_changes(w: Workload, **kw) -> Workload:
    return dataclasses.replace(w, **kw)


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


# ---------------------------------------------------------------- activations
def f64_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp64 -> fp32 -> bf16 (nearest-even each step); return uint16 bits."""
    f = np.ascontiguousarray(a, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def router_weights(w: Workload, layer: int) -> np.ndarray:
    """fp32 [E, H], N(0, 0.02)."""
    g = _rng(w.seed, layer, 0, _F_ROUTER)
    return (g.standard_normal((w.n_experts, w.hidden)) * 0.02).astype(np.float32)


def router_bias(w: Workload, layer: int) -> Optional[np.ndarray]:
    """fp32 [E] Zipf-skewed bias -s*ln(1+pi(e)) with pi a seeded permutation, or None."""
    if w.zipf_s <= 0.0:
        return None
    g = _rng(w.seed, layer, 0, _F_BIAS)
    pi = g.permutation(w.n_experts)
    return (-w.zipf_s * np.log1p(pi.astype(np.float64))).astype(np.float32)


def activations(w: Workload, layer: int, n_tokens: Optional[int] = None,
                token0: int = 0) -> np.ndarray:
    """Layer inputs for tokens [token0, token0 + n_tokens) of the trace.

    Returns float32 [n, H] for f32 workloads, else uint16 bf16 bits [n, H].
    Each layer's sequence is drawn independently. "ar1": x_0 ~ N(0,1),
    x_t = rho x_{t-1} + sqrt(1 - rho^2) eps_t, in fp64, before rounding.
    """
    total = w.n_tokens
    if n_tokens is None:
        n_tokens = total - token0
    assert 0 <= token0 and token0 + n_tokens <= total
    g = _rng(w.seed, layer, 0, _F_X)
    if w.x_recipe == "ar1":
        eps = g.standard_normal((token0 + n_tokens, w.hidden))
        x = np.empty_like(eps)
        x[0] = eps[0]
        c = np.sqrt(1.0 - w.rho * w.rho)
        for t in range(1, x.shape[0]):
            x[t] = w.rho * x[t - 1] + c * eps[t]
        x = x[token0:]
    else:
        x = g.standard_normal((token0 + n_tokens, w.hidden))[token0:]
    if w.x_dtype == "f32":
        return x.astype(np.float32)
    return f64_to_bf16_bits(x)


# ---------------------------------------------------------------- experts
def _matrix_shapes(w: Workload, inter: int):
    return [(inter, w.hidden), (inter, w.hidden), (w.hidden, inter)]


def _fill_quant(g: np.random.Generator, out: np.ndarray, quant: int) -> None:
    n = out.shape[0]
    u = g.integers(0, 256, size=n, dtype=np.uint8)
    if quant == Q8_0:
        # uniform on 1..255 by redrawing zeros, then u - 128 -> [-127, 127]
        z = np.flatnonzero(u == 0)
        while z.size:
            u[z] = g.integers(0, 256, size=z.size, dtype=np.uint8)
            z = z[u[z] == 0]
        np.bitwise_xor(u, np.uint8(0x80), out=out)
    else:
        out[:] = u


def expert_payload(w: Workload, layer: int, expert: int,
                   out: Optional[np.ndarray] = None) -> np.ndarray:
    """Packed bytes (uint8) of routed expert ``expert`` (or the shared expert
    when ``expert == E``) in the split-plane layout described above."""
    shared = expert == w.n_experts
    inter = w.shared_inter if shared else w.inter
    nbytes = w.shared_payload_bytes if shared else w.payload_bytes
    if out is None:
        out = np.empty(nbytes, dtype=np.uint8)
    assert out.shape == (nbytes,) and out.dtype == np.uint8
    off = 0
    for m, (rows, k) in enumerate(_matrix_shapes(w, inter)):
        qbytes = rows * k if w.quant == Q8_0 else rows * k // 2
        _fill_quant(_rng(w.seed, layer, expert, _F_QUANT + m), out[off:off + qbytes], w.quant)
        off += qbytes
        nblk = rows * (k // 32)
        g = _rng(w.seed, layer, expert, _F_SCALE + m)
        if w.quant == I4_G64:
            ngrp = rows * (k // 64)
            sc = g.uniform(1e-3, 2e-2, ngrp)
            bi = -sc * g.uniform(7.0, 8.0, ngrp)
            sb = np.empty((ngrp, 2), dtype=np.uint16)
            sb[:, 0] = f64_to_bf16_bits(sc)
            sb[:, 1] = f64_to_bf16_bits(bi)
            out[off:off + 4 * ngrp] = sb.astype("<u2").view(np.uint8).ravel()
            off += 4 * ngrp
            continue
        d = g.uniform(1e-3, 2e-2, nblk).astype(np.float16)
        out[off:off + 2 * nblk] = d.astype("<f2").view(np.uint8)
        off += 2 * nblk
    assert off == nbytes
    return out


def fill_store(w: Workload, store: np.ndarray, layers=None, experts=None,
               threads: Optional[int] = None) -> None:
    """Fill ``store`` (uint8 [L, E, payload]) with routed expert payloads.

    ``layers``/``experts`` restrict the (layer, expert) pairs written.
    """
    L, E, P = store.shape
    assert E == w.n_experts and P == w.payload_bytes
    layers = range(L) if layers is None else layers
    experts = range(E) if experts is None else experts
    jobs = [(l, e) for l in layers for e in experts]
    threads = threads or min(32, os.cpu_count() or 1)

    def job(le):
        l, e = le
        expert_payload(w, l, e, out=store[l, e])

    with _cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(job, jobs))
