"""Pins for the oracle's quantised formats and byte accounting (CPU only)."""
import os

import numpy as np
import pytest

import oracle
from oracle import formats


def _page_numbers(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "page_numbers.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, val = line.split()[:2]
            vals[key] = float(val)
    return vals


def test_fp16_known_values():
    bits = np.array([0x3C00, 0x3555, 0x0001, 0x7BFF, 0xC000, 0x0000, 0x8000, 0x0400],
                    dtype=np.uint16)
    want = [1.0, 0.333251953125, 2.0 ** -24, 65504.0, -2.0, 0.0, -0.0, 2.0 ** -14]
    assert oracle.f16_bits_to_f64(bits).tolist() == want


def test_bf16_known_values():
    bits = np.array([0x3F80, 0xC000, 0x3EAB, 0x0001, 0x7F7F], dtype=np.uint16)
    want = [1.0, -2.0, 0.333984375, 2.0 ** -133, 3.3895313892515355e38]
    assert oracle.bf16_bits_to_f64(bits).tolist() == want


def test_q8_0_exhaustive_int8():
    # every int8 code with d = 1.0 and d = 0.5 (exact in fp16)
    q = np.arange(-128, 128, dtype=np.int64).astype(np.int8).reshape(8, 32)
    one = np.full((8, 1), 0x3C00, dtype=np.uint16)
    half = np.full((8, 1), 0x3800, dtype=np.uint16)
    assert np.array_equal(formats.dequant_q8_0(q, one), np.arange(-128, 128).reshape(8, 32))
    assert np.array_equal(formats.dequant_q8_0(q, half), np.arange(-128, 128).reshape(8, 32) / 2)


def test_q8_0_scale_per_block():
    # two blocks per row, each with its own scale
    q = np.full((2, 64), 3, dtype=np.int8)
    d = np.array([[0x3C00, 0x4000], [0x3400, 0xBC00]], dtype=np.uint16)  # 1, 2, 0.25, -1
    x = formats.dequant_q8_0(q, d)
    assert np.all(x[0, :32] == 3) and np.all(x[0, 32:] == 6)
    assert np.all(x[1, :32] == 0.75) and np.all(x[1, 32:] == -3)


def test_q4_0_nibble_order_and_offset():
    # byte j: low nibble j, high nibble 15 - j  ->  element j = j - 8,
    # element j + 16 = (15 - j) - 8, times d
    b = np.array([(j & 0xF) | ((15 - j) << 4) for j in range(16)], dtype=np.uint8).reshape(1, 16)
    for bits, d in ((0x3C00, 1.0), (0x3800, 0.5)):
        x = formats.dequant_q4_0(b, np.array([[bits]], dtype=np.uint16))
        want = [d * (j - 8) for j in range(16)] + [d * (7 - j) for j in range(16)]
        assert x.ravel().tolist() == want


def test_q4_0_exhaustive_nibbles():
    # all 256 byte values across 16 blocks: low nibble -> element j,
    # high nibble -> element j + 16
    b = np.arange(256, dtype=np.uint8).reshape(16, 16)
    x = formats.dequant_q4_0(b.reshape(1, 256), np.full((1, 16), 0x3C00, dtype=np.uint16))
    x = x.reshape(16, 32)
    for blk in range(16):
        for j in range(16):
            v = blk * 16 + j
            assert x[blk, j] == (v & 15) - 8
            assert x[blk, j + 16] == (v >> 4) - 8


def test_i4_g64_nibble_order_scale_and_bias():
    # byte j: element 2j in the low nibble, element 2j + 1 in the high one;
    # x = s*q + b with one (s, b) per 64 weights
    b = np.array([(j & 0xF) | ((15 - (j & 0xF)) << 4) for j in range(64)], dtype=np.uint8).reshape(1, 64)
    # two groups: (s, b) = (1, 0) and (0.5, -2) as bf16 bits
    sb = np.array([[[0x3F80, 0x0000], [0x3F00, 0xC000]]], dtype=np.uint16)
    x = formats.dequant_i4_g64(b, sb).ravel()
    for j in range(64):
        lo, hi = j & 0xF, 15 - (j & 0xF)
        s_, b_ = (1.0, 0.0) if j < 32 else (0.5, -2.0)
        assert x[2 * j] == s_ * lo + b_ and x[2 * j + 1] == s_ * hi + b_


def test_i4_g64_exhaustive_codes():
    # every byte value, with an exactly representable scale and bias
    b = np.arange(256, dtype=np.uint8).reshape(1, 256)  # 512 weights, 8 groups
    s_bits, b_bits = 0x3E80, 0xBF40  # 0.25, -0.75
    sb = np.tile(np.array([s_bits, b_bits], dtype=np.uint16), (1, 8, 1))
    x = formats.dequant_i4_g64(b, sb).ravel()
    for v in range(256):
        assert x[2 * v] == 0.25 * (v & 15) - 0.75
        assert x[2 * v + 1] == 0.25 * (v >> 4) - 0.75


def test_i4_g64_expert_layout():
    # quant plane then (scale, bias) plane per matrix; gate/up/down in order
    H, I = 128, 64
    parts = []
    for m, (rows, k) in enumerate(((I, H), (I, H), (H, I))):
        nib = np.full(rows * k // 2, (m + 1) | ((m + 2) << 4), dtype=np.uint8)
        parts.append(nib)
        sb = np.tile(np.array([0x3F80, [0x0000, 0x3F80, 0x4000][m]], dtype="<u2"), rows * (k // 64))
        parts.append(sb.view(np.uint8))
    p = np.concatenate(parts)
    assert p.size == oracle.payload_bytes(H, I, oracle.I4_G64) == oracle.payload_bytes(H, I, oracle.Q4_0)
    wg, wu, wd = oracle.expert_matrices(p, H, I, oracle.I4_G64)
    for m, w in enumerate((wg, wu, wd)):
        bias = [0.0, 1.0, 2.0][m]
        assert np.all(w[:, 0::2] == (m + 1) + bias) and np.all(w[:, 1::2] == (m + 2) + bias)


def test_i4_g64_payload_matches_routide():
    # Routide §3.2: 540 MiB for 320 experts at hidden 2048, intermediate 512
    # is 4.5 bits per weight: 36 B per 64 affine INT4 weights
    assert oracle.payload_bytes(2048, 512, oracle.I4_G64) * 320 == 540 * 2**20


def _hand_payload_q8(H, I):
    """Payload whose quant value at (matrix m, row r, col c) is
    (m*7 + r*3 + c) mod 101 - 50, with every scale of matrix m equal to 2^-m."""
    parts = []
    for m, (rows, k) in enumerate(((I, H), (I, H), (H, I))):
        r = np.arange(rows)[:, None]
        c = np.arange(k)[None, :]
        q = ((m * 7 + r * 3 + c) % 101 - 50).astype(np.int8)
        parts.append(q.view(np.uint8).ravel())
        d = np.full(rows * (k // 32), [0x3C00, 0x3800, 0x3400][m], dtype="<u2")
        parts.append(d.view(np.uint8))
    return np.concatenate(parts)


def test_expert_layout_q8_0():
    H, I = 64, 32  # distinct so a transposed matrix would not fit
    p = _hand_payload_q8(H, I)
    assert p.size == oracle.payload_bytes(H, I, oracle.Q8_0)
    wg, wu, wd = oracle.expert_matrices(p, H, I, oracle.Q8_0)
    assert wg.shape == (I, H) and wu.shape == (I, H) and wd.shape == (H, I)
    for m, w in enumerate((wg, wu, wd)):
        rows, k = w.shape
        for r in (0, 1, rows - 1):
            for c in sorted({0, 5, 31, min(32, k - 1), k - 1}):
                assert w[r, c] == ((m * 7 + r * 3 + c) % 101 - 50) * 2.0 ** -m


def test_payload_bytes_match_pages(golden_dir):
    v = _page_numbers(golden_dir)
    # MawForge §V-C: the 50% -> 65% step of the Gemma Q8 static minimum is 15%
    # of every routed expert's bytes.
    per_pct = (v["gemma_static_min_65_gib"] - v["gemma_static_min_50_gib"]) / 0.15
    total = v["gemma_layers"] * v["gemma_experts"] * oracle.payload_bytes(2816, 704, oracle.Q8_0)
    assert abs(total / 2 ** 30 - per_pct) < 1e-3
    # Routide §3.2: 540 MiB for 320 experts at hidden 2048, intermediate 512, 4.5 bits/weight
    per_expert = v["routide_all_miss_mib"] * 2 ** 20 / v["routide_distinct_experts"]
    assert oracle.payload_bytes(2048, 512, oracle.Q4_0) == per_expert
    # Routide §5.1: 303 payloads fit in 512 MiB, below the 313 reuse threshold
    s = oracle.slot_count(int(v["routide_budget_mib"]) * 2 ** 20,
                          oracle.payload_bytes(2048, 512, oracle.Q4_0))
    assert s == v["routide_fitting_payloads"] and s < v["routide_reuse_threshold"]


def test_workload_payload_sizes():
    from workloads import WORKLOADS
    want = {"tiny": 104448, "decode": 3342336, "mtp_decode": 1769472,
            "prefill": 3342336, "wide_prefill": 6319104, "i4_decode": 1769472}
    for name, w in WORKLOADS.items():
        assert oracle.payload_bytes(w.hidden, w.inter, w.quant) == want[name]
        assert w.payload_bytes == want[name]


@pytest.mark.parametrize("name", ["tiny", "mtp_decode", "i4_decode"])
def test_generated_payload_ranges(name):
    from workloads import WORKLOADS, expert_payload
    w = WORKLOADS[name]
    if name in ("mtp_decode", "i4_decode"):
        w = __import__("workloads").with_changes(w, hidden=256, inter=64)
    p = expert_payload(w, 0, 3)
    wg, wu, wd = oracle.expert_matrices(p, w.hidden, w.inter, w.quant)
    for m in (wg, wu, wd):
        assert np.isfinite(m).all()
    # scales are fp16 values in [1e-3, 2e-2] (after rounding), quants in range
    if w.quant == oracle.Q8_0:
        q = p[:w.inter * w.hidden].view(np.int8)
        assert q.min() >= -127 and q.max() <= 127
        assert len(np.unique(q)) == 255
    else:
        nib = p[:w.inter * w.hidden // 2]
        assert len(np.unique(nib & 15)) == 16 and len(np.unique(nib >> 4)) == 16
    off = w.inter * w.hidden if w.quant == oracle.Q8_0 else w.inter * w.hidden // 2
    if w.quant == oracle.I4_G64:
        sb = p[off:off + w.inter * w.hidden // 16].view("<u2").reshape(-1, 2)
        sc, bi = oracle.bf16_bits_to_f64(sb[:, 0]), oracle.bf16_bits_to_f64(sb[:, 1])
        # bf16 rounding: within 2^-8 relative of the drawn values
        assert sc.min() >= 1e-3 * (1 - 2**-8) and sc.max() <= 2e-2 * (1 + 2**-8)
        assert np.all(bi <= -6.9 * sc) and np.all(bi >= -8.1 * sc)
        return
    d = oracle.f16_bits_to_f64(p[off:off + w.inter * w.hidden // 16].view("<u2"))
    assert d.min() >= 0.000999 and d.max() <= 0.02001


def test_generator_deterministic():
    from workloads import WORKLOADS, expert_payload, activations, router_weights
    w = WORKLOADS["tiny"]
    assert np.array_equal(expert_payload(w, 0, 5), expert_payload(w, 0, 5))
    assert not np.array_equal(expert_payload(w, 0, 5), expert_payload(w, 0, 6))
    assert np.array_equal(activations(w, 0), activations(w, 0))
    assert np.array_equal(router_weights(w, 0), router_weights(w, 0))
    d = WORKLOADS["decode"]
    a = activations(d, 3, 4, token0=10)
    b = activations(d, 3)[10:14]
    assert np.array_equal(a, b)
