"""Quantised expert formats (oracle; test infrastructure only).

GGUF Q8_0 and Q4_0 blocks of 32 weights with one fp16 scale d each
(MawForge §III and §V-B name GGUF Q8_0 expert tensors; Routide §3.1 stores
gate, up and down projections per expert):

* Q8_0: x = d * q, q a signed byte;
* Q4_0: x = d * (q - 8), q an unsigned nibble; byte j of a block holds
  element j (low nibble) and element j + 16 (high nibble).
* I4_G64 (affine INT4, group size 64; Routide §3.1 stores gate, up and down
  with scales and biases, BF16 quantisation metadata): x = s * q + b, q an
  unsigned nibble, one bf16 scale s and one bf16 bias b per 64 weights; byte
  j of a row holds element 2j (low nibble) and element 2j + 1 (high nibble).
  At 36 B per 64 weights it is 4.5 bits per weight, as Q4_0.

An expert's payload stores, for gate [I, H], up [I, H] and down [H, I] in that
order, a quant plane (all rows, row-major) followed by a scale plane
(fp16 [rows][K/32]; for I4_G64 the (scale, bias) bf16 pairs [rows][K/64][2]).
Blocks run along the input dimension K.
"""
from __future__ import annotations

import numpy as np

Q8_0 = 0
Q4_0 = 1
I4_G64 = 2


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 numbers given as uint16 bit patterns."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of IEEE binary16 numbers given as uint16 bit patterns."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def block_bytes(quant: int) -> int:
    return 34 if quant == Q8_0 else 18


def payload_bytes(hidden: int, inter: int, quant: int) -> int:
    """Bytes of one expert: three matrices of hidden*inter weights, stored as
    32-weight blocks of 34 B (Q8_0) or 18 B (Q4_0)."""
    return 3 * (hidden * inter // 32) * block_bytes(quant)


def dequant_q8_0(q: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """q int8 [rows, K], d_bits uint16 [rows, K/32] -> fp64 [rows, K], x = d*q."""
    rows, k = q.shape
    d = f16_bits_to_f64(d_bits).reshape(rows, k // 32)
    x = q.astype(np.float64).reshape(rows, k // 32, 32) * d[:, :, None]
    return x.reshape(rows, k)


def dequant_q4_0(nib: np.ndarray, d_bits: np.ndarray) -> np.ndarray:
    """nib uint8 [rows, K/2], d_bits uint16 [rows, K/32] -> fp64 [rows, K],
    x = d*(q-8) with the low/high nibble order of each 16-byte block."""
    rows, kh = nib.shape
    k = 2 * kh
    b = nib.reshape(rows, k // 32, 16)
    q = np.empty((rows, k // 32, 32), dtype=np.int64)
    q[:, :, :16] = b & 0x0F
    q[:, :, 16:] = b >> 4
    d = f16_bits_to_f64(d_bits).reshape(rows, k // 32)
    x = (q.astype(np.float64) - 8.0) * d[:, :, None]
    return x.reshape(rows, k)


def dequant_i4_g64(nib: np.ndarray, sb_bits: np.ndarray) -> np.ndarray:
    """nib uint8 [rows, K/2], sb_bits uint16 [rows, K/64, 2] (bf16 scale,
    bf16 bias) -> fp64 [rows, K], x = s*q + b; byte j holds elements 2j (low
    nibble) and 2j+1 (high nibble)."""
    rows, kh = nib.shape
    k = 2 * kh
    q = np.empty((rows, k), dtype=np.int64)
    q[:, 0::2] = nib & 0x0F
    q[:, 1::2] = nib >> 4
    s = bf16_bits_to_f64(sb_bits[:, :, 0]).reshape(rows, k // 64)
    b = bf16_bits_to_f64(sb_bits[:, :, 1]).reshape(rows, k // 64)
    x = q.astype(np.float64).reshape(rows, k // 64, 64) * s[:, :, None] + b[:, :, None]
    return x.reshape(rows, k)


def _matrix(buf: np.ndarray, off: int, rows: int, k: int, quant: int):
    if quant == Q8_0:
        qn = rows * k
        q = buf[off:off + qn].view(np.int8).reshape(rows, k)
    else:
        qn = rows * k // 2
        q = buf[off:off + qn].reshape(rows, k // 2)
    off += qn
    sn = rows * (k // 32) * 2
    if quant == I4_G64:
        sb = buf[off:off + sn].view("<u2").reshape(rows, k // 64, 2)
        return dequant_i4_g64(q, sb), off + sn
    d = buf[off:off + sn].view("<u2").reshape(rows, k // 32)
    off += sn
    x = dequant_q8_0(q, d) if quant == Q8_0 else dequant_q4_0(q, d)
    return x, off


def expert_matrices(payload: np.ndarray, hidden: int, inter: int, quant: int):
    """Dequantise one expert payload (uint8) to fp64 (Wg [I,H], Wu [I,H], Wd [H,I])."""
    buf = np.ascontiguousarray(payload, dtype=np.uint8)
    assert buf.shape == (payload_bytes(hidden, inter, quant),), buf.shape
    wg, off = _matrix(buf, 0, inter, hidden, quant)
    wu, off = _matrix(buf, off, inter, hidden, quant)
    wd, off = _matrix(buf, off, hidden, inter, quant)
    assert off == buf.shape[0]
    return wg, wu, wd
