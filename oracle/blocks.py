"""GGUF block dequantisation, float64 (test infrastructure; see package doc).

Sources: "EdgeRunner Core Architecture" section 1.3 (type codes and bytes per
block: Q4_0 = 2, 18 bytes; Q8_0 = 8, 34 bytes), section 3.1 (format table) and
section 3.2 (Q8_0 block = [2-byte fp16 scale][32 one-byte quantised values]).
The pages give Q4_0 only its size; its nibble order (element j in the low
nibble of byte j, element j + 16 in the high nibble) and the offset of 8 are
the workload statement's reading of the format.

Every value is d * q with d the block's fp16 scale and q an integer of at
most 8 bits, so the float64 result is exact (and equals its float32 rounding).
"""

from __future__ import annotations

import numpy as np

QK = 32
BLOCK_BYTES = {"q8_0": 2 + QK, "q4_0": 2 + QK // 2}


def _blocks(raw: np.ndarray, rows: int, cols: int, nbytes: int) -> np.ndarray:
    if cols % QK:
        raise ValueError("cols must be a multiple of 32")
    a = np.ascontiguousarray(raw, dtype=np.uint8).reshape(rows, cols // QK, nbytes)
    return a


def _scales(blk: np.ndarray) -> np.ndarray:
    # bytes 0-1 of a block: IEEE binary16, little-endian
    return np.ascontiguousarray(blk[..., :2]).view("<f2")[..., 0].astype(np.float64)


def dequant_q8_0(raw: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Q8_0 bytes [rows, cols/32*34] -> float64 [rows, cols]: w_j = d * q_j, q_j int8."""
    blk = _blocks(raw, rows, cols, BLOCK_BYTES["q8_0"])
    d = _scales(blk)
    q = np.ascontiguousarray(blk[..., 2:]).view(np.int8).astype(np.float64)
    return (d[..., None] * q).reshape(rows, cols)


def dequant_q4_0(raw: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Q4_0 bytes [rows, cols/32*18] -> float64 [rows, cols].

    For j < 16: w_j = d * ((b_j & 15) - 8) and w_{j+16} = d * ((b_j >> 4) - 8).
    """
    blk = _blocks(raw, rows, cols, BLOCK_BYTES["q4_0"])
    d = _scales(blk)
    b = blk[..., 2:].astype(np.int64)
    q = np.empty(b.shape[:-1] + (QK,), dtype=np.float64)
    q[..., :16] = (b & 0xF) - 8
    q[..., 16:] = (b >> 4) - 8
    return (d[..., None] * q).reshape(rows, cols)


def dequant(raw: np.ndarray, kind: str, rows: int, cols: int) -> np.ndarray:
    if kind == "q8_0":
        return dequant_q8_0(raw, rows, cols)
    if kind == "q4_0":
        return dequant_q4_0(raw, rows, cols)
    if kind == "f16":
        return np.asarray(raw, dtype=np.float16).reshape(rows, cols).astype(np.float64)
    if kind == "f32":
        return np.asarray(raw, dtype=np.float32).reshape(rows, cols).astype(np.float64)
    raise ValueError(kind)


def dequant_rows(raw: np.ndarray, kind: str, rows: int, cols: int, idx) -> np.ndarray:
    """Dequantise only rows `idx` (a row gather, as an embedding lookup does)."""
    idx = np.atleast_1d(np.asarray(idx, dtype=np.int64))
    sub = np.asarray(raw).reshape(rows, -1)[idx]
    return dequant(sub, kind, len(idx), cols)


def quantize_kv_q8_0(x) -> tuple[np.ndarray, np.ndarray]:
    """Quantise cache rows to Q8_0 blocks: x float32 [..., n] (n a multiple of 32) -> (d fp16 [..., n/32],
    q int8 [..., n]).

    The pages store K/V optionally as packed Q8_0 ("llama.cpp Metal (MPS) End-to-End Inference Path", P9
    quantized-KV flash-attention variants and section 5, minfer's packed Q8_0 cache; "EdgeRunner Core
    Architecture" section 4.1, cache precision options) but give no quantiser for the cache.  The reading
    here: the Q8_0 rule of the weights (scale = largest |x| / 127, q = round(x / scale)) with the division by
    the scale as stored, so that d * q is the stored value, and every step in float32, the precision the
    kernel takes the decision in:
      amax = max |x_j|                      (exact)
      d    = fp16(float32(amax / 127))      (float32 division, then round to nearest even in fp16)
      q_j  = clamp(round(float32(x_j / d)), -127, 127), round half away from zero; q = 0 when d = 0.
    """
    x = np.asarray(x, dtype=np.float32)
    if x.shape[-1] % QK:
        raise ValueError("rows must be whole blocks of 32")
    xb = x.reshape(x.shape[:-1] + (x.shape[-1] // QK, QK))
    amax = np.max(np.abs(xb), axis=-1)
    d = (amax / np.float32(127.0)).astype(np.float32).astype(np.float16)
    d32 = d.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d32[..., None] > 0, xb / d32[..., None], np.float32(0.0)).astype(np.float32)
    # round the float32 quotient half away from zero; the addition is exact in float64 (in float32 it
    # would round a quotient just below one half, such as 0.49999997, up to 1)
    r64 = r.astype(np.float64)
    q = np.sign(r64) * np.floor(np.abs(r64) + 0.5)
    q = np.clip(q, -127, 127).astype(np.int8)
    return d, q.reshape(x.shape)


def dequant_kv_q8_0(d, q) -> np.ndarray:
    """d fp16 [..., n/32], q int8 [..., n] -> float64 [..., n]: value = d * q (exact)."""
    d = np.asarray(d, dtype=np.float16).astype(np.float64)
    q = np.asarray(q, dtype=np.int8).astype(np.float64)
    qb = q.reshape(q.shape[:-1] + (q.shape[-1] // QK, QK))
    return (d[..., None] * qb).reshape(q.shape)
