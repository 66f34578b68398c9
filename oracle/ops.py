"""Float64 building blocks of the decode step (test infrastructure; see package doc)."""

from __future__ import annotations

import numpy as np


def matvec(w: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y = W x for W [rows = outputs, cols = inputs]; x [cols] or [B, cols] -> [rows] / [B, rows].

    Weight orientation: GGUF rows are output features, each row cols/32
    consecutive blocks ("EdgeRunner Core Architecture" section 3.2 counts
    blocks per element along a row).
    """
    w = np.asarray(w, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    return x @ w.T


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis.

    "EdgeRunner Core Architecture" section 6 (input * RMS(input)^-1 * weight;
    the bias term is absent: alpaca.swift README, "Limitations", no biases).
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def rope(u: np.ndarray, pos: int, base: float) -> np.ndarray:
    """Rotate each head vector u[..., hd] of one token at position `pos`.

    "EdgeRunner Core Architecture" section 7: adjacent pairs (2i, 2i+1),
    u'[2i] = u[2i] cos - u[2i+1] sin, u'[2i+1] = u[2i+1] cos + u[2i] sin, with
    the angle pos * base^(-2i/hd) (frequency base "theta", scaling factor 1).
    """
    u = np.asarray(u, dtype=np.float64)
    hd = u.shape[-1]
    i = np.arange(hd // 2, dtype=np.float64)
    theta = float(pos) * np.power(float(base), -2.0 * i / hd)
    c, s = np.cos(theta), np.sin(theta)
    ev, od = u[..., 0::2], u[..., 1::2]
    out = np.empty_like(u)
    out[..., 0::2] = ev * c - od * s
    out[..., 1::2] = od * c + ev * s
    return out


def softmax(s: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis."""
    s = np.asarray(s, dtype=np.float64)
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_gqa(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Decode attention of one token over cache rows 0..T-1 (causal, inclusive).

    q [H, hd]; k, v [T, KV, hd] -> o [H, hd].  Query head h reads KV head
    h // (H / KV) (contiguous groups of gqaRatio = H / KV heads), scores are
    q . k_t / sqrt(hd), softmax over t, o = sum_t a_t v_t.
    "EdgeRunner Core Architecture" sections 1.1 (gqaRatio) and 5.2 (GQA params:
    scale 1/sqrt(headDim), causal, a query at position p attends 0..p).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    H, hd = q.shape
    KV = k.shape[1]
    group = H // KV
    o = np.empty((H, hd), dtype=np.float64)
    for h in range(H):
        g = h // group
        s = k[:, g, :] @ q[h] / np.sqrt(hd)
        o[h] = softmax(s) @ v[:, g, :]
    return o


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z * sigmoid(z) = z / (1 + e^-z) ("EdgeRunner Core Architecture" section 8)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """SiLU(gate) * up ("EdgeRunner Core Architecture" section 8)."""
    return silu(gate) * np.asarray(up, dtype=np.float64)
