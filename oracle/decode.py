"""Float64 decode step of a block-quantized Llama decoder (test infrastructure; see package doc).

Per layer ("EdgeRunner Core Architecture" section 5.1, decode case of one token
per sequence):

  h  = rmsnorm(x, attn_norm)
  q, k, v = Wq h, Wk h, Wv h
  q, k = rope(q, pos), rope(k, pos)                       (section 7)
  Kc[pos], Vc[pos] = fp16(k), fp16(v)                     (section 4.3: K/V written
                                                           at row `pos`, fp16 cache)
  o  = GQA attention of q over Kc[0..pos], Vc[0..pos]     (section 5.2)
  x  = x + Wo o
  h2 = rmsnorm(x, ffn_norm)
  x  = x + Wdown (silu(Wgate h2) * (Wup h2))              (section 8)

then logits = Wout rmsnorm(x, output_norm) and the greedy token is the argmax
(section 2.3, greedyToken with a hasNonFinite flag).  The embedding is a row of
token_embd; with a tied head that same matrix is the output projection (alpaca.swift
README, "Capabilities": tied or untied output head).

Readings where the pages are silent (each listed in the design notes):
  * cached K rows are post-RoPE keys; V is not rotated;
  * argmax ties go to the lowest index, NaN never wins, any non-finite logit
    sets the flag;
  * prefilled cache rows are given, already in cache form (fp16);
  * a Q8_0 cache (OracleCache kv_type "q8_0", an option the pages name without
    a quantiser) stores each head's row as Q8_0 blocks quantised by
    blocks.quantize_kv_q8_0, and attention reads d * q.
"""

from __future__ import annotations

import dataclasses
from typing import Callable, Mapping

import numpy as np

from .blocks import dequant, dequant_kv_q8_0, dequant_rows, quantize_kv_q8_0
from .ops import attention_gqa, matvec, rmsnorm, rope, swiglu


@dataclasses.dataclass(frozen=True)
class OracleConfig:
    n_layers: int
    dim: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_base: float
    rms_eps: float
    w_type: str
    tied: bool

    @property
    def qd(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kvd(self) -> int:
        return self.n_kv_heads * self.head_dim


class OracleModel:
    """Config plus a tensor source.

    `tensors` maps GGUF names ("blk.{l}.attn_q.weight", "token_embd.weight", ...)
    to stored arrays: float32 gains, float16 embedding, or uint8 block bytes.
    It may be a lazy mapping (only `__getitem__` is used).  With
    `cache_dequant`, each dequantised matrix is kept after first use, as
    `cache_dtype`.  float32 halves the memory of a large model and loses
    nothing: every dequantised value d * q has at most 19 significant bits
    (an 11-bit fp16 significand times an integer of at most 8 bits), and an
    fp16 embedding value is exact in float32 too; `matvec` widens the stored
    matrix back to float64, so the products are the same.
    """

    def __init__(self, cfg: OracleConfig, tensors: Mapping[str, np.ndarray] | Callable[[str], np.ndarray],
                 cache_dequant: bool = False, cache_dtype=np.float64):
        self.cfg = cfg
        self._get = tensors if callable(tensors) else tensors.__getitem__
        self._cache: dict[str, np.ndarray] | None = {} if cache_dequant else None
        self._cache_dtype = np.dtype(cache_dtype)
        if self._cache_dtype not in (np.dtype(np.float64), np.dtype(np.float32)):
            raise ValueError("cache_dtype must be float64 or float32")

    def _shape(self, name: str) -> tuple[str, int, int]:
        c = self.cfg
        leaf = name.split(".")[-2] if name.startswith("blk.") else name.split(".")[0]
        shapes = {
            "attn_q": (c.qd, c.dim), "attn_k": (c.kvd, c.dim), "attn_v": (c.kvd, c.dim),
            "attn_output": (c.dim, c.qd), "ffn_gate": (c.ffn_dim, c.dim), "ffn_up": (c.ffn_dim, c.dim),
            "ffn_down": (c.dim, c.ffn_dim), "output": (c.vocab, c.dim), "token_embd": (c.vocab, c.dim),
        }
        kind = c.w_type
        if leaf == "token_embd" and not c.tied:
            kind = "f16"
        return (kind,) + shapes[leaf]

    def matrix(self, name: str) -> np.ndarray:
        if self._cache is not None and name in self._cache:
            return self._cache[name]
        kind, rows, cols = self._shape(name)
        w = dequant(self._get(name), kind, rows, cols)
        if self._cache is not None:
            if self._cache_dtype != w.dtype:
                narrow = w.astype(self._cache_dtype)
                if not np.array_equal(narrow, w):
                    raise ValueError(f"{name}: dequantised values are not exact in {self._cache_dtype}")
                w = narrow
            self._cache[name] = w
        return w

    def gain(self, name: str) -> np.ndarray:
        return np.asarray(self._get(name), dtype=np.float32).astype(np.float64)

    def embedding_rows(self, tokens) -> np.ndarray:
        kind, rows, cols = self._shape("token_embd.weight")
        return dequant_rows(self._get("token_embd.weight"), kind, rows, cols, tokens)

    def head_name(self) -> str:
        return "token_embd.weight" if self.cfg.tied else "output.weight"


class OracleCache:
    """K and V rows per (sequence, layer): arrays [capacity, n_kv_heads, head_dim].

    kv_type "f16" (the pages' default cache precision): the rows are fp16.
    kv_type "q8_0": each head's row is stored as Q8_0 blocks (blocks.quantize_kv_q8_0); k / v then hold
    the dequantised values d * q (exact in float32) and kd / kq / vd / vq the blocks themselves.
    """

    def __init__(self, cfg: OracleConfig, batch: int, capacity: int, kv_type: str = "f16"):
        if kv_type not in ("f16", "q8_0"):
            raise ValueError(kv_type)
        self.cfg, self.batch, self.capacity, self.kv_type = cfg, batch, capacity, kv_type
        shp = (capacity, cfg.n_kv_heads, cfg.head_dim)
        dt = np.float16 if kv_type == "f16" else np.float32
        self.k = [[np.zeros(shp, dt) for _ in range(cfg.n_layers)] for _ in range(batch)]
        self.v = [[np.zeros(shp, dt) for _ in range(cfg.n_layers)] for _ in range(batch)]
        if kv_type == "q8_0":
            dshp = (capacity, cfg.n_kv_heads, cfg.head_dim // 32)
            self.kd = [[np.zeros(dshp, np.float16) for _ in range(cfg.n_layers)] for _ in range(batch)]
            self.vd = [[np.zeros(dshp, np.float16) for _ in range(cfg.n_layers)] for _ in range(batch)]
            self.kq = [[np.zeros(shp, np.int8) for _ in range(cfg.n_layers)] for _ in range(batch)]
            self.vq = [[np.zeros(shp, np.int8) for _ in range(cfg.n_layers)] for _ in range(batch)]

    def put(self, b: int, layer: int, rows: slice | int, k, v) -> None:
        """Store K and V values [..., n_kv_heads, head_dim] at `rows` in the cache's precision."""
        if self.kv_type == "f16":
            self.k[b][layer][rows] = np.asarray(k, np.float64).astype(np.float16)
            self.v[b][layer][rows] = np.asarray(v, np.float64).astype(np.float16)
            return
        for vals, full, ds, qs in ((k, self.k, self.kd, self.kq), (v, self.v, self.vd, self.vq)):
            d, q = quantize_kv_q8_0(np.asarray(vals, np.float64).astype(np.float32))
            ds[b][layer][rows] = d
            qs[b][layer][rows] = q
            full[b][layer][rows] = dequant_kv_q8_0(d, q).astype(np.float32)

    def fill(self, b: int, layer: int, k_rows: np.ndarray, v_rows: np.ndarray, start: int = 0) -> None:
        """Store token-major fp16 rows [n, n_kv_heads*head_dim] at rows start..start+n-1."""
        n = k_rows.shape[0]
        c = self.cfg
        k = np.asarray(k_rows, np.float16).reshape(n, c.n_kv_heads, c.head_dim)
        v = np.asarray(v_rows, np.float16).reshape(n, c.n_kv_heads, c.head_dim)
        self.put(b, layer, slice(start, start + n), k, v)


def _argmax_flag(logits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    finite = np.isfinite(logits)
    nonfinite = ~finite.all(axis=-1)
    clean = np.where(np.isnan(logits), -np.inf, logits)
    return np.argmax(clean, axis=-1).astype(np.int64), nonfinite


def decode_step(model: OracleModel, cache: OracleCache, tokens, positions,
                seqs=None) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """One decode step for every sequence b (or only `seqs`): token tokens[b] at position positions[b].

    Writes the new K/V rows into `cache` and returns (logits [B, vocab] float64,
    argmax [B], non_finite [B]) for the sequences computed (in `seqs` order).
    """
    c = model.cfg
    seqs = list(range(len(tokens))) if seqs is None else list(seqs)
    tok = np.asarray(tokens)[seqs]
    pos = np.asarray(positions)[seqs]
    B = len(seqs)
    x = model.embedding_rows(tok)                                   # [B, dim]
    for l in range(c.n_layers):
        p = f"blk.{l}."
        h = rmsnorm(x, model.gain(p + "attn_norm.weight"), c.rms_eps)
        q = matvec(model.matrix(p + "attn_q.weight"), h)           # [B, qd]
        k = matvec(model.matrix(p + "attn_k.weight"), h)           # [B, kvd]
        v = matvec(model.matrix(p + "attn_v.weight"), h)
        o = np.empty((B, c.qd), dtype=np.float64)
        for i, b in enumerate(seqs):
            pb = int(pos[i])
            qh = rope(q[i].reshape(c.n_heads, c.head_dim), pb, c.rope_base)
            kh = rope(k[i].reshape(c.n_kv_heads, c.head_dim), pb, c.rope_base)
            cache.put(b, l, pb, kh, v[i].reshape(c.n_kv_heads, c.head_dim))
            o[i] = attention_gqa(qh, cache.k[b][l][:pb + 1], cache.v[b][l][:pb + 1]).reshape(-1)
        x = x + matvec(model.matrix(p + "attn_output.weight"), o)
        h2 = rmsnorm(x, model.gain(p + "ffn_norm.weight"), c.rms_eps)
        a = swiglu(matvec(model.matrix(p + "ffn_gate.weight"), h2), matvec(model.matrix(p + "ffn_up.weight"), h2))
        x = x + matvec(model.matrix(p + "ffn_down.weight"), a)
    hf = rmsnorm(x, model.gain("output_norm.weight"), c.rms_eps)
    logits = matvec(model.matrix(model.head_name()), hf)
    am, nf = _argmax_flag(logits)
    return logits, am, nf


def greedy(model: OracleModel, cache: OracleCache, tokens, positions, steps: int, seqs=None):
    """Chain `steps` greedy decode steps: next token = argmax, position + 1.

    Returns (tokens fed per step [steps, B], logits per step [steps, B, vocab]).
    """
    tok = np.array(tokens, dtype=np.int64)
    pos = np.array(positions, dtype=np.int64)
    seqs = list(range(len(tok))) if seqs is None else list(seqs)
    fed, out = [], []
    for _ in range(steps):
        fed.append(tok[seqs].copy())
        logits, am, _ = decode_step(model, cache, tok, pos, seqs=seqs)
        out.append(logits)
        tok[seqs] = am
        pos[seqs] += 1
    return np.array(fed), np.array(out)


def uncached_logits(model: OracleModel, token_seq, kv_type: str = "f16") -> np.ndarray:
    """Logits at the last position of `token_seq` (positions 0..n-1) recomputed from scratch.

    Every position's K and V are computed together, rounded as a cache of
    `kv_type` would hold them (fp16, or Q8_0 blocks), and each query attends to
    positions 0..itself.
    Used to check incremental decoding ("cached == uncached", alpaca.swift README,
    "Numerical validation", levels 2-4).
    """
    c = model.cfg
    toks = np.asarray(token_seq)
    n = len(toks)
    x = model.embedding_rows(toks)                                  # [n, dim]
    for l in range(c.n_layers):
        p = f"blk.{l}."
        h = rmsnorm(x, model.gain(p + "attn_norm.weight"), c.rms_eps)
        q = matvec(model.matrix(p + "attn_q.weight"), h)
        k = matvec(model.matrix(p + "attn_k.weight"), h)
        v = matvec(model.matrix(p + "attn_v.weight"), h)
        K = np.stack([rope(k[t].reshape(c.n_kv_heads, c.head_dim), t, c.rope_base) for t in range(n)])
        V = v.reshape(n, c.n_kv_heads, c.head_dim)
        if kv_type == "f16":
            K, V = K.astype(np.float16), V.astype(np.float16)
        else:
            K = dequant_kv_q8_0(*quantize_kv_q8_0(K.astype(np.float32)))
            V = dequant_kv_q8_0(*quantize_kv_q8_0(V.astype(np.float32)))
        o = np.stack([attention_gqa(rope(q[t].reshape(c.n_heads, c.head_dim), t, c.rope_base),
                                    K[:t + 1], V[:t + 1]).reshape(-1) for t in range(n)])
        x = x + matvec(model.matrix(p + "attn_output.weight"), o)
        h2 = rmsnorm(x, model.gain(p + "ffn_norm.weight"), c.rms_eps)
        a = swiglu(matvec(model.matrix(p + "ffn_gate.weight"), h2), matvec(model.matrix(p + "ffn_up.weight"), h2))
        x = x + matvec(model.matrix(p + "ffn_down.weight"), a)
    hf = rmsnorm(x[-1:], model.gain("output_norm.weight"), c.rms_eps)
    return matvec(model.matrix(model.head_name()), hf)[0]
