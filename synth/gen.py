"""Workload shapes, seeded draws and the two block quantisers (see package doc)."""

from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# Bytes per 32-element block: fp16 scale + 32 int8 (Q8_0) or + 16 bytes of
# nibbles (Q4_0).  "EdgeRunner Core Architecture" section 3.1 table.
BLOCK_BYTES = {"q8_0": 34, "q4_0": 18}
QK = 32

SEED_WEIGHTS = 0
SEED_KV = 1


@dataclasses.dataclass(frozen=True)
class ModelShape:
    n_layers: int
    dim: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn_dim: int
    vocab: int
    rope_base: float
    rms_eps: float
    w_type: str          # "q8_0" | "q4_0": every 2-D weight
    tied: bool           # tied: token_embd is a w_type matrix and is the head

    @property
    def qd(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kvd(self) -> int:
        return self.n_kv_heads * self.head_dim


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    batch: int
    steps: int
    prefill: int
    first_token: int = 7
    kv_type: str = "f16"  # K/V cache storage: "f16" or "q8_0" (rows quantised as they are written)

    @property
    def capacity(self) -> int:
        return self.prefill + self.steps

    def tokens0(self) -> np.ndarray:
        return np.arange(self.batch, dtype=np.int32) + self.first_token

    def positions0(self) -> np.ndarray:
        return np.full(self.batch, self.prefill, dtype=np.int32)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


_SMOL = dict(n_layers=30, dim=576, n_heads=9, n_kv_heads=3, head_dim=64, ffn_dim=1536,
             vocab=49152, rope_base=10000.0, rms_eps=1e-5, tied=True)

WORKLOADS = {
    "tiny": Workload("tiny", ModelShape(n_layers=2, dim=576, n_heads=9, n_kv_heads=3, head_dim=64,
                                        ffn_dim=1536, vocab=4096, rope_base=10000.0, rms_eps=1e-5,
                                        w_type="q8_0", tied=False),
                     batch=1, steps=1, prefill=16),
    "smollm_q8": Workload("smollm_q8", ModelShape(w_type="q8_0", **_SMOL), batch=1, steps=64, prefill=2048),
    "smollm_q4": Workload("smollm_q4", ModelShape(w_type="q4_0", **_SMOL), batch=1, steps=64, prefill=16),
    "llama2_7b_q4": Workload("llama2_7b_q4", ModelShape(n_layers=32, dim=4096, n_heads=32, n_kv_heads=32,
                                                        head_dim=128, ffn_dim=11008, vocab=32000,
                                                        rope_base=10000.0, rms_eps=1e-5, w_type="q4_0",
                                                        tied=False),
                             batch=1, steps=64, prefill=4096),
    "llama3_8b_q8_b16": Workload("llama3_8b_q8_b16", ModelShape(n_layers=32, dim=4096, n_heads=32, n_kv_heads=8,
                                                                head_dim=128, ffn_dim=14336, vocab=128256,
                                                                rope_base=500000.0, rms_eps=1e-5, w_type="q8_0",
                                                                tied=False),
                                 batch=16, steps=32, prefill=8192),
}
# the same 16-sequence workload with a packed Q8_0 K/V cache (the same seeded rows, quantised when written)
WORKLOADS["llama3_8b_q8_b16_kvq8"] = WORKLOADS["llama3_8b_q8_b16"].with_(name="llama3_8b_q8_b16_kvq8",
                                                                         kv_type="q8_0")


def workload(name: str) -> Workload:
    return WORKLOADS[name]


# ----------------------------------------------------------------------------------------------
# tensor order, names and shapes (GGUF naming: "EdgeRunner Core Architecture" section 1.2)
# ----------------------------------------------------------------------------------------------
_LAYER_TENSORS = ("attn_norm", "attn_q", "attn_k", "attn_v", "attn_output",
                  "ffn_norm", "ffn_gate", "ffn_up", "ffn_down")


def tensor_names(shape: ModelShape) -> list[str]:
    """All tensor names in draw order (index in this list = the draw seed's second word)."""
    names = [f"blk.{l}.{t}.weight" for l in range(shape.n_layers) for t in _LAYER_TENSORS]
    names += ["token_embd.weight", "output_norm.weight", "output.weight"]
    return names


def tensor_kind(shape: ModelShape, name: str) -> tuple[str, tuple[int, ...]]:
    """(storage kind, logical shape [rows, cols] / [n]) of one tensor.

    Kinds: "f32" (norm gain), "f16" (untied embedding), "q8_0"/"q4_0" (2-D weight,
    rows = output features, cols = input features, each row cols/32 blocks).
    """
    s = shape
    leaf = name.split(".")[-2] if name.startswith("blk.") else name.split(".")[0]
    if leaf in ("attn_norm", "ffn_norm", "output_norm"):
        return "f32", (s.dim,)
    mats = {
        "attn_q": (s.qd, s.dim), "attn_k": (s.kvd, s.dim), "attn_v": (s.kvd, s.dim),
        "attn_output": (s.dim, s.qd), "ffn_gate": (s.ffn_dim, s.dim), "ffn_up": (s.ffn_dim, s.dim),
        "ffn_down": (s.dim, s.ffn_dim), "output": (s.vocab, s.dim),
    }
    if leaf == "token_embd":
        return (s.w_type if s.tied else "f16"), (s.vocab, s.dim)
    return s.w_type, mats[leaf]


# ----------------------------------------------------------------------------------------------
# quantisers (the generator's packing step; the recipe the workload statement gives)
# ----------------------------------------------------------------------------------------------
def _round_half_away(r: np.ndarray) -> np.ndarray:
    return np.sign(r) * np.floor(np.abs(r) + 0.5)


def _fp16_le_bytes(d: np.ndarray) -> np.ndarray:
    return d.astype("<f2").view(np.uint8).reshape(d.shape + (2,))


def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """float [rows, cols] -> Q8_0 bytes uint8 [rows, cols/32*34].

    Per 32-block in float64: d = max|x| / 127, q = round(x / d) (ties away from
    zero), stored [fp16 d (round to nearest even), 32 x int8 q].  An all-zero
    block stores d = 0, q = 0.
    """
    rows, cols = x.shape
    assert cols % QK == 0
    nb = cols // QK
    xb = np.asarray(x, dtype=np.float64).reshape(rows, nb, QK)
    d = np.abs(xb).max(axis=-1) / 127.0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d[..., None] > 0, xb / d[..., None], 0.0)
    q = _round_half_away(r).astype(np.int8)
    out = np.empty((rows, nb, 34), dtype=np.uint8)
    out[..., :2] = _fp16_le_bytes(d)
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(rows, nb * 34)


def quantize_q4_0(x: np.ndarray) -> np.ndarray:
    """float [rows, cols] -> Q4_0 bytes uint8 [rows, cols/32*18].

    Per 32-block in float64: m = the element of largest |x| (first on ties),
    d = m / -8, q = clamp(round(x / d) + 8, 0, 15) (ties away from zero); stored
    [fp16 d][16 bytes], byte j holding element j in its low nibble and element
    j + 16 in its high nibble.  An all-zero block stores d = 0 and q = 8.
    """
    rows, cols = x.shape
    assert cols % QK == 0
    nb = cols // QK
    xb = np.asarray(x, dtype=np.float64).reshape(rows, nb, QK)
    idx = np.argmax(np.abs(xb), axis=-1)
    m = np.take_along_axis(xb, idx[..., None], axis=-1)[..., 0]
    d = m / -8.0
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(d[..., None] != 0, xb / d[..., None], 0.0)
    q = np.clip(_round_half_away(r) + 8.0, 0, 15).astype(np.uint8)
    out = np.empty((rows, nb, 18), dtype=np.uint8)
    out[..., :2] = _fp16_le_bytes(d)
    out[..., 2:] = q[..., :16] | (q[..., 16:] << 4)
    return out.reshape(rows, nb * 18)


def quantize(x: np.ndarray, w_type: str, chunk_rows: int = 4096) -> np.ndarray:
    fn = {"q8_0": quantize_q8_0, "q4_0": quantize_q4_0}[w_type]
    rows = x.shape[0]
    if rows <= chunk_rows:
        return fn(x)
    return np.concatenate([fn(x[r:r + chunk_rows]) for r in range(0, rows, chunk_rows)], axis=0)


# ----------------------------------------------------------------------------------------------
# draws
# ----------------------------------------------------------------------------------------------
def weight_tensor(shape: ModelShape, name: str, seed: int = SEED_WEIGHTS) -> np.ndarray:
    """One tensor's stored bytes/values, drawn from its own seed.

    Returns float32 [n] (norm gain), float16 [vocab, dim] (untied embedding) or
    uint8 [rows, cols/32*bytes_per_block] (quantised weight).
    """
    names = tensor_names(shape)
    i = names.index(name)
    kind, shp = tensor_kind(shape, name)
    rng = np.random.default_rng([seed, i])
    if kind == "f32":
        return (np.float32(1.0) + np.float32(0.1) * rng.standard_normal(shp, dtype=np.float32)).astype(np.float32)
    if kind == "f16":
        return (np.float32(0.02) * rng.standard_normal(shp, dtype=np.float32)).astype(np.float16)
    rows, cols = shp
    out = np.empty((rows, cols // QK * BLOCK_BYTES[kind]), dtype=np.uint8)
    step = 8192
    for r in range(0, rows, step):  # same stream as one draw of the whole matrix
        n = min(step, rows - r)
        x = np.float32(0.02) * rng.standard_normal((n, cols), dtype=np.float32)
        out[r:r + n] = quantize(x, kind)
    return out


def model_weights(shape: ModelShape, threads: int = 8, seed: int = SEED_WEIGHTS) -> dict[str, np.ndarray]:
    """Every tensor of the model (the head is absent when tied)."""
    names = [n for n in tensor_names(shape) if not (shape.tied and n == "output.weight")]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        arrays = list(ex.map(lambda n: weight_tensor(shape, n, seed), names))
    return dict(zip(names, arrays))


def kv_prefill(wl: Workload, b: int, layer: int, seed: int = SEED_KV) -> tuple[np.ndarray, np.ndarray]:
    """fp16 K and V rows [prefill, n_kv_heads*head_dim] of sequence b, layer `layer`."""
    kvd = wl.shape.kvd
    rng = np.random.default_rng([seed, b, layer])
    k = rng.standard_normal((wl.prefill, kvd), dtype=np.float32).astype(np.float16)
    v = rng.standard_normal((wl.prefill, kvd), dtype=np.float32).astype(np.float16)
    return k, v
