"""Writes a workload's seeded tensors as a GGUF v3 file (the container the pages load models from).

The pages load models from GGUF files ("EdgeRunner Core Architecture" section
2.2; "alpaca.swift" Capabilities: GGUF v2/v3, F16/Q8_0/Q4_0 used in place),
name tensors "blk.N.attn_q.weight" and so on (section 1.2) and read the shape
from metadata keys such as llama.embedding_length, llama.block_count and
llama.attention.head_count (section 1.1).  The byte layout written here is
the published GGUF layout, little-endian throughout:

  header    "GGUF", uint32 version (3), uint64 tensor count, uint64 metadata count
  metadata  per entry: string key, uint32 value type, value
  tensors   per tensor: string name, uint32 n_dims, uint64 dims[n_dims]
            (dims[0] is the innermost: the columns of a matrix), uint32 type,
            uint64 offset of its data from the start of the data section
  padding   to general.alignment (32)
  data      the tensors, each at an offset that is a multiple of the alignment

A string is a uint64 byte length followed by the bytes (no terminator).
Metadata value types: 0 u8, 1 i8, 2 u16, 3 i16, 4 u32, 5 i32, 6 f32, 7 bool,
8 string, 9 array (uint32 element type, uint64 count, elements), 10 u64,
11 i64, 12 f64.  Tensor types are the codes of section 1.3 (f32 = 0,
f16 = 1, q4_0 = 2, q8_0 = 8).

This module only packs the generator's bytes; it holds none of the decode
step's arithmetic.
"""

from __future__ import annotations

import struct
from typing import Mapping

import numpy as np

from .gen import ModelShape, tensor_kind, tensor_names

ALIGN = 32
GGML_TYPE = {"f32": 0, "f16": 1, "q4_0": 2, "q8_0": 8}
T_U32, T_I32, T_F32, T_STRING, T_ARRAY, T_U64, T_F64 = 4, 5, 6, 8, 9, 10, 12


def _str(s: str) -> bytes:
    b = s.encode()
    return struct.pack("<Q", len(b)) + b


def _kv(key: str, vtype: int, value) -> bytes:
    out = _str(key) + struct.pack("<I", vtype)
    if vtype == T_U32:
        return out + struct.pack("<I", value)
    if vtype == T_I32:
        return out + struct.pack("<i", value)
    if vtype == T_F32:
        return out + struct.pack("<f", value)
    if vtype == T_U64:
        return out + struct.pack("<Q", value)
    if vtype == T_F64:
        return out + struct.pack("<d", value)
    if vtype == T_STRING:
        return out + _str(value)
    if vtype == T_ARRAY:
        etype, items = value
        body = struct.pack("<IQ", etype, len(items))
        for it in items:
            body += _str(it) if etype == T_STRING else struct.pack("<i", it)
        return out + body
    raise ValueError(vtype)


def metadata(shape: ModelShape, context: int = 4096) -> list[tuple[str, int, object]]:
    """The llama.* keys a loader reads the shape from (rope base and epsilon as float32, as GGUF files store them)."""
    s = shape
    return [
        ("general.architecture", T_STRING, "llama"),
        ("general.name", T_STRING, "synthetic"),
        ("general.alignment", T_U32, ALIGN),
        ("llama.context_length", T_U32, context),
        ("llama.embedding_length", T_U32, s.dim),
        ("llama.block_count", T_U32, s.n_layers),
        ("llama.feed_forward_length", T_U32, s.ffn_dim),
        ("llama.attention.head_count", T_U32, s.n_heads),
        ("llama.attention.head_count_kv", T_U32, s.n_kv_heads),
        ("llama.attention.key_length", T_U32, s.head_dim),
        ("llama.rope.dimension_count", T_U32, s.head_dim),
        ("llama.rope.freq_base", T_F32, float(s.rope_base)),
        ("llama.attention.layer_norm_rms_epsilon", T_F32, float(s.rms_eps)),
        ("llama.vocab_size", T_U32, s.vocab),
        ("tokenizer.ggml.tokens", T_ARRAY, (T_STRING, ["<unk>", "<s>", "</s>"])),
    ]


def gguf_bytes(shape: ModelShape, tensors: Mapping[str, np.ndarray], context: int = 4096,
               extra_metadata: list | None = None, version: int = 3) -> bytes:
    """The whole GGUF file of a model's tensors (every tensor of `tensors`, in the generator's draw order)."""
    names = [n for n in tensor_names(shape) if n in tensors]
    meta = metadata(shape, context) + list(extra_metadata or [])
    head = b"GGUF" + struct.pack("<IQQ", version, len(names), len(meta))
    head += b"".join(_kv(k, t, v) for k, t, v in meta)
    infos, blobs, off = [], [], 0
    for n in names:
        kind, shp = tensor_kind(shape, n)
        data = np.ascontiguousarray(tensors[n]).tobytes()
        dims = list(reversed(shp))  # innermost first
        infos.append(_str(n) + struct.pack("<I", len(dims)) + struct.pack(f"<{len(dims)}Q", *dims) +
                     struct.pack("<IQ", GGML_TYPE[kind], off))
        pad = (-len(data)) % ALIGN
        blobs.append(data + b"\0" * pad)
        off += len(data) + pad
    body = head + b"".join(infos)
    body += b"\0" * ((-len(body)) % ALIGN)
    return body + b"".join(blobs)


def write_gguf(path: str, shape: ModelShape, tensors: Mapping[str, np.ndarray], **kw) -> int:
    data = gguf_bytes(shape, tensors, **kw)
    with open(path, "wb") as f:
        f.write(data)
    return len(data)
