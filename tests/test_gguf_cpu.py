"""The GGUF reader of the C ABI without a GPU: round trip of generated files, and hostile input.

The reader treats files as untrusted ("alpaca.swift" Highlights: every length bounded by the bytes present,
overflow-checked arithmetic, mutation-fuzzed files without a crash).  Here: every tensor of a written file reads
back byte-identical with its type and dimensions; the configuration matches the shape the file was written from;
truncations at every offset, a fixed list of malformed files and a few thousand random mutations each give
ER_EINVAL or a consistent parse, and never crash (the fuzz runs in a child process so that a crash fails the test
instead of ending the session).
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
import struct
import subprocess
import sys

import numpy as np
import pytest

import synth
import synth.gguf as sg
from helpers import TINY

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def er():
    from block_quantized_token_gb300 import build
    build.build()
    from block_quantized_token_gb300 import er as mod
    return mod


SHAPES = {"q8_untied": TINY, "q4_tied": dataclasses.replace(TINY, w_type="q4_0", tied=True, rope_base=500000.0)}


def _write(tmp_path, shape, name="m.gguf", **kw):
    tensors = synth.model_weights(shape)
    path = str(tmp_path / name)
    sg.write_gguf(path, shape, tensors, **kw)
    return path, tensors


@pytest.mark.parametrize("key", list(SHAPES))
def test_round_trip(er, tmp_path, key):
    shape = SHAPES[key]
    path, tensors = _write(tmp_path, shape)
    g = er.er_gguf_open(path)
    try:
        assert er.er_gguf_tensor_count(g) == len(tensors)
        for n, arr in tensors.items():
            i = er.er_gguf_find(g, n)
            name, typ, dims, addr, nbytes = er.er_gguf_tensor_info(g, i)
            kind, shp = synth.gen.tensor_kind(shape, n)
            assert name == n and typ == sg.GGML_TYPE[kind] and dims == list(reversed(shp))
            raw = np.ascontiguousarray(arr).tobytes()
            assert nbytes == len(raw) and addr % 32 == 0
            assert ctypes.string_at(addr, nbytes) == raw, n
        cfg = er.er_gguf_config(g, 3)
        want = dict(dim=shape.dim, n_layers=shape.n_layers, n_heads=shape.n_heads, n_kv_heads=shape.n_kv_heads,
                    head_dim=shape.head_dim, ffn_dim=shape.ffn_dim, vocab=shape.vocab,
                    w_type=er.DTYPES[shape.w_type], tied=int(shape.tied), max_batch=3)
        for k, v in want.items():
            assert getattr(cfg, k) == v, k
        # stored as float32, as GGUF files keep them
        assert cfg.rope_base == float(np.float32(shape.rope_base))
        assert cfg.rms_eps == float(np.float32(shape.rms_eps))
    finally:
        er.er_gguf_close(g)


def test_version_2_and_defaults(er, tmp_path):
    """A v2 file without head_count_kv / key_length / rope / eps keys: the documented defaults apply."""
    shape = dataclasses.replace(TINY, n_kv_heads=TINY.n_heads, rope_base=10000.0, rms_eps=1e-5)
    tensors = synth.model_weights(shape)
    drop = {"llama.attention.head_count_kv", "llama.attention.key_length", "llama.rope.freq_base",
            "llama.attention.layer_norm_rms_epsilon"}
    orig = sg.metadata
    try:
        sg.metadata = lambda s, c=4096: [m for m in orig(s, c) if m[0] not in drop]
        data = sg.gguf_bytes(shape, tensors, version=2)
    finally:
        sg.metadata = orig
    p = tmp_path / "v2.gguf"
    p.write_bytes(data)
    g = er.er_gguf_open(str(p))
    try:
        cfg = er.er_gguf_config(g, 1)
        assert (cfg.n_kv_heads, cfg.head_dim, cfg.rope_base) == (shape.n_heads, shape.dim // shape.n_heads, 10000.0)
        assert cfg.rms_eps == 1e-5
    finally:
        er.er_gguf_close(g)


def _expect_einval(er, path, what=None):
    with pytest.raises(er.ErError) as e:
        g = er.er_gguf_open(path)
        try:
            er.er_gguf_config(g, 1)
        finally:
            er.er_gguf_close(g)
    assert e.value.status == er.ER_EINVAL
    if what:
        assert what in er.er_last_error(), er.er_last_error()


def _header_end(data: bytes) -> int:
    """Offset of the data section of a file written by synth.gguf."""
    pos = 24
    nt, nm = struct.unpack_from("<QQ", data, 8)

    def s(p):
        n = struct.unpack_from("<Q", data, p)[0]
        return p + 8 + n
    for _ in range(nm):
        pos = s(pos)
        t = struct.unpack_from("<I", data, pos)[0]
        pos += 4
        if t == 8:
            pos = s(pos)
        elif t == 9:
            et, cnt = struct.unpack_from("<IQ", data, pos)
            pos += 12
            for _ in range(cnt):
                pos = s(pos)
        else:
            pos += {4: 4, 5: 4, 6: 4, 10: 8, 12: 8}[t]
    for _ in range(nt):
        pos = s(pos)
        nd = struct.unpack_from("<I", data, pos)[0]
        pos += 4 + 8 * nd + 12
    return pos + (-pos) % 32


def test_truncations(er, tmp_path):
    path, _ = _write(tmp_path, TINY)
    data = open(path, "rb").read()
    end = _header_end(data)
    p = tmp_path / "t.gguf"
    cuts = list(range(0, end + 64)) + [len(data) - 1, len(data) - 17]
    for n in cuts:
        p.write_bytes(data[:n])
        _expect_einval(er, str(p))


def _patched(data: bytes, off: int, fmt: str, value) -> bytes:
    b = bytearray(data)
    struct.pack_into(fmt, b, off, value)
    return bytes(b)


def test_malformed_files(er, tmp_path):
    path, tensors = _write(tmp_path, TINY)
    data = open(path, "rb").read()
    # offsets of the first tensor entry's fields
    end_meta = _header_end(data)  # not used for offsets below; entries are located by name
    first = b"blk.0.attn_norm.weight"
    t0 = data.index(struct.pack("<Q", len(first)) + first)
    nd_off = t0 + 8 + len(first)
    dim0_off = nd_off + 4
    type_off = dim0_off + 8
    offs_off = type_off + 4
    q = b"blk.0.attn_q.weight"
    tq = data.index(struct.pack("<Q", len(q)) + q)
    q_type_off = tq + 8 + len(q) + 4 + 16
    key = b"general.alignment"
    al_off = data.index(struct.pack("<Q", len(key)) + key) + 8 + len(key) + 4
    cases = {
        "magic": (_patched(data, 0, "<I", 0x46554748), "magic"),
        "version": (_patched(data, 4, "<I", 1), "version"),
        "tensor count": (_patched(data, 8, "<Q", 1 << 60), "tensor count"),
        "metadata count": (_patched(data, 16, "<Q", (1 << 64) - 1), "metadata count"),
        "key length": (_patched(data, 24, "<Q", 1 << 62), "metadata"),
        "n_dims": (_patched(data, nd_off, "<I", 5), "dimensions"),
        "zero dim": (_patched(data, dim0_off, "<Q", 0), "dimensions"),
        "huge dim": (_patched(data, dim0_off, "<Q", 1 << 63), "dimensions"),
        "unknown type": (_patched(data, type_off, "<I", 77), "unknown type"),
        "misaligned": (_patched(data, offs_off, "<Q", 8), "aligned"),
        "offset past end": (_patched(data, offs_off, "<Q", len(data) * 4 // 32 * 32), "past the end"),
        "alignment": (_patched(data, al_off, "<I", 48), "alignment"),
        "weight type": (_patched(data, q_type_off, "<I", 2), "type"),
    }
    p = tmp_path / "bad.gguf"
    for name, (blob, what) in cases.items():
        p.write_bytes(blob)
        _expect_einval(er, str(p), what)
    # a tensor present twice, a required key missing, a tensor missing
    dup = sg.gguf_bytes(TINY, tensors).replace(b"blk.0.attn_v.weight", b"blk.0.attn_k.weight")
    p.write_bytes(dup)
    _expect_einval(er, str(p), "duplicate")
    orig = sg.metadata
    try:
        sg.metadata = lambda s, c=4096: [m for m in orig(s, c) if m[0] != "llama.block_count"]
        p.write_bytes(sg.gguf_bytes(TINY, tensors))
    finally:
        sg.metadata = orig
    _expect_einval(er, str(p), "llama")
    p.write_bytes(sg.gguf_bytes(TINY, {k: v for k, v in tensors.items() if k != "blk.1.ffn_down.weight"}))
    _expect_einval(er, str(p), "missing")
    # a file that is not there
    _expect_einval(er, str(tmp_path / "absent.gguf"), "cannot open")


FUZZ = r"""
import os, random, sys
sys.path.insert(0, ROOT)
from block_quantized_token_gb300 import er
data = open(PATH, "rb").read()
end = HEADER_END
rng = random.Random(1234)
out = PATH + ".m"
counts = {"open_fail": 0, "config_fail": 0, "ok": 0}
for it in range(N):
    b = bytearray(data[:end + 4096])
    for _ in range(rng.randint(1, 8)):
        pos = rng.randrange(end) if rng.random() < 0.9 else rng.randrange(len(b))
        b[pos] = rng.randrange(256)
    with open(out, "wb") as f:
        f.write(b)
    try:
        g = er.er_gguf_open(out)
    except er.ErError as e:
        assert e.status == er.ER_EINVAL, e
        counts["open_fail"] += 1
        continue
    try:
        for i in range(er.er_gguf_tensor_count(g)):
            er.er_gguf_tensor_info(g, i)
        er.er_gguf_config(g, 1)
        counts["ok"] += 1
    except er.ErError as e:
        assert e.status == er.ER_EINVAL, e
        counts["config_fail"] += 1
    finally:
        er.er_gguf_close(g)
print(counts)
"""


def test_mutation_fuzz(er, tmp_path):
    """Random byte mutations of the header and tensor table (plus a few in the data) of a truncated file: every
    one is rejected or parsed consistently; the child process must exit cleanly."""
    path, _ = _write(tmp_path, TINY)
    data = open(path, "rb").read()
    end = _header_end(data)
    code = FUZZ.replace("ROOT", repr(ROOT)).replace("PATH", repr(path)).replace("HEADER_END", str(end)) \
        .replace("N)", "3000)")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, f"fuzz child failed (rc {r.returncode}):\n{r.stdout}\n{r.stderr[-2000:]}"
    assert "open_fail" in r.stdout
