"""Pins of the float64 oracle to things other than itself (CPU only).

Each `check_*` function states what it pins and against what: printed values of
the pages (tests/golden/), hand-built inputs whose results follow from the
format or formula by hand, closed forms, invariants, and torch/scipy float64
library routines.  `test_planted_mistakes` plants plausible mistakes in the
oracle and shows that a pin catches each one.
"""

from __future__ import annotations

import math
import os
import struct

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import oracle.blocks
import oracle.ops
import synth
from helpers import TINY, oracle_config, oracle_model

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_formats():
    rows, extra = {}, {}
    with open(os.path.join(GOLDEN, "block_formats.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            if len(parts) == 4:
                rows[parts[0]] = tuple(int(p) for p in parts[1:])
            else:
                extra[parts[0]] = float(parts[1])
    return rows, extra


# ------------------------------------------------------------------------------------------
# block formats
# ------------------------------------------------------------------------------------------
# fp16 bit patterns with their exact IEEE-754 binary16 values (sign, exponent 5, mantissa 10)
FP16 = [(0x3C00, 1.0), (0xB800, -0.5), (0x7BFF, 65504.0), (0x0400, 2.0 ** -14),
        (0x0001, 2.0 ** -24), (0x8000, -0.0), (0x3555, 0.333251953125), (0xC200, -3.0)]


def check_block_sizes():
    fmts, extra = _golden_formats()
    assert oracle.blocks.BLOCK_BYTES["q8_0"] == fmts["q8_0"][2]
    assert oracle.blocks.BLOCK_BYTES["q4_0"] == fmts["q4_0"][2]
    assert synth.BLOCK_BYTES == {"q8_0": fmts["q8_0"][2], "q4_0": fmts["q4_0"][2]}
    # bytes of float32 over bytes of Q8_0 for 32 elements: 128 / 34 = 3.76..., printed as ~3.8
    ratio = (4 * fmts["q8_0"][1]) / fmts["q8_0"][2]
    assert round(ratio, 1) == extra["bandwidth_reduction_q8_0_vs_f32"]


def _q8_block(bits: int, qs) -> bytes:
    return struct.pack("<H", bits) + struct.pack("<32b", *qs)


def check_q8_0_hand_blocks():
    raw, want = b"", []
    for i, (bits, dval) in enumerate(FP16):
        # block i sweeps 32 int8 values; the 8 blocks together cover all 256
        qs = [-128 + 32 * i + j for j in range(32)]
        raw += _q8_block(bits, qs)
        want += [dval * q for q in qs]
    got = oracle.blocks.dequant_q8_0(np.frombuffer(raw, np.uint8), 1, 32 * len(FP16))
    np.testing.assert_array_equal(got.reshape(-1), np.array(want))
    # signed zero scale keeps exact zeros
    assert got.shape == (1, 32 * len(FP16))


def check_q4_0_hand_blocks():
    raw, want = b"", []
    for i, (bits, dval) in enumerate(FP16):
        lo = [(j + i) % 16 for j in range(16)]          # element j: low nibble of byte j
        hi = [(15 - j + 3 * i) % 16 for j in range(16)]  # element j + 16: high nibble of byte j
        raw += struct.pack("<H", bits) + bytes(l | (h << 4) for l, h in zip(lo, hi))
        want += [dval * (n - 8) for n in lo] + [dval * (n - 8) for n in hi]
    got = oracle.blocks.dequant_q4_0(np.frombuffer(raw, np.uint8), 1, 32 * len(FP16))
    np.testing.assert_array_equal(got.reshape(-1), np.array(want))


def check_quantize_roundtrip():
    rng = np.random.default_rng(5)
    # values d * integer with d a power of two: the quantiser must hit them exactly
    q8 = rng.integers(-127, 128, size=(3, 64)).astype(np.float64)
    q8[:, 0], q8[:, 32] = 127, -127                     # one max-|q| element per block
    x8 = q8 * 2.0 ** -9
    b8 = synth.quantize_q8_0(x8.astype(np.float32))
    np.testing.assert_array_equal(oracle.blocks.dequant_q8_0(b8, 3, 64), x8)
    blk = b8.reshape(3, 2, 34)
    # the max-|x| element of each block maps to +-127
    assert (blk[:, 0, 2].view(np.int8) == 127).all() and (blk[:, 1, 2].view(np.int8) == -127).all()
    q4 = rng.integers(-7, 8, size=(3, 64)).astype(np.float64)
    q4[:, 5], q4[:, 40] = -8, -8                         # the max-|x| element of each block is -8 d
    x4 = q4 * 2.0 ** -6
    b4 = synth.quantize_q4_0(x4.astype(np.float32))
    np.testing.assert_array_equal(oracle.blocks.dequant_q4_0(b4, 3, 64), x4)
    # the max-|x| element maps to stored nibble 0
    nib = b4.reshape(3, 2, 18)[:, 0, 2 + 5] & 0xF
    assert (nib == 0).all()


def check_matvec():
    rng = np.random.default_rng(7)
    w = rng.standard_normal((5, 96))
    x = rng.standard_normal(96)
    np.testing.assert_allclose(oracle.ops.matvec(w, x), np.dot(w, x), rtol=1e-12)
    X = rng.standard_normal((3, 96))
    np.testing.assert_allclose(oracle.ops.matvec(w, X), np.array([np.dot(w, r) for r in X]), rtol=1e-12)


# ------------------------------------------------------------------------------------------
# RMSNorm, RoPE, softmax, attention, SiLU
# ------------------------------------------------------------------------------------------
def check_rmsnorm():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((4, 80)) * 3.0
    g = 1.0 + 0.1 * rng.standard_normal(80)
    eps = 1e-5
    want = F.rms_norm(torch.from_numpy(x), (80,), weight=torch.from_numpy(g), eps=eps).numpy()
    np.testing.assert_allclose(oracle.ops.rmsnorm(x, g, eps), want, rtol=1e-13, atol=0)
    # g = 1: mean(y^2) = mean(x^2) / (mean(x^2) + eps)
    y = oracle.ops.rmsnorm(x, np.ones(80), eps)
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), ms / (ms + eps), rtol=1e-13)


def check_rope():
    rng = np.random.default_rng(13)
    u = rng.standard_normal((3, 16))
    # position 0 is the identity
    np.testing.assert_array_equal(oracle.ops.rope(u, 0, 10000.0), u)
    # head dim 2: the single pair turns by exactly `pos` radians (base^0 = 1)
    v = np.array([0.3, -1.7])
    p = 5
    want = np.array([0.3 * math.cos(p) + 1.7 * math.sin(p), -1.7 * math.cos(p) + 0.3 * math.sin(p)])
    np.testing.assert_allclose(oracle.ops.rope(v, p, 10000.0), want, rtol=1e-14)
    # head dim 4, base 100, pos 10: pair 1 turns by 10 * 100^(-2/4) = 1 radian
    w = np.array([0.0, 0.0, 1.0, 0.0])
    np.testing.assert_allclose(oracle.ops.rope(w, 10, 100.0), [0, 0, math.cos(1.0), math.sin(1.0)], atol=1e-15)
    # pairs as complex numbers: u'_i = u_i * exp(i * pos * base^(-2i/hd))
    z = u[:, 0::2] + 1j * u[:, 1::2]
    ang = 37 * 10000.0 ** (-np.arange(8) * 2 / 16)
    zz = z * np.exp(1j * ang)
    r = oracle.ops.rope(u, 37, 10000.0)
    np.testing.assert_allclose(r[:, 0::2] + 1j * r[:, 1::2], zz, rtol=1e-12, atol=1e-14)
    # rotations compose and keep each pair's norm
    np.testing.assert_allclose(oracle.ops.rope(oracle.ops.rope(u, 3, 500.0), 4, 500.0),
                               oracle.ops.rope(u, 7, 500.0), rtol=1e-12, atol=1e-14)
    # <R(p) q, R(p') k> depends only on p - p'
    q, k = rng.standard_normal(16), rng.standard_normal(16)
    d0 = np.dot(oracle.ops.rope(q, 9, 10000.0), oracle.ops.rope(k, 4, 10000.0))
    d1 = np.dot(oracle.ops.rope(q, 105, 10000.0), oracle.ops.rope(k, 100, 10000.0))
    assert abs(d0 - d1) < 1e-12


def check_softmax():
    import scipy.special
    rng = np.random.default_rng(17)
    s = rng.standard_normal((5, 40)) * 10
    a = oracle.ops.softmax(s)
    np.testing.assert_allclose(a.sum(-1), 1.0, rtol=0, atol=1e-15)
    np.testing.assert_allclose(a, scipy.special.softmax(s, axis=-1), rtol=1e-13)
    np.testing.assert_allclose(oracle.ops.softmax(s + 1000.0), a, rtol=1e-12)


def _sdpa(q, k, v):
    # q [H, hd], k/v [T, KV, hd] -> torch [1, H, 1, hd] etc., GQA by contiguous groups
    qt = torch.from_numpy(np.asarray(q, np.float64))[None, :, None, :]
    kt = torch.from_numpy(np.asarray(k, np.float64)).permute(1, 0, 2)[None]
    vt = torch.from_numpy(np.asarray(v, np.float64)).permute(1, 0, 2)[None]
    return F.scaled_dot_product_attention(qt, kt, vt, enable_gqa=True)[0, :, 0, :].numpy()


def check_attention():
    rng = np.random.default_rng(19)
    # one cached position: every head returns its group's V row
    q = rng.standard_normal((6, 8))
    k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 8))
    o = oracle.ops.attention_gqa(q, k, v)
    np.testing.assert_allclose(o, np.repeat(v[0], 3, axis=0), rtol=1e-15)
    # hd = 4, T = 3, one head: the sum written out by hand
    q1 = np.array([[0.5, -1.0, 2.0, 0.25]])
    k1 = np.array([[[1.0, 0.0, 0.0, 0.0]], [[0.0, 1.0, 0.0, 0.0]], [[0.0, 0.0, 1.0, 1.0]]])
    v1 = np.array([[[1.0, 2.0, 3.0, 4.0]], [[-1.0, 0.0, 1.0, 0.0]], [[0.0, 0.0, 0.0, 8.0]]])
    s = np.array([0.5, -1.0, 2.25]) / 2.0
    e = np.exp(s)
    want = (e[0] * v1[0, 0] + e[1] * v1[1, 0] + e[2] * v1[2, 0]) / e.sum()
    np.testing.assert_allclose(oracle.ops.attention_gqa(q1, k1, v1)[0], want, rtol=1e-14)
    # GQA against torch's SDPA (enable_gqa) and against MHA with KV heads repeated
    for H, KV in ((9, 3), (8, 2), (4, 4), (32, 8)):
        q = rng.standard_normal((H, 16))
        k = rng.standard_normal((37, KV, 16))
        v = rng.standard_normal((37, KV, 16))
        o = oracle.ops.attention_gqa(q, k, v)
        np.testing.assert_allclose(o, _sdpa(q, k, v), rtol=1e-12, atol=1e-14)
        rep = H // KV
        np.testing.assert_allclose(o, oracle.ops.attention_gqa(q, np.repeat(k, rep, 1), np.repeat(v, rep, 1)),
                                   rtol=1e-14)


def check_silu():
    z = np.linspace(-30, 30, 301)
    np.testing.assert_allclose(oracle.ops.silu(z), F.silu(torch.from_numpy(z)).numpy(), rtol=1e-14, atol=1e-300)
    assert oracle.ops.silu(np.array([0.0]))[0] == 0.0
    g, u = np.array([1.0, -2.0]), np.array([3.0, 0.5])
    np.testing.assert_allclose(oracle.ops.swiglu(g, u), F.silu(torch.from_numpy(g)).numpy() * u, rtol=1e-15)


# ------------------------------------------------------------------------------------------
# whole step
# ------------------------------------------------------------------------------------------
def _pure_dequant(raw: np.ndarray, kind: str, rows: int, cols: int) -> np.ndarray:
    """Byte-by-byte dequantisation with struct (independent of the oracle's numpy views)."""
    data = bytes(np.asarray(raw, np.uint8).reshape(-1))
    bpb = {"q8_0": 34, "q4_0": 18}[kind]
    out = np.empty(rows * cols)
    for b in range(rows * cols // 32):
        blk = data[b * bpb:(b + 1) * bpb]
        d = struct.unpack("<e", blk[:2])[0]
        if kind == "q8_0":
            qs = struct.unpack("<32b", blk[2:])
        else:
            qs = [(x & 15) - 8 for x in blk[2:]] + [(x >> 4) - 8 for x in blk[2:]]
        out[b * 32:(b + 1) * 32] = [d * q for q in qs]
    return out.reshape(rows, cols)


def _torch_step(shape, weights, kcache, vcache, token, pos):
    """One decode step built from torch float64 library routines (rms_norm, SDPA, silu)."""
    s = shape
    T = lambda a: torch.from_numpy(np.asarray(a, np.float64))  # noqa: E731

    def mat(name, rows, cols):
        return T(_pure_dequant(weights[name], s.w_type, rows, cols))

    def rot(u, p):  # pairs as complex numbers times e^{i p base^(-2i/hd)}
        hd = u.shape[-1]
        z = torch.view_as_complex(u.reshape(*u.shape[:-1], hd // 2, 2).contiguous())
        ang = p * torch.pow(torch.tensor(s.rope_base, dtype=torch.float64),
                            -torch.arange(0, hd, 2, dtype=torch.float64) / hd)
        return torch.view_as_real(z * torch.polar(torch.ones_like(ang), ang)).reshape(u.shape)

    if s.tied:
        x = mat("token_embd.weight", s.vocab, s.dim)[token]
    else:
        x = T(np.asarray(weights["token_embd.weight"], np.float16)[token].astype(np.float64))
    for l in range(s.n_layers):
        p = f"blk.{l}."
        h = F.rms_norm(x, (s.dim,), weight=T(weights[p + "attn_norm.weight"]), eps=s.rms_eps)
        q = mat(p + "attn_q.weight", s.qd, s.dim) @ h
        k = mat(p + "attn_k.weight", s.kvd, s.dim) @ h
        v = mat(p + "attn_v.weight", s.kvd, s.dim) @ h
        q = rot(q.reshape(s.n_heads, s.head_dim), pos)
        k = rot(k.reshape(s.n_kv_heads, s.head_dim), pos)
        kcache[l][pos] = k.numpy().astype(np.float16)
        vcache[l][pos] = v.reshape(s.n_kv_heads, s.head_dim).numpy().astype(np.float16)
        K = T(kcache[l][:pos + 1].astype(np.float64)).permute(1, 0, 2)[None]
        V = T(vcache[l][:pos + 1].astype(np.float64)).permute(1, 0, 2)[None]
        o = F.scaled_dot_product_attention(q[None, :, None, :], K, V, enable_gqa=True)[0, :, 0, :].reshape(-1)
        x = x + mat(p + "attn_output.weight", s.dim, s.qd) @ o
        h2 = F.rms_norm(x, (s.dim,), weight=T(weights[p + "ffn_norm.weight"]), eps=s.rms_eps)
        a = F.silu(mat(p + "ffn_gate.weight", s.ffn_dim, s.dim) @ h2) * (mat(p + "ffn_up.weight", s.ffn_dim, s.dim) @ h2)
        x = x + mat(p + "ffn_down.weight", s.dim, s.ffn_dim) @ a
    hf = F.rms_norm(x, (s.dim,), weight=T(weights["output_norm.weight"]), eps=s.rms_eps)
    head = "token_embd.weight" if s.tied else "output.weight"
    return (mat(head, s.vocab, s.dim) @ hf).numpy()


TINY_SHAPES = [TINY, synth.ModelShape(**{**TINY.__dict__, "w_type": "q4_0", "tied": True}),
               synth.ModelShape(**{**TINY.__dict__, "n_kv_heads": 4, "w_type": "q4_0"}),
               synth.ModelShape(**{**TINY.__dict__, "n_kv_heads": 1, "tied": True, "rope_base": 500000.0})]


def check_step_vs_torch(shape=TINY):
    weights = synth.gen.model_weights(shape)
    model = oracle_model(shape, weights)
    wl = synth.Workload("t", shape, batch=1, steps=3, prefill=5)
    cache = oracle.OracleCache(oracle_config(shape), 1, wl.capacity)
    kc = [np.zeros((wl.capacity, shape.n_kv_heads, shape.head_dim), np.float16) for _ in range(shape.n_layers)]
    vc = [np.zeros_like(a) for a in kc]
    for l in range(shape.n_layers):
        k, v = synth.kv_prefill(wl, 0, l)
        cache.fill(0, l, k, v)
        kc[l][:5] = k.reshape(5, shape.n_kv_heads, shape.head_dim)
        vc[l][:5] = v.reshape(5, shape.n_kv_heads, shape.head_dim)
    tok, pos = 7, 5
    for _ in range(3):
        logits, am, nf = oracle.decode_step(model, cache, [tok], [pos])
        want = _torch_step(shape, weights, kc, vc, tok, pos)
        np.testing.assert_allclose(logits[0], want, rtol=1e-10, atol=1e-12)
        assert not nf[0]
        tok, pos = int(am[0]), pos + 1


def check_cached_equals_uncached(shape=TINY):
    model = oracle_model(shape)
    toks = [3, 17, 99, 5, 64, 1]
    cache = oracle.OracleCache(oracle_config(shape), 1, len(toks))
    for n, t in enumerate(toks):
        logits, _, _ = oracle.decode_step(model, cache, [t], [n])
        np.testing.assert_allclose(logits[0], oracle.uncached_logits(model, toks[:n + 1]), rtol=1e-11, atol=1e-13)


def check_batch_equals_single(shape=TINY):
    """Sequences of a batch are independent: a batched step equals per-sequence steps."""
    model = oracle_model(shape)
    wl = synth.Workload("t", shape, batch=3, steps=1, prefill=4)
    from helpers import oracle_cache
    cb = oracle_cache(wl)
    lb, ab, _ = oracle.decode_step(model, cb, [7, 8, 9], [4, 2, 0])
    for i, (t, p) in enumerate(((7, 4), (8, 2), (9, 0))):
        cs = oracle_cache(wl, seqs=[i])
        ls, _, _ = oracle.decode_step(model, cs, [7, 8, 9], [4, 2, 0], seqs=[i])
        np.testing.assert_allclose(lb[i], ls[0], rtol=1e-13, atol=1e-15)


def check_greedy(shape=TINY):
    """A greedy chain feeds each sequence's own argmax back at the next position.

    Pinned against the uncached recompute (itself pinned by the cached-vs-uncached
    and torch checks): from an empty cache, the logits of step s of sequence b
    equal the from-scratch logits of the tokens fed to b so far at positions
    0..s, and the token fed at step s + 1 is their argmax.  Three sequences with
    different first tokens, of which only two (out of order) are computed.
    """
    model = oracle_model(shape)
    steps, tokens0, seqs = 4, [5, 9, 11], [2, 0]
    cache = oracle.OracleCache(oracle_config(shape), 3, steps)
    fed, logits = oracle.decode.greedy(model, cache, tokens0, [0, 0, 0], steps, seqs=seqs)
    assert fed.shape == (steps, 2) and logits.shape == (steps, 2, shape.vocab)
    for i, b in enumerate(seqs):
        seq = [tokens0[b]]
        for s in range(steps):
            assert fed[s, i] == seq[s], (b, s, fed[:, i], seq)
            want = oracle.uncached_logits(model, seq)
            np.testing.assert_allclose(logits[s, i], want, rtol=1e-11, atol=1e-13)
            seq.append(int(np.argmax(want)))


def check_kv_q8_0():
    """The Q8_0 cache quantizer: hand-derived blocks and the bound every block satisfies.

    - 0.5 * (integers up to 127): the scale 63.5 / 127 = 0.5 is exact, the round trip is exact.
    - a block of largest |x| = 127 (scale 1): 2.5 -> 3 and -2.5 -> -3 (ties away from zero), 0.49 -> 0, and
      the largest float32 below one half -> 0.
    - a block of largest |x| = 100: 100 / 127 = 0.787401... is stored as fp16 1613 * 2^-11 = 0.78759765625;
      50 / 0.78759765625 = 63.484... -> 63 (dividing by the unrounded scale would give 63.5 -> 64), and the
      largest element 100 / 0.78759765625 = 126.97 -> 127.
    - an all-zero block stores d = 0, q = 0.
    - random blocks: |x - d q| <= d / 2 + 2^-20 |x| element-wise, |q| <= 127, and the largest element maps
      to +-127.
    """
    qz = oracle.blocks.quantize_kv_q8_0
    x = np.zeros(64, np.float32)
    x[:32] = 0.5 * (np.arange(32) * 8 - 127).clip(-127, 127)
    d, q = qz(x)
    assert d[0] == np.float16(0.5) and d[1] == 0 and not q[32:].any()
    np.testing.assert_array_equal(oracle.blocks.dequant_kv_q8_0(d, q), x.astype(np.float64))
    blk = np.zeros(32, np.float32)
    blk[:5] = [127.0, 2.5, -2.5, 0.49, np.nextafter(np.float32(0.5), np.float32(0))]
    d, q = qz(blk)
    assert d[0] == np.float16(1.0) and list(q[:5]) == [127, 3, -3, 0, 0]
    blk = np.zeros(32, np.float32)
    blk[:2] = [100.0, 50.0]
    d, q = qz(blk)
    assert float(d[0]) == 1613 * 2.0 ** -11 and list(q[:2]) == [127, 63]
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((50, 128)) * rng.uniform(0.01, 100, (50, 1))).astype(np.float32)
    d, q = qz(x)
    assert np.abs(q.astype(int)).max() <= 127
    dd = np.repeat(d.astype(np.float64), 32, axis=-1)
    err = np.abs(x.astype(np.float64) - oracle.blocks.dequant_kv_q8_0(d, q))
    assert (err <= dd / 2 + 2.0 ** -20 * np.abs(x)).all()
    xb, qb = x.reshape(50, 4, 32), q.reshape(50, 4, 32)
    top = np.argmax(np.abs(xb), axis=-1)
    assert (np.abs(np.take_along_axis(qb, top[..., None], -1)) == 127).all()


TINY_HD32 = synth.ModelShape(**{**TINY.__dict__, "n_heads": 2, "n_kv_heads": 1, "head_dim": 32})


def check_cached_equals_uncached_q8(shape=TINY_HD32):
    """With a Q8_0 cache, incremental decoding equals the from-scratch recompute that quantises K and V the
    same way (head rows of whole 32-element blocks)."""
    model = oracle_model(shape)
    toks = [3, 17, 99, 5, 64]
    cache = oracle.OracleCache(oracle_config(shape), 1, len(toks), kv_type="q8_0")
    for n, t in enumerate(toks):
        logits, _, _ = oracle.decode_step(model, cache, [t], [n])
        np.testing.assert_allclose(logits[0], oracle.uncached_logits(model, toks[:n + 1], kv_type="q8_0"),
                                   rtol=1e-11, atol=1e-13)


def check_argmax():
    lg = np.array([[1.0, 3.0, 3.0, -np.inf], [np.nan, 0.5, 0.5, 0.1], [np.inf, 2.0, np.inf, 1.0]])
    am, nf = oracle.decode._argmax_flag(lg)
    assert list(am) == [1, 1, 0]
    assert list(nf) == [True, True, True]
    am, nf = oracle.decode._argmax_flag(np.array([[0.0, -1.0, 0.0]]))
    assert list(am) == [0] and not nf[0]


# ------------------------------------------------------------------------------------------
PINS = [check_block_sizes, check_q8_0_hand_blocks, check_q4_0_hand_blocks, check_quantize_roundtrip, check_matvec,
        check_rmsnorm, check_rope, check_softmax, check_attention, check_silu, check_argmax, check_kv_q8_0,
        check_cached_equals_uncached_q8]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


@pytest.mark.parametrize("shape", TINY_SHAPES, ids=["q8_untied", "q4_tied", "q4_mha", "q8_mqa_tied"])
def test_step_vs_torch(shape):
    check_step_vs_torch(shape)


@pytest.mark.parametrize("shape", TINY_SHAPES[:2], ids=["q8_untied", "q4_tied"])
def test_cached_equals_uncached(shape):
    check_cached_equals_uncached(shape)


def test_batch_equals_single():
    check_batch_equals_single()


def test_greedy_chain():
    check_greedy()


# ------------------------------------------------------------------------------------------
# planted mistakes: each must be caught by a pin
# ------------------------------------------------------------------------------------------
def _q4_swapped(raw, rows, cols):
    blk = oracle.blocks._blocks(raw, rows, cols, 18)
    d = oracle.blocks._scales(blk)
    b = blk[..., 2:].astype(np.int64)
    q = np.empty(b.shape[:-1] + (32,))
    q[..., 16:] = (b & 0xF) - 8
    q[..., :16] = (b >> 4) - 8
    return (d[..., None] * q).reshape(rows, cols)


def _q8_unsigned(raw, rows, cols):
    blk = oracle.blocks._blocks(raw, rows, cols, 34)
    d = oracle.blocks._scales(blk)
    return (d[..., None] * blk[..., 2:].astype(np.float64)).reshape(rows, cols)


def _rope_sign(u, pos, base):
    return oracle.ops.__dict__["_orig_rope"](u, -pos, base)


def _rope_neox(u, pos, base):
    u = np.asarray(u, np.float64)
    hd = u.shape[-1]
    perm = np.concatenate([np.arange(0, hd, 2), np.arange(1, hd, 2)])
    inv = np.argsort(perm)
    return oracle.ops.__dict__["_orig_rope"](u[..., perm], pos, base)[..., inv]


def _attn_modmap(q, k, v):
    H, KV = q.shape[0], k.shape[1]
    o = np.empty_like(np.asarray(q, np.float64))
    for h in range(H):
        s = np.asarray(k, np.float64)[:, h % KV, :] @ q[h] / np.sqrt(q.shape[1])
        o[h] = oracle.ops.softmax(s) @ np.asarray(v, np.float64)[:, h % KV, :]
    return o


def _attn_noscale(q, k, v):
    return oracle.ops.__dict__["_orig_attention_gqa"](np.asarray(q) * np.sqrt(q.shape[1]), k, v)


def _rms_eps_out(x, g, eps):
    x = np.asarray(x, np.float64)
    return x / (np.sqrt(np.mean(x * x, axis=-1, keepdims=True)) + eps) * g


def _silu_sigmoid(z):
    return 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64)))


def _matvec_T(w, x):
    w = np.asarray(w, np.float64)
    return np.asarray(x, np.float64) @ w.T[: w.shape[1], : w.shape[0]].T if w.shape[0] == w.shape[1] else (w.T @ np.asarray(x).T).T


def _greedy_variant(stuck_position: bool, wrong_slot: bool):
    """oracle.greedy with one plausible slip: the position never advances, or the argmax is written to the
    first len(seqs) sequences instead of the computed ones."""
    def run(model, cache, tokens, positions, steps, seqs=None):
        tok = np.array(tokens, dtype=np.int64)
        pos = np.array(positions, dtype=np.int64)
        seqs = list(range(len(tok))) if seqs is None else list(seqs)
        fed, out = [], []
        for _ in range(steps):
            fed.append(tok[seqs].copy())
            logits, am, _ = oracle.decode.decode_step(model, cache, tok, pos, seqs=seqs)
            out.append(logits)
            if wrong_slot:
                tok[:len(seqs)] = am
            else:
                tok[seqs] = am
            if not stuck_position:
                pos[seqs] += 1
        return np.array(fed), np.array(out)
    run.__name__ = "_greedy_stuck_position" if stuck_position else "_greedy_wrong_slot"
    return run


def _kvq_unrounded(x):
    """The cache quantizer dividing by the unrounded scale."""
    x = np.asarray(x, np.float32)
    xb = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
    s = (np.max(np.abs(xb), axis=-1) / np.float32(127)).astype(np.float32)
    r = np.where(s[..., None] > 0, xb / np.where(s > 0, s, 1)[..., None], 0).astype(np.float32)
    q = np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -127, 127).astype(np.int8)
    return s.astype(np.float16), q.reshape(x.shape)


def _kvq_half_even(x):
    """The cache quantizer rounding ties to even."""
    d, _ = oracle.blocks.__dict__["_orig_quantize_kv_q8_0"](x)
    x = np.asarray(x, np.float32)
    xb = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
    d32 = d.astype(np.float32)
    r = np.where(d32[..., None] > 0, xb / np.where(d32 > 0, d32, 1)[..., None], 0).astype(np.float32)
    return d, np.clip(np.rint(r), -127, 127).astype(np.int8).reshape(x.shape)


MISTAKES = [
    ("blocks", "dequant_q4_0", _q4_swapped, check_q4_0_hand_blocks),
    ("blocks", "dequant_q8_0", _q8_unsigned, check_q8_0_hand_blocks),
    ("ops", "rope", _rope_sign, check_rope),
    ("ops", "rope", _rope_neox, check_rope),
    ("ops", "attention_gqa", _attn_modmap, check_attention),
    ("ops", "attention_gqa", _attn_noscale, check_attention),
    ("ops", "rmsnorm", _rms_eps_out, check_rmsnorm),
    ("ops", "silu", _silu_sigmoid, check_silu),
    ("ops", "matvec", _matvec_T, check_matvec),
    ("blocks", "quantize_kv_q8_0", _kvq_unrounded, check_kv_q8_0),
    ("blocks", "quantize_kv_q8_0", _kvq_half_even, check_kv_q8_0),
    ("decode", "greedy", _greedy_variant(True, False), check_greedy),
    ("decode", "greedy", _greedy_variant(False, True), check_greedy),
]


@pytest.mark.parametrize("mod,name,bad,pin", MISTAKES, ids=[m[2].__name__ for m in MISTAKES])
def test_planted_mistakes(monkeypatch, mod, name, bad, pin):
    module = {"blocks": oracle.blocks, "ops": oracle.ops, "decode": oracle.decode}[mod]
    monkeypatch.setitem(module.__dict__, "_orig_" + name, getattr(module, name))
    monkeypatch.setattr(module, name, bad)
    with pytest.raises((AssertionError, ValueError)):
        pin()
