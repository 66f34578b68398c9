"""The packed Q8_0 K/V cache on the GPU against the oracle's (oracle.quantize_kv_q8_0, OracleCache kv_type q8_0).

* rows written through er_kv_write are quantised bit-exactly (fp16 rows: both sides quantise the same float32
  values), read back as GGUF blocks through er_kv_read_blocks;
* the new rows a step appends come from the GPU's fp32 projection, so a code may sit one step off the
  oracle's only where the exact value lies within the derived error bound of a rounding boundary
  (helpers.check_q8_blocks; layer 0, where the bound is derived);
* greedy chains with the Q8_0 cache against the oracle run with the same cache type: tokens equal, logits
  within the logits gate, over the per-phase schedule with both batch-1 and batched GEMVs.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import oracle
import synth
import helpers
from helpers import (check_q8_blocks, gpu_chain, gpu_model, gpu_state, layer0_kv_exact, oracle_cache, oracle_model,
                     rel_l2, top2_gap)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

KERNELS = 2  # er_schedule: ER_SCHEDULE_KERNELS
PERSISTENT = 1

SHAPES = {
    "q8_hd64_g2": synth.ModelShape(n_layers=2, dim=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=256, vocab=512,
                                   rope_base=10000.0, rms_eps=1e-5, w_type="q8_0", tied=False),
    "q4_hd128_g4": synth.ModelShape(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=320,
                                    vocab=1000, rope_base=500000.0, rms_eps=1e-5, w_type="q4_0", tied=False),
    "q8_hd64_g3_odd": synth.ModelShape(n_layers=3, dim=96 * 3, n_heads=9, n_kv_heads=3, head_dim=64, ffn_dim=416,
                                       vocab=777, rope_base=10000.0, rms_eps=1e-6, w_type="q8_0", tied=True),
    "q8_k2048_g4": synth.ModelShape(n_layers=2, dim=2048, n_heads=16, n_kv_heads=4, head_dim=128, ffn_dim=2560,
                                    vocab=1000, rope_base=10000.0, rms_eps=1e-5, w_type="q8_0", tied=False),
}


class Setup:
    def __init__(self, wl, max_batch=None):
        self.wl = wl
        self.weights = synth.gen.model_weights(wl.shape)
        self.om = oracle_model(wl.shape, self.weights)
        self.model = gpu_model(wl.shape, self.weights, max_batch=max_batch or wl.batch)
        self.state = gpu_state(self.model, wl, kv_type="q8_0")

    def close(self):
        self.state.close()
        self.model.close()


def _blocks_of(rows, nkv, hd):
    d, q = oracle.quantize_kv_q8_0(np.asarray(rows, np.float16).astype(np.float32).reshape(-1, nkv * hd))
    return d, q


@pytest.mark.parametrize("name", ["q8_hd64_g2", "q4_hd128_g4"])
def test_write_read_blocks_bit_exact(name):
    """er_kv_write quantises fp16 rows exactly as the oracle does: special blocks (all zero, one non-zero
    value, exact ties x / d = k + 1/2, the largest fp16 values, subnormals) and seeded rows, at a ragged
    start and count."""
    shape = SHAPES[name]
    nkv, hd = shape.n_kv_heads, shape.head_dim
    wl = synth.Workload("t", shape, batch=2, steps=79, prefill=1)  # capacity 80; row 0 prefilled
    s = Setup(wl)
    try:
        rng = np.random.default_rng(11)
        n = 37
        k = (rng.standard_normal((n, nkv * hd)) * rng.uniform(0.01, 8.0, (n, 1))).astype(np.float16)
        v = (rng.standard_normal((n, nkv * hd)) * 0.5).astype(np.float16)
        k[0] = 0                                              # d = 0: every code 0
        k[1] = 0
        k[1, 5] = -3.0                                        # one value: q = -127
        k[2, :32] = 0
        k[2, 0] = 127.0                                       # d = 1: ties of x / d at k + 1/2
        k[2, 1:8] = np.array([2.5, -2.5, 0.5, -0.5, 126.5, 1.5, -1.5], np.float16)
        k[3] = np.float16(65504.0) * np.sign(rng.standard_normal(nkv * hd))  # the largest fp16 values
        v[4] = np.float16(2.0 ** -24) * rng.integers(-5, 6, nkv * hd)        # subnormal fp16 values: d = 0
        v[5, :32] = np.float16(2.0 ** -14)                                   # d underflows fp16 too
        start = 9
        s.state.write_rows(1, 1, k, v, start=start)
        kd, kq, vd, vq = s.state.read_blocks(1, 1, start, n)
        for (dg, qg), rows in (((kd, kq), k), ((vd, vq), v)):
            dr, qr = _blocks_of(rows, nkv, hd)
            np.testing.assert_array_equal(dg.view(np.uint16), dr.reshape(n, -1).view(np.uint16))
            np.testing.assert_array_equal(qg, qr.reshape(n, -1))
        assert list(kq[2, :8]) == [127, 3, -3, 1, -1, 127, 2, -2]
        # untouched rows stay zero
        d0, q0, _, _ = s.state.read_blocks(1, 1, 1, start - 1)
        assert not d0.view(np.uint16).any() and not q0.any()
    finally:
        s.close()


def test_q8_cache_api_rules():
    """fp16-only calls refuse a Q8_0 cache and the reverse; the persistent step refuses a Q8_0 cache."""
    from block_quantized_token_gb300 import er
    shape = SHAPES["q8_hd64_g2"]
    wl = synth.Workload("t", shape, batch=1, steps=12, prefill=4)
    s = Setup(wl)
    try:
        assert er.er_kv_type(s.state.handle) == er.ER_Q8_0
        assert s.state.schedule == KERNELS
        with pytest.raises(er.ErError) as e:
            s.state.set_schedule(PERSISTENT)
        assert e.value.status == er.ER_EUNSUPPORTED
        with pytest.raises(er.ErError) as e:
            er.er_kv_layer_ptrs(s.state.handle, 0, 0)
        assert e.value.status == er.ER_EUNSUPPORTED
        with pytest.raises(er.ErError) as e:
            s.state.read_rows(0, 0, 0, 1)
        assert e.value.status == er.ER_EUNSUPPORTED
        with pytest.raises(er.ErError) as e:
            s.state.read_blocks(0, 0, 10, 7)
        assert e.value.status == er.ER_EINVAL
        with pytest.raises(er.ErError) as e:
            er.er_kv_create_typed(s.model.handle, 1, 16, er.ER_Q4_0)
        assert e.value.status == er.ER_EINVAL
        f16 = gpu_state(s.model, wl)
        try:
            assert er.er_kv_type(f16.handle) == er.ER_F16
            with pytest.raises(er.ErError) as e:
                f16.read_blocks(0, 0, 0, 1)
            assert e.value.status == er.ER_EUNSUPPORTED
        finally:
            f16.close()
        # the attention kernel quantises the step's new rows itself: no launch beyond the fp16 cache's
        assert er.er_kv_launches_per_step(s.state.handle) == 1 + shape.n_layers * 5 + 1
    finally:
        s.close()


# ------------------------------------------------------------------------------------------
# chains: the legitimate one-code differences of the new rows, and their effect on the logits
# ------------------------------------------------------------------------------------------
def _flip_tolerance(om, wl, fed, base, positions, steps):
    """Per (step, sequence): sums over the legitimate alternatives of the new layer-0 rows (steps <= this one)
    of the max-abs and L2 change each alone makes to the oracle's logits, the next tokens held fixed."""
    s = wl.shape
    B = wl.batch
    cfg = helpers.oracle_config(s)
    tol_abs = np.zeros((steps, B))
    tol_l2 = np.zeros((steps, B))
    n_alt = 0
    for b in range(B):
        k0, v0 = synth.kv_prefill(wl, b, 0)
        for st in range(steps):
            p = int(positions[b]) + st
            k_x, v_x, dk, dv = layer0_kv_exact(om, s, int(fed[st, b]), p)
            for side, xv, dl in (("k", k_x, dk), ("v", v_x, dv)):
                for blk, d2, q2 in helpers.q8_alternatives(xv, dl):
                    n_alt += 1
                    c = helpers.OverrideCache(cfg, B, wl.capacity, (b, p, side, blk, d2, q2))
                    c.fill(b, 0, k0, v0)
                    for s2 in range(st, steps):
                        if s2 == st:  # the rows before step st are the oracle's own: replay them unchanged
                            for s1 in range(st):
                                tok1 = np.zeros(B, np.int64)
                                tok1[b] = fed[s1, b]
                                pos1 = np.zeros(B, np.int64)
                                pos1[b] = positions[b] + s1
                                oracle.decode_step(om, c, tok1, pos1, seqs=[b])
                        tok = np.zeros(B, np.int64)
                        tok[b] = fed[s2, b]
                        pos = np.zeros(B, np.int64)
                        pos[b] = positions[b] + s2
                        lg, _, _ = oracle.decode_step(om, c, tok, pos, seqs=[b])
                        dlt = lg[0] - base[s2, b]
                        tol_abs[s2, b] += np.abs(dlt).max()
                        tol_l2[s2, b] += np.linalg.norm(dlt)
    return tol_abs, tol_l2, n_alt


# K = 256: at K = 2048 the derived bound of the GEMV (linear in K) admits thousands of alternatives per step
ONE_LAYER = {
    "q8_hd64_g2_1l": dataclasses.replace(SHAPES["q8_hd64_g2"], n_layers=1),
    "q4_hd128_g4_1l": dataclasses.replace(SHAPES["q4_hd128_g4"], n_layers=1),
}


@pytest.mark.parametrize("name,batch", [("q8_hd64_g2_1l", 1), ("q4_hd128_g4_1l", 3), ("q8_hd64_g2_1l", 16),
                                        ("q4_hd128_g4_1l", 16)])
def test_q8_cache_chain_one_layer(name, batch):
    """Greedy chains of 3 steps with a Q8_0 cache against the oracle with the same cache, on one-layer models
    (every new row is a layer-0 row, whose GPU error bound is derived), sequences at different positions.

    The GPU quantises its own fp32 rows, so a code may legitimately sit one step off the oracle's where the
    exact value lies within the derived bound of a rounding boundary (helpers.check_q8_blocks checks every
    new block against that rule).  The logits gate is the step's (max-abs 2e-3, relative L2 1e-4) widened by
    the change each such alternative alone makes to the oracle's logits (summed, times 1.25 for their
    interaction, which is of second order)."""
    shape = ONE_LAYER[name]
    wl = synth.Workload("t", shape, batch=batch, steps=3, prefill=37)
    s = Setup(wl)
    try:
        rng = np.random.default_rng(batch + shape.dim)
        tokens = rng.integers(0, shape.vocab, batch)
        positions = np.array([37, 0, 5, 36, 12, 37, 1, 20, 30, 7, 2, 33, 15, 9, 25, 37][:batch])
        fed, hist = gpu_chain(s.state, wl, 3, tokens0=tokens, positions0=positions)
        ofed, ohist = oracle.greedy(s.om, oracle_cache(wl, kv_type="q8_0"), tokens, positions, 3)
        for b in range(batch):
            for st in range(3):
                p = int(positions[b]) + st
                kd, kq, vd, vq = s.state.read_blocks(b, 0, p, 1)
                k_x, v_x, dk, dv = layer0_kv_exact(s.om, shape, int(fed[st, b]), p)
                check_q8_blocks(kd, kq, k_x, dk)
                check_q8_blocks(vd, vq, v_x, dv)
        tol_abs, tol_l2, n_alt = _flip_tolerance(s.om, wl, ofed, ohist, positions, 3)
        for b in range(batch):
            for st in range(3):
                g, w = hist[st, b], ohist[st, b]
                e = np.abs(g - w).max()
                r = np.linalg.norm(g - w)
                assert e <= 2e-3 + 1.25 * tol_abs[st, b], (b, st, e, tol_abs[st, b], n_alt)
                assert r <= 1e-4 * np.linalg.norm(w) + 1.25 * tol_l2[st, b], (b, st, r, tol_l2[st, b], n_alt)
                if fed[st, b] != ofed[st, b]:
                    # only where the oracle's top-2 gap is within reach; the chains part there
                    assert top2_gap(ohist[st - 1, b]) <= 2 * (2e-3 + 1.25 * tol_abs[st - 1, b]), (b, st)
                    break
    finally:
        s.close()


@pytest.mark.parametrize("name,batch", [("q8_hd64_g3_odd", 6), ("q4_hd128_g4", 16), ("q8_k2048_g4", 16)])
def test_q8_cache_chain_depth(name, batch):
    """Chains over several layers with the Q8_0 cache, for the layer indexing of the cache writes and reads.

    Beyond layer 0 the GPU's new rows have no derived error bound, so their legitimate one-code differences
    cannot be enumerated: the logits are held to a sanity bound ten times the step's gate (a wrong layer or
    row would move them by orders of magnitude more), and the greedy tokens to the oracle's where its top-2
    gap exceeds 0.05."""
    shape = SHAPES[name]
    wl = synth.Workload("t", shape, batch=batch, steps=3, prefill=37)
    s = Setup(wl)
    try:
        rng = np.random.default_rng(batch + shape.dim)
        tokens = rng.integers(0, shape.vocab, batch)
        positions = np.array([37, 0, 5, 36, 12, 37, 1, 20, 30, 7, 2, 33, 15, 9, 25, 37][:batch])
        fed, hist = gpu_chain(s.state, wl, 3, tokens0=tokens, positions0=positions)
        ofed, ohist = oracle.greedy(s.om, oracle_cache(wl, kv_type="q8_0"), tokens, positions, 3)
        for b in range(batch):
            for st in range(3):
                if st and fed[st, b] != ofed[st, b]:
                    assert top2_gap(ohist[st - 1, b]) <= 0.05, (b, st)
                    break
                g, w = hist[st, b], ohist[st, b]
                assert np.abs(g - w).max() <= 2e-2 and rel_l2(g, w) <= 1e-3, (b, st)
    finally:
        s.close()


def test_q8_cache_graph_equals_eager():
    """The captured step and the eager launches give identical logits on the Q8_0 cache."""
    shape = SHAPES["q4_hd128_g4"]
    wl = synth.Workload("t", shape, batch=3, steps=2, prefill=20)
    a = Setup(wl)
    b = Setup(wl)
    try:
        tokens = np.array([1, 2, 3])
        positions = np.array([20, 3, 0])
        _, h1 = gpu_chain(a.state, wl, 2, tokens0=tokens, positions0=positions, graph=True)
        _, h2 = gpu_chain(b.state, wl, 2, tokens0=tokens, positions0=positions, graph=False)
        np.testing.assert_array_equal(h1, h2)
    finally:
        a.close()
        b.close()
