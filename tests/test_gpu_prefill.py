"""Chunked prefill (er_prefill) against the oracle's token-by-token decode of the same tokens.

A prefill of n tokens at positions start.. equals n decode steps of that sequence, so the oracle side is
oracle.decode_step fed the tokens one by one (pinned against the uncached recompute).  Checked: every layer-0
K/V row the prefill writes, within the derived bound of the GPU's fp32 arithmetic
(helpers.layer0_kv_tolerance); the last token's logits within the step's gate (max-abs 2e-3, relative L2
1e-4); greedy decode steps after the prefill; other sequences' rows untouched; argument and device-flag
errors.  Chunks of 16 tokens with a ragged last chunk, continuation from a start above zero, tied/untied,
Q4_0/Q8_0, hd 64/128, K a multiple of 64 (the one-pass batched GEMV) or not (column groups).
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import helpers
import oracle
import synth
from helpers import (check_q8_blocks, gpu_chain, gpu_model, gpu_state, layer0_kv_exact, layer0_kv_tolerance,
                     logits_close, oracle_config, oracle_model)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

SHAPES = {
    "q8_hd64_g2": synth.ModelShape(n_layers=2, dim=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn_dim=256, vocab=512,
                                   rope_base=10000.0, rms_eps=1e-5, w_type="q8_0", tied=False),
    "q4_hd128_g4_tied": synth.ModelShape(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=320,
                                         vocab=1000, rope_base=500000.0, rms_eps=1e-5, w_type="q4_0", tied=True),
    "q8_hd64_g3_odd": synth.ModelShape(n_layers=3, dim=96 * 3, n_heads=9, n_kv_heads=3, head_dim=64, ffn_dim=416,
                                       vocab=777, rope_base=10000.0, rms_eps=1e-6, w_type="q8_0", tied=True),
}


def _er():
    from block_quantized_token_gb300 import er
    return er


def _oracle_prefill(om, cache, seq, tokens, start, batch):
    """The oracle's decode of `tokens` one by one for sequence `seq` (positions start..); last logits."""
    lg = None
    for i, t in enumerate(tokens):
        tok = np.zeros(batch, np.int64)
        pos = np.zeros(batch, np.int64)
        tok[seq], pos[seq] = int(t), start + i
        lg, _, _ = oracle.decode_step(om, cache, tok, pos, seqs=[seq])
    return lg[0]


def _dev_tokens(tokens):
    return torch.tensor(np.asarray(tokens, np.int32), dtype=torch.int32, device="cuda")


def _check_layer0_rows(state, om, shape, seq, tokens, start):
    k, v = state.read_rows(seq, 0, start, len(tokens))
    k, v = k.cpu().numpy().astype(np.float64), v.cpu().numpy().astype(np.float64)
    for i, t in enumerate(tokens):
        kx, vx, _, _ = layer0_kv_exact(om, shape, int(t), start + i)
        tk, tv = layer0_kv_tolerance(om, shape, int(t), start + i)
        assert (np.abs(k[i] - kx.astype(np.float16).astype(np.float64)) <= tk).all(), (i, "k")
        assert (np.abs(v[i] - vx.astype(np.float16).astype(np.float64)) <= tv).all(), (i, "v")


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("n", [1, 16, 37])
def test_prefill_matches_oracle(name, n):
    """Prefill n tokens of a fresh sequence (chunks of 16, ragged tail), then continue with 7 more from
    position n: every layer-0 row and the last logits of both calls against the oracle."""
    shape = SHAPES[name]
    wl = synth.Workload("t", shape, batch=1, steps=8, prefill=n)  # capacity n + 8
    weights = synth.gen.model_weights(shape)
    om = oracle_model(shape, weights)
    model = gpu_model(shape, weights, max_batch=1)
    from block_quantized_token_gb300 import runtime
    st = runtime.DecodeState(model, 1, wl.capacity)
    try:
        rng = np.random.default_rng(n + shape.dim)
        toks = rng.integers(0, shape.vocab, n + 7)
        cache = oracle.OracleCache(oracle_config(shape), 1, wl.capacity)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        st.prefill(0, _dev_tokens(toks[:n]), 0, logits)
        torch.cuda.synchronize()
        want = _oracle_prefill(om, cache, 0, toks[:n], 0, 1)
        logits_close(logits.cpu().numpy(), want)
        _check_layer0_rows(st, om, shape, 0, toks[:n], 0)
        st.prefill(0, _dev_tokens(toks[n:]), n, logits)
        torch.cuda.synchronize()
        want = _oracle_prefill(om, cache, 0, toks[n:], n, 1)
        logits_close(logits.cpu().numpy(), want)
        _check_layer0_rows(st, om, shape, 0, toks[n:], n)
        assert st.device_error()[1] == 0
    finally:
        st.close()
        model.close()


@pytest.mark.parametrize("name", ["q8_hd64_g2", "q8_hd64_g3_odd"])
def test_prefill_then_greedy(name):
    """Prefill 29 tokens, then 3 greedy decode steps on the device: tokens and logits against the oracle's
    cache after its own token-by-token prefill."""
    shape = SHAPES[name]
    n = 29
    wl = synth.Workload("t", shape, batch=1, steps=3, prefill=n)
    weights = synth.gen.model_weights(shape)
    om = oracle_model(shape, weights)
    model = gpu_model(shape, weights, max_batch=1)
    from block_quantized_token_gb300 import runtime
    st = runtime.DecodeState(model, 1, wl.capacity)
    try:
        toks = np.random.default_rng(3).integers(0, shape.vocab, n)
        st.prefill(0, _dev_tokens(toks), 0)
        cache = oracle.OracleCache(oracle_config(shape), 1, wl.capacity)
        lg = _oracle_prefill(om, cache, 0, toks, 0, 1)
        first = int(np.argmax(lg))
        fed, hist = gpu_chain(st, wl, 3, tokens0=[first], positions0=[n])
        ofed, ohist = oracle.greedy(om, cache, [first], [n], 3)
        np.testing.assert_array_equal(fed, ofed)
        for s in range(3):
            logits_close(hist[s], ohist[s])
    finally:
        st.close()
        model.close()


def test_prefill_one_sequence_of_a_batch():
    """Prefill sequence 2 of a 16-sequence state (the batched schedule) at a start above zero: its rows match
    the oracle, the other sequences' rows are untouched, and a following batched step agrees with the oracle
    for every sequence."""
    shape = SHAPES["q4_hd128_g4_tied"]
    wl = synth.Workload("t", shape, batch=16, steps=24, prefill=20)
    weights = synth.gen.model_weights(shape)
    om = oracle_model(shape, weights)
    model = gpu_model(shape, weights, max_batch=16)
    st = gpu_state(model, wl)
    try:
        before = [st.read_rows(b, 1, 0, wl.capacity) for b in (0, 1, 3, 15)]
        toks = np.random.default_rng(9).integers(0, shape.vocab, 21)
        st.prefill(2, _dev_tokens(toks), 20)
        torch.cuda.synchronize()
        for b, (k0, v0) in zip((0, 1, 3, 15), before):
            k1, v1 = st.read_rows(b, 1, 0, wl.capacity)
            assert torch.equal(k0, k1) and torch.equal(v0, v1), b
        cfg = oracle_config(shape)
        cache = oracle.OracleCache(cfg, 16, wl.capacity)
        for b in range(16):
            for l in range(shape.n_layers):
                cache.fill(b, l, *synth.kv_prefill(wl, b, l))
        _oracle_prefill(om, cache, 2, toks, 20, 16)
        _check_layer0_rows(st, om, shape, 2, toks, 20)
        tokens = np.arange(16) + 3
        positions = np.full(16, 20)
        positions[2] = 41
        fed, hist = gpu_chain(st, wl, 2, tokens0=tokens, positions0=positions)
        ofed, ohist = oracle.greedy(om, cache, tokens, positions, 2)
        np.testing.assert_array_equal(fed, ofed)
        for s in range(2):
            logits_close(hist[s], ohist[s])
    finally:
        st.close()
        model.close()


def test_prefill_q8_cache():
    """Prefill into a Q8_0 cache (one layer: every row is a layer-0 row with a derived bound): each block is
    the oracle's quantisation up to the legitimate one-step alternatives (helpers.check_q8_blocks), and the
    last logits lie within the step's gate widened by the change each such alternative alone makes to the
    oracle's last logits (the oracle's prefill rerun with that one block replaced; summed, times 1.25)."""
    shape = dataclasses.replace(SHAPES["q8_hd64_g2"], n_layers=1)
    n = 21
    wl = synth.Workload("t", shape, batch=1, steps=2, prefill=n)
    weights = synth.gen.model_weights(shape)
    om = oracle_model(shape, weights)
    model = gpu_model(shape, weights, max_batch=1)
    from block_quantized_token_gb300 import runtime
    st = runtime.DecodeState(model, 1, wl.capacity, kv_type="q8_0")
    try:
        toks = np.random.default_rng(4).integers(0, shape.vocab, n)
        logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
        st.prefill(0, _dev_tokens(toks), 0, logits)
        kd, kq, vd, vq = st.read_blocks(0, 0, 0, n)
        rows = []
        for i, t in enumerate(toks):
            kx, vx, dk, dv = layer0_kv_exact(om, shape, int(t), i)
            check_q8_blocks(kd[i], kq[i], kx, dk)
            check_q8_blocks(vd[i], vq[i], vx, dv)
            rows.append((kx, vx, dk, dv))
        cfg = oracle_config(shape)
        want = _oracle_prefill(om, oracle.OracleCache(cfg, 1, wl.capacity, kv_type="q8_0"), 0, toks, 0, 1)
        tol_abs = tol_l2 = 0.0
        for i, (kx, vx, dk, dv) in enumerate(rows):
            for side, xv, dl in (("k", kx, dk), ("v", vx, dv)):
                for blk, d2, q2 in helpers.q8_alternatives(xv, dl):
                    c = helpers.OverrideCache(cfg, 1, wl.capacity, (0, i, side, blk, d2, q2))
                    dlt = _oracle_prefill(om, c, 0, toks, 0, 1) - want
                    tol_abs += np.abs(dlt).max()
                    tol_l2 += np.linalg.norm(dlt)
        got = logits.cpu().numpy().astype(np.float64)
        assert np.abs(got - want).max() <= 2e-3 + 1.25 * tol_abs
        assert np.linalg.norm(got - want) <= 1e-4 * np.linalg.norm(want) + 1.25 * tol_l2
    finally:
        st.close()
        model.close()


def test_prefill_errors():
    er = _er()
    shape = SHAPES["q8_hd64_g2"]
    wl = synth.Workload("t", shape, batch=2, steps=4, prefill=4)
    weights = synth.gen.model_weights(shape)
    model = gpu_model(shape, weights, max_batch=2)
    st = gpu_state(model, wl)
    try:
        t = _dev_tokens([1, 2, 3])
        for args in ((2, t.data_ptr(), 3, 0), (-1, t.data_ptr(), 3, 0), (0, t.data_ptr(), 3, 6),
                     (0, t.data_ptr(), -1, 0), (0, None, 3, 0), (0, t.data_ptr(), 3, -1)):
            with pytest.raises(er.ErError) as e:
                er.er_prefill(st.handle, *args, None, 0)
            assert e.value.status == er.ER_EINVAL, args
        er.er_prefill(st.handle, 0, None, 0, 8, None, 0)  # nothing to do
        bad = _dev_tokens([1, shape.vocab + 5, 2])
        st.prefill(1, bad, 0)
        torch.cuda.synchronize()
        _, code, _ = st.device_error()
        assert code & 1  # token out of range
        assert st.device_error()[1] == 0  # read and cleared
    finally:
        st.close()
        model.close()
