"""GPU parity of the whole decode step (C ABI) against the float64 oracle.

Gates: logits max |err| <= 2e-3 and relative L2 <= 1e-4 per step; greedy tokens
identical over the chained steps; the K/V rows layer 0 appends within the bound
derived from the GPU's fp32 arithmetic (helpers.layer0_kv_tolerance: the GEMV
bound, the RMSNorm factor's rounding, the rotation's, and one fp16 ulp).
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from helpers import (gpu_chain, gpu_model, gpu_state, layer0_kv_tolerance, logits_close, oracle_cache,
                     oracle_config, oracle_model, top2_gap)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _er():
    from block_quantized_token_gb300 import er
    return er


PERSISTENT, KERNELS = 1, 2  # er_schedule values


class Setup:
    def __init__(self, wl, max_batch=None, seqs=None, schedule=None):
        self.wl = wl
        self.weights = synth.gen.model_weights(wl.shape)
        self.model = gpu_model(wl.shape, self.weights, max_batch=max_batch or wl.batch)
        self.state = gpu_state(self.model, wl)
        if schedule is not None:
            self.state.set_schedule(schedule)
        self.om = oracle_model(wl.shape, self.weights)

    def ocache(self, seqs=None):
        return oracle_cache(self.wl, seqs)

    def reset_kv(self):
        """Rewrite the prefill rows and zero the rest, as a fresh oracle cache holds them."""
        wl = self.wl
        zeros = np.zeros((wl.capacity - wl.prefill, wl.shape.kvd), np.float16)
        for b in range(wl.batch):
            for l in range(wl.shape.n_layers):
                k, v = synth.kv_prefill(wl, b, l)
                self.state.write_rows(b, l, k, v)
                self.state.write_rows(b, l, zeros, zeros, start=wl.prefill)

    def close(self):
        self.state.close()
        self.model.close()


@pytest.fixture(scope="module")
def tiny():
    s = Setup(synth.workload("tiny").with_(steps=4))
    yield s
    s.close()


def _step(state, wl, tokens, positions, graph=True):
    dev = state.model.device
    t = torch.tensor(tokens, dtype=torch.int32, device=dev)
    p = torch.tensor(positions, dtype=torch.int32, device=dev)
    lg = torch.empty((wl.batch, wl.shape.vocab), dtype=torch.float32, device=dev)
    am = torch.empty(wl.batch, dtype=torch.int32, device=dev)
    state.step(t, p, lg, am, graph=graph)
    torch.cuda.synchronize()
    return lg.cpu().numpy().astype(np.float64), am.cpu().numpy()


def test_tiny_single_step(tiny):
    """2-layer Q8_0 model, token 7 at position 16 over a 16-row prefill."""
    wl = tiny.wl
    got, am = _step(tiny.state, wl, wl.tokens0(), wl.positions0())
    oc = tiny.ocache()
    want, oam, onf = oracle.decode_step(tiny.om, oc, wl.tokens0(), wl.positions0())
    logits_close(got, want)
    assert list(am) == list(oam), f"top-2 gap {top2_gap(want[0]):.3e}"
    assert not onf.any()
    # the rows layer 0 appended (post-RoPE K, V) against the oracle's fp16 rows, within the derived bound
    p = wl.prefill
    k, v = tiny.state.read_rows(0, 0, p, 1)
    tk, tv = layer0_kv_tolerance(tiny.om, wl.shape, int(wl.tokens0()[0]), p)
    for g, w, tol in ((k, oc.k[0][0][p], tk), (v, oc.v[0][0][p], tv)):
        g = g.cpu().numpy().reshape(-1).astype(np.float64)
        w = w.reshape(-1).astype(np.float64)
        d = np.abs(g - w)
        assert (d <= tol).all(), f"worst excess {np.max(d - tol):.3e} at {np.argmax(d - tol)}"
    st, code, nf = tiny.state.device_error()
    assert code == 0 and nf == 0


def test_schedules_agree(tiny):
    """The persistent step and the per-phase kernels compute the same step."""
    wl = tiny.wl
    assert tiny.state.schedule == PERSISTENT  # chosen automatically for this shape
    tiny.reset_kv()
    a, am_a = _step(tiny.state, wl, wl.tokens0(), wl.positions0())
    tiny.state.set_schedule(KERNELS)
    try:
        b, am_b = _step(tiny.state, wl, wl.tokens0(), wl.positions0())
    finally:
        tiny.state.set_schedule(PERSISTENT)
    want, oam, _ = oracle.decode_step(tiny.om, tiny.ocache(), wl.tokens0(), wl.positions0())
    logits_close(a, want)
    logits_close(b, want)
    assert list(am_a) == list(am_b) == list(oam)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-4)


def test_graph_equals_eager_and_deterministic(tiny):
    wl = tiny.wl
    a, am_a = _step(tiny.state, wl, wl.tokens0(), wl.positions0(), graph=True)
    b, am_b = _step(tiny.state, wl, wl.tokens0(), wl.positions0(), graph=False)
    c, am_c = _step(tiny.state, wl, wl.tokens0(), wl.positions0(), graph=True)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, c)
    assert list(am_a) == list(am_b) == list(am_c)


def test_tiny_chain(tiny):
    """Four chained greedy steps (tokens fed back on the device)."""
    wl = tiny.wl
    fed, hist = gpu_chain(tiny.state, wl, 4)
    ofed, ohist = oracle.greedy(tiny.om, tiny.ocache(), wl.tokens0(), wl.positions0(), 4)
    np.testing.assert_array_equal(fed, ofed)
    for s in range(4):
        logits_close(hist[s], ohist[s])


@pytest.mark.parametrize("pos", [0, 1, 15, 16, 19])
def test_positions_edge(tiny, pos):
    """Position 0 (one row attended), the prefill boundary and the last row of the cache (19)."""
    tiny.reset_kv()
    got, am = _step(tiny.state, tiny.wl, [3], [pos])
    oc = tiny.ocache()
    want, oam, _ = oracle.decode_step(tiny.om, oc, [3], [pos])
    logits_close(got, want)
    assert list(am) == list(oam)


def test_device_errors(tiny):
    wl = tiny.wl
    er = _er()
    for tok, pos, bit in ((wl.shape.vocab, 16, 1), (-1, 16, 1), (5, wl.capacity, 2), (5, -3, 2)):
        _step(tiny.state, wl, [tok], [pos])
        st, code, nf = tiny.state.device_error()
        assert st == er.ER_EDEVICE and code & bit, (tok, pos, code)
    st, code, nf = tiny.state.device_error()
    assert st == er.ER_OK and code == 0


SMALL_SHAPES = {
    "q4_tied_g2": synth.ModelShape(n_layers=2, dim=128, n_heads=2, n_kv_heads=1, head_dim=64, ffn_dim=160,
                                   vocab=300, rope_base=10000.0, rms_eps=1e-5, w_type="q4_0", tied=True),
    "q8_mha": synth.ModelShape(n_layers=2, dim=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn_dim=256, vocab=512,
                               rope_base=10000.0, rms_eps=1e-5, w_type="q8_0", tied=False),
    "q4_hd128_g4": synth.ModelShape(n_layers=2, dim=256, n_heads=8, n_kv_heads=2, head_dim=128, ffn_dim=320,
                                    vocab=1000, rope_base=500000.0, rms_eps=1e-5, w_type="q4_0", tied=False),
    "q8_hd64_g3_odd": synth.ModelShape(n_layers=3, dim=96 * 3, n_heads=9, n_kv_heads=3, head_dim=64, ffn_dim=416,
                                       vocab=777, rope_base=10000.0, rms_eps=1e-6, w_type="q8_0", tied=True),
}


@pytest.mark.parametrize("schedule", [PERSISTENT, KERNELS], ids=["persistent", "kernels"])
@pytest.mark.parametrize("name", list(SMALL_SHAPES))
@pytest.mark.parametrize("batch", [1, 3, 6, 16])
def test_small_models_ragged_batch(name, batch, schedule):
    """Tied/untied, Q4_0/Q8_0, G = 1/3/4, hd 64/128, odd sizes; sequences at different positions.

    Batches above 4 run the one-pass batched GEMV where K is a multiple of 64
    (the odd shape keeps the column-group path)."""
    shape = SMALL_SHAPES[name]
    wl = synth.Workload("t", shape, batch=batch, steps=3, prefill=37)
    if schedule == PERSISTENT and batch > 4:
        s = Setup(wl)
        try:
            with pytest.raises(_er().ErError) as e:
                s.state.set_schedule(PERSISTENT)
            assert e.value.status == _er().ER_EUNSUPPORTED
            assert s.state.schedule == KERNELS
        finally:
            s.close()
        return
    s = Setup(wl, schedule=schedule)
    try:
        rng = np.random.default_rng(batch)
        tokens = rng.integers(0, shape.vocab, batch)
        positions = np.array([37, 0, 5, 36, 12, 37, 1, 20, 30, 7, 2, 33, 15, 9, 25, 37][:batch])
        dev = s.model.device
        t = torch.tensor(tokens, dtype=torch.int32, device=dev)
        p = torch.tensor(positions, dtype=torch.int32, device=dev)
        fed, hist = gpu_chain(s.state, wl, 3, tokens0=tokens, positions0=positions)
        ofed, ohist = oracle.greedy(s.om, s.ocache(), tokens, positions, 3)
        np.testing.assert_array_equal(fed, ofed)
        for st in range(3):
            logits_close(hist[st], ohist[st])
        del t, p
    finally:
        s.close()


WIDE_SHAPES = {
    # K = 2048 and 2560 span 2 and 3 slices of the batched GEMV (the last one partial)
    "q8_k2048": synth.ModelShape(n_layers=2, dim=2048, n_heads=16, n_kv_heads=4, head_dim=128, ffn_dim=2560,
                                 vocab=1000, rope_base=10000.0, rms_eps=1e-5, w_type="q8_0", tied=False),
    "q4_k2048_tied": synth.ModelShape(n_layers=2, dim=2048, n_heads=32, n_kv_heads=8, head_dim=64, ffn_dim=2560,
                                      vocab=700, rope_base=500000.0, rms_eps=1e-6, w_type="q4_0", tied=True),
}


WIDE_VARIANTS = {"mma_sync": 1, "tcgen05": 2}  # er_wide_gemv: ER_WIDE_MMA_SYNC, ER_WIDE_TCGEN05


@pytest.mark.parametrize("variant", list(WIDE_VARIANTS))
@pytest.mark.parametrize("name", list(WIDE_SHAPES))
@pytest.mark.parametrize("batch", [6, 16])
def test_batched_gemv_multi_slice(name, batch, variant):
    """Batches of 5..16 on the per-phase schedule with matrices of several K-slices, under both batched GEMV
    kernels: logits of every sequence against the oracle over 2 chained steps, sequences at different positions."""
    shape = WIDE_SHAPES[name]
    wl = synth.Workload("t", shape, batch=batch, steps=2, prefill=29)
    s = Setup(wl, schedule=KERNELS)
    try:
        s.state.set_wide_gemv(WIDE_VARIANTS[variant])
        rng = np.random.default_rng(batch + shape.dim)
        tokens = rng.integers(0, shape.vocab, batch)
        positions = rng.integers(0, 30, batch)
        fed, hist = gpu_chain(s.state, wl, 2, tokens0=tokens, positions0=positions)
        ofed, ohist = oracle.greedy(s.om, s.ocache(), tokens, positions, 2)
        np.testing.assert_array_equal(fed, ofed)
        for st in range(2):
            logits_close(hist[st], ohist[st])
    finally:
        s.close()


@pytest.mark.parametrize("name", ["q4_tied_g2", "q8_mha", "q4_hd128_g4"])
@pytest.mark.parametrize("batch", [5, 16])
def test_small_models_tcgen05_batched_gemv(name, batch):
    """The tcgen05 batched GEMV forced on small shapes (one K-slice, ragged 128-row tiles, tied Q4_0 heads):
    greedy tokens and logits of 3 chained steps against the oracle."""
    shape = SMALL_SHAPES[name]
    wl = synth.Workload("t", shape, batch=batch, steps=3, prefill=37)
    s = Setup(wl, schedule=KERNELS)
    try:
        s.state.set_wide_gemv(WIDE_VARIANTS["tcgen05"])
        rng = np.random.default_rng(batch + 7)
        tokens = rng.integers(0, shape.vocab, batch)
        positions = rng.integers(0, 38, batch)
        fed, hist = gpu_chain(s.state, wl, 3, tokens0=tokens, positions0=positions)
        ofed, ohist = oracle.greedy(s.om, s.ocache(), tokens, positions, 3)
        np.testing.assert_array_equal(fed, ofed)
        for st in range(3):
            logits_close(hist[st], ohist[st])
    finally:
        s.close()


def test_wide_gemv_variant_rejected():
    """An unknown batched GEMV variant is refused with ER_EINVAL."""
    wl = synth.Workload("t", SMALL_SHAPES["q8_mha"], batch=6, steps=1, prefill=4)
    s = Setup(wl, schedule=KERNELS)
    try:
        with pytest.raises(_er().ErError) as e:
            s.state.set_wide_gemv(7)
        assert e.value.status == _er().ER_EINVAL
    finally:
        s.close()


def test_nonfinite_flag():
    """An infinite block scale in the head makes logits non-finite: flag set, argmax stays in range."""
    shape = SMALL_SHAPES["q8_mha"]
    weights = synth.gen.model_weights(shape)
    head = weights["output.weight"].copy()
    blk = head.reshape(shape.vocab, -1, 34)
    blk[5, 0, 0:2] = np.frombuffer(np.float16(np.inf).tobytes(), np.uint8)
    weights["output.weight"] = head
    wl = synth.Workload("t", shape, batch=1, steps=1, prefill=4)
    model = gpu_model(shape, weights)
    st = gpu_state(model, wl)
    try:
        got, am = _step(st, wl, [1], [4])
        status, code, nf = st.device_error()
        assert nf == 1 and code == 0
        assert 0 <= am[0] < shape.vocab
    finally:
        st.close()
        model.close()


def test_bad_config_rejected():
    er = _er()
    from block_quantized_token_gb300 import runtime
    shape = SMALL_SHAPES["q8_mha"]
    for field, val, status in (("head_dim", 96, er.ER_EUNSUPPORTED), ("n_kv_heads", 3, er.ER_EINVAL),
                               ("max_batch", 17, er.ER_EINVAL), ("dim", 48, er.ER_EINVAL)):
        cfg = runtime.make_config(shape)
        setattr(cfg, field, val)
        w = er.er_weights()
        with pytest.raises(er.ErError) as e:
            er.er_model_create(cfg, w, 0)
        assert e.value.status == status, (field, e.value)


# ------------------------------------------------------------------------------------------
# the pages' workload shapes
# ------------------------------------------------------------------------------------------
@pytest.mark.parametrize("schedule", [PERSISTENT, KERNELS], ids=["persistent", "kernels"])
@pytest.mark.parametrize("name", ["smollm_q8", "smollm_q4"])
def test_smollm_chain_64(name, schedule):
    """SmolLM2-135M shape, 64 chained greedy steps (context 2048 for Q8_0, 16 for Q4_0)."""
    wl = synth.workload(name)
    s = Setup(wl, schedule=schedule)
    try:
        fed, hist = gpu_chain(s.state, wl, wl.steps)
        ofed, ohist = oracle.greedy(s.om, s.ocache(), wl.tokens0(), wl.positions0(), wl.steps)
        for st in range(wl.steps):
            assert fed[st, 0] == ofed[st, 0], f"step {st}: token {fed[st, 0]} vs {ofed[st, 0]}, " \
                                              f"top-2 gap {top2_gap(ohist[st - 1, 0]):.3e}"
            logits_close(hist[st], ohist[st])
    finally:
        s.close()
