"""GPU parity at the benchmark's full sizes (the 7B-shaped Q4_0 and the 8B-shaped
16-sequence Q8_0 workloads), in the schedule bench.py times.

A whole float64 step of these models takes the oracle minutes, so the step is
checked on outputs the oracle computes cheaply, and on properties that hold at
any size:

* the new K/V cache rows of layers 0 and 1 at each sampled sequence's position
  (layer 1's rows depend on all of layer 0: RMSNorm, the Q/K/V projection,
  RoPE, attention over the whole context, Wo, the SwiGLU FFN and both
  residuals), against the oracle run on the model cut to its first two
  layers with the same tensors;
* the returned argmax is the first maximum of the returned logits, the logits
  are finite, no device flag is raised;
* replaying the step graph gives bit-identical logits.
"""

from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import oracle
import synth
from helpers import oracle_config

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")

CASES = {"llama2_7b_q4": [0], "llama3_8b_q8_b16": [0, 15]}


def _setup(wl):
    from block_quantized_token_gb300 import runtime
    s = wl.shape
    threads = min(32, os.cpu_count() or 1)
    model = runtime.DecodeModel(s, synth.model_weights(s, threads=threads), max_batch=wl.batch)
    state = runtime.DecodeState(model, wl.batch, wl.capacity)
    with ThreadPoolExecutor(max_workers=threads) as ex:
        jobs = [(b, l) for b in range(wl.batch) for l in range(s.n_layers)]
        for (b, l), (k, v) in zip(jobs, ex.map(lambda bl: synth.kv_prefill(wl, *bl), jobs)):
            state.write_rows(b, l, k, v)
    return model, state


def _row_close(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    ulp = np.abs(np.spacing(want.astype(np.float16)).astype(np.float64))
    tol = ulp + 1e-5 * np.max(np.abs(want))
    bad = np.abs(got - want) > tol
    assert not bad.any(), f"{bad.sum()} of {bad.size} elements, worst {np.max(np.abs(got - want) - tol)}"


@pytest.mark.parametrize("name", list(CASES))
def test_full_size_step(name):
    from block_quantized_token_gb300 import er
    wl = synth.workload(name).with_(steps=2)
    s = wl.shape
    seqs = CASES[name]
    model, state = _setup(wl)
    try:
        dev = model.device
        tok = torch.tensor(wl.tokens0(), dtype=torch.int32, device=dev)
        pos = torch.tensor(wl.positions0(), dtype=torch.int32, device=dev)
        logits = torch.empty((wl.batch, s.vocab), dtype=torch.float32, device=dev)
        argmax = torch.empty(wl.batch, dtype=torch.int32, device=dev)
        state.step(tok, pos, logits, argmax)  # the graph bench.py replays
        torch.cuda.synchronize()
        _, code, nonfinite = state.device_error()
        assert code == 0 and nonfinite == 0
        lg = logits.cpu().numpy()
        am = argmax.cpu().numpy()
        assert np.isfinite(lg).all()
        np.testing.assert_array_equal(am, np.argmax(lg, axis=1))
        # replay: the new cache rows are rewritten with the same values
        state.step(tok, pos, logits, argmax)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(logits.cpu().numpy(), lg)

        rows = {(b, l): state.read_rows(b, l, int(wl.positions0()[b]), 1) for b in seqs for l in (0, 1)}
    finally:
        state.close()
        model.close()

    # the oracle on the first two layers, with the full model's tensors
    cut = dataclasses.replace(s, n_layers=2)
    om = oracle.OracleModel(oracle_config(cut), lambda n: synth.weight_tensor(s, n))
    cache = oracle.OracleCache(oracle_config(cut), wl.batch, wl.capacity)
    for b in seqs:
        for l in (0, 1):
            k, v = synth.kv_prefill(wl, b, l)
            cache.fill(b, l, k, v)
    oracle.decode_step(om, cache, wl.tokens0(), wl.positions0(), seqs=seqs)
    for (b, l), (k, v) in rows.items():
        p = int(wl.positions0()[b])
        _row_close(k.cpu().numpy().reshape(-1), cache.k[b][l][p].reshape(-1))
        _row_close(v.cpu().numpy().reshape(-1), cache.v[b][l][p].reshape(-1))
