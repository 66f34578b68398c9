"""Glue between the seeded generator and the oracle (tests only)."""

from __future__ import annotations

import dataclasses

import numpy as np

import oracle
import synth


def oracle_config(shape: synth.ModelShape) -> oracle.OracleConfig:
    return oracle.OracleConfig(**{f.name: getattr(shape, f.name) for f in dataclasses.fields(oracle.OracleConfig)})


def oracle_model(shape: synth.ModelShape, weights=None, cache_dequant=True) -> oracle.OracleModel:
    if weights is None:
        weights = synth.gen.model_weights(shape)
    return oracle.OracleModel(oracle_config(shape), weights, cache_dequant=cache_dequant)


def oracle_cache(wl: synth.Workload, seqs=None) -> oracle.OracleCache:
    cfg = oracle_config(wl.shape)
    cache = oracle.OracleCache(cfg, wl.batch, wl.capacity)
    for b in (range(wl.batch) if seqs is None else seqs):
        for l in range(wl.shape.n_layers):
            k, v = synth.kv_prefill(wl, b, l)
            cache.fill(b, l, k, v)
    return cache


TINY = synth.ModelShape(n_layers=2, dim=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96, vocab=128,
                        rope_base=10000.0, rms_eps=1e-5, w_type="q8_0", tied=False)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ------------------------------------------------------------------------------------------
# GPU side (imports the CUDA binding lazily; only GPU tests call these)
# ------------------------------------------------------------------------------------------
def gpu_model(shape, weights, max_batch=1):
    from block_quantized_token_gb300 import runtime
    return runtime.DecodeModel(shape, weights, max_batch=max_batch)


def gpu_state(model, wl, seqs=None):
    from block_quantized_token_gb300 import runtime
    st = runtime.DecodeState(model, wl.batch, wl.capacity)
    for b in (range(wl.batch) if seqs is None else seqs):
        for l in range(wl.shape.n_layers):
            k, v = synth.kv_prefill(wl, b, l)
            st.write_rows(b, l, k, v)
    return st


def gpu_chain(state, wl, steps, tokens0=None, positions0=None, graph=True):
    """Run `steps` greedy steps chained on the device; returns (tokens fed [steps, B], logits [steps, B, V])."""
    import torch
    dev = state.model.device
    tok = torch.tensor(wl.tokens0() if tokens0 is None else tokens0, dtype=torch.int32, device=dev)
    pos = torch.tensor(wl.positions0() if positions0 is None else positions0, dtype=torch.int32, device=dev)
    logits = torch.empty((wl.batch, wl.shape.vocab), dtype=torch.float32, device=dev)
    fed = torch.empty((steps, wl.batch), dtype=torch.int32, device=dev)
    hist = torch.empty((steps, wl.batch, wl.shape.vocab), dtype=torch.float32, device=dev)
    from block_quantized_token_gb300 import er
    stream = torch.cuda.current_stream(dev).cuda_stream
    for s in range(steps):
        fed[s].copy_(tok)
        state.step(tok, pos, logits, tok, graph=graph)
        hist[s].copy_(logits)
        er.er_positions_increment(pos.data_ptr(), wl.batch, stream)
    torch.cuda.synchronize()
    return fed.cpu().numpy(), hist.cpu().numpy().astype(np.float64)


def logits_close(got, want, max_abs=2e-3, rel=1e-4):
    """The logits gate: max |got - want| <= 2e-3 and ||got - want|| / ||want|| <= 1e-4 per row."""
    got = np.asarray(got, np.float64).reshape(-1, np.shape(want)[-1])
    want = np.asarray(want, np.float64).reshape(got.shape)
    for g, w in zip(got, want):
        e = np.abs(g - w).max()
        r = rel_l2(g, w)
        assert e <= max_abs and r <= rel, f"max abs {e:.3e} (<= {max_abs}), rel L2 {r:.3e} (<= {rel})"


def top2_gap(logits):
    s = np.sort(np.asarray(logits, np.float64))
    return float(s[-1] - s[-2])
