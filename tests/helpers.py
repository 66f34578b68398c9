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
