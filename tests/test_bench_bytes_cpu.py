"""The roofline numerator of bench.py: its weight bytes equal the GGUF tensors the workloads are built from."""
import dataclasses
import os
import sys

import numpy as np
import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
import synth  # noqa: E402

TINY = synth.workload("tiny").shape
SHAPES = [TINY, dataclasses.replace(TINY, w_type="q4_0", tied=True, vocab=1000)]


@pytest.mark.parametrize("shape", SHAPES, ids=["q8_untied", "q4_tied"])
def test_matrix_bytes_match_generated_tensors(shape):
    w = synth.model_weights(shape, threads=4)
    nb = {k: v.nbytes for k, v in w.items()}
    got = bench.matrix_bytes(shape)
    for l in range(shape.n_layers):
        p = f"blk.{l}."
        assert got["qkv"] == nb[p + "attn_q.weight"] + nb[p + "attn_k.weight"] + nb[p + "attn_v.weight"]
        assert got["wo"] == nb[p + "attn_output.weight"]
        assert got["gateup"] == nb[p + "ffn_gate.weight"] + nb[p + "ffn_up.weight"]
        assert got["down"] == nb[p + "ffn_down.weight"]
    head = "token_embd.weight" if shape.tied else "output.weight"
    assert got["head"] == nb[head]


def test_step_bytes_grow_with_cached_rows():
    """One more cached row of every sequence adds exactly one K and one V row of fp16 per layer."""
    wl = synth.workload("tiny").with_(batch=3)
    pos = np.array([5, 9, 0])
    s = wl.shape
    diff = bench.step_bytes(wl, pos + 1) - bench.step_bytes(wl, pos)
    assert diff == s.n_layers * wl.batch * s.kvd * 2 * 2


def test_q8_cache_bytes():
    """With a Q8_0 cache a cached row costs kvd/32 blocks of 34 bytes per side, read once by attention."""
    wl = synth.workload("tiny").with_(batch=2, kv_type="q8_0")
    s = wl.shape
    pos = np.array([4, 11])
    diff = bench.step_bytes(wl, pos + 1) - bench.step_bytes(wl, pos)
    assert diff == s.n_layers * wl.batch * (s.kvd // 32) * 34 * 2
    # the new rows: fp32 staging written and read, then their blocks written, per side
    f16 = bench.stage_bytes(wl.with_(kv_type="f16"), pos)["qkv"]
    q8 = bench.stage_bytes(wl, pos)["qkv"]
    assert q8 - f16 == wl.batch * 2 * (s.kvd * 4 * 2 + s.kvd / 32 * 34 - s.kvd * 2)


def test_q8_cache_workload_is_the_8b_batch_with_a_q8_cache():
    a, b = synth.workload("llama3_8b_q8_b16"), synth.workload("llama3_8b_q8_b16_kvq8")
    assert b.kv_type == "q8_0" and a.kv_type == "f16"
    assert (a.shape, a.batch, a.steps, a.prefill) == (b.shape, b.batch, b.steps, b.prefill)
    assert np.array_equal(synth.kv_prefill(a.with_(shape=TINY), 1, 0)[0], synth.kv_prefill(b.with_(shape=TINY), 1, 0)[0])
