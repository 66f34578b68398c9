"""GPU: a model built from a GGUF file (er_model_create_from_gguf) decodes exactly as one built from the same
tensors in memory, and matches the oracle.

GGUF files store rope_base and rms_eps as float32, so both the in-memory model and the oracle use those values."""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest

import oracle
import synth
import synth.gguf as sg
from helpers import gpu_model, gpu_state, logits_close, oracle_cache, oracle_model

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


class _GgufModel:
    """The attributes DecodeState uses, around a handle from er_model_create_from_gguf."""

    def __init__(self, er, handle, shape):
        self.er, self.handle, self.shape, self.device = er, handle, shape, torch.device("cuda")

    def close(self):
        if self.handle:
            self.er.er_model_destroy(self.handle)
            self.handle = None


SHAPES = {
    "q4_tied_g2": synth.ModelShape(n_layers=2, dim=128, n_heads=2, n_kv_heads=1, head_dim=64, ffn_dim=160,
                                   vocab=300, rope_base=500000.0, rms_eps=1e-5, w_type="q4_0", tied=True),
    "q8_mha_hd128": synth.ModelShape(n_layers=2, dim=256, n_heads=2, n_kv_heads=2, head_dim=128, ffn_dim=256,
                                     vocab=512, rope_base=10000.0, rms_eps=1e-6, w_type="q8_0", tied=False),
    "tiny_576": synth.workload("tiny").shape,
}


@pytest.mark.parametrize("shape", list(SHAPES.values()), ids=list(SHAPES))
def test_model_from_gguf(tmp_path, shape):
    from block_quantized_token_gb300 import er
    shape = dataclasses.replace(shape, rope_base=float(np.float32(shape.rope_base)),
                                rms_eps=float(np.float32(shape.rms_eps)))
    tensors = synth.model_weights(shape)
    path = str(tmp_path / "m.gguf")
    sg.write_gguf(path, shape, tensors)
    wl = synth.Workload("t", shape, batch=2, steps=2, prefill=9)
    g = er.er_gguf_open(path)
    try:
        a = _GgufModel(er, er.er_model_create_from_gguf(g, 2, torch.cuda.current_stream().cuda_stream), shape)
    finally:
        er.er_gguf_close(g)  # the model keeps its own copy
    b = gpu_model(shape, tensors, max_batch=2)
    sa, sb = gpu_state(a, wl), gpu_state(b, wl)
    try:
        tok = torch.tensor([3, 11], dtype=torch.int32, device="cuda")
        pos = torch.tensor([9, 4], dtype=torch.int32, device="cuda")
        outs = []
        for st in (sa, sb):
            lg = torch.empty((2, shape.vocab), device="cuda")
            st.step(tok, pos, lg, None)
            torch.cuda.synchronize()
            outs.append(lg.cpu().numpy().astype(np.float64))
        np.testing.assert_array_equal(outs[0], outs[1])
        om = oracle_model(shape, tensors)
        want, _, _ = oracle.decode_step(om, oracle_cache(wl), [3, 11], [9, 4])
        logits_close(outs[0], want)
    finally:
        sa.close()
        sb.close()
        a.close()
        b.close()
