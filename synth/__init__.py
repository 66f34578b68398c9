"""Seeded synthetic inputs for the block-quantized decode step.

This module is the one piece both sides of a parity check consume: it draws the
random weights and KV-cache rows of a workload and packs the weights into GGUF
Q8_0 / Q4_0 block bytes.  It holds none of the decode-step arithmetic (no
dequantisation, norm, projection, rotation or attention): the CUDA library and
the float64 oracle each implement those on their own, from these bytes.

Workloads (shapes of the pages' models, synthetic values):

* ``tiny``  -- 2 layers, dim 576, GQA 9/3, head dim 64, FFN 1536, vocab 4096,
  untied head, Q8_0, one decode step of token 7 at position 16.
* ``smollm_q8``  -- SmolLM2-135M shape (30 layers, dim 576, GQA 9/3, head dim 64,
  FFN 1536, vocab 49152, tied head), Q8_0, context 2048, 64 greedy steps.  The
  alpaca.swift README ("Results") measures this model's decode at contexts 16
  and 2048.
* ``smollm_q4``  -- the same shape in Q4_0, context 16, 64 greedy steps.
* ``llama2_7b_q4``  -- Llama-2-7B shape (32 layers, dim 4096, 32/32 heads of 128,
  FFN 11008, vocab 32000), Q4_0, context 4096, 64 greedy steps.
* ``llama3_8b_q8_b16``  -- Llama-3-8B shape (32 layers, dim 4096, GQA 32/8, head
  dim 128, FFN 14336, vocab 128256, RoPE base 5e5), Q8_0, 16 independent
  sequences at context 8192, 32 greedy steps.

Draw recipe (numpy PCG64 via ``default_rng``):

* Tensor ``i`` of the fixed order (per layer: attn_norm, attn_q, attn_k, attn_v,
  attn_output, ffn_norm, ffn_gate, ffn_up, ffn_down; then token_embd,
  output_norm, output) is drawn from ``default_rng([0, i])``.
* 2-D weights: float32 N(0, 1) * 0.02, then quantised (``quantize_q8_0`` /
  ``quantize_q4_0``).  Norm gains: float32 1 + 0.1 * N(0, 1).  An untied
  token_embd is fp16 (float32 draw rounded to nearest even); a tied one is
  stored in the weight block format and doubles as the output head.
* KV prefill of sequence ``b``, layer ``l``: ``default_rng([1, b, l])`` draws K
  then V, each float32 N(0, 1) of shape [prefill, n_kv_heads * head_dim]
  (token-major, heads contiguous), rounded to fp16.
* Sequence ``b`` starts at token ``7 + b`` and position ``prefill``.
"""

from .gen import (  # noqa: F401
    BLOCK_BYTES,
    WORKLOADS,
    ModelShape,
    Workload,
    kv_prefill,
    model_weights,
    quantize,
    quantize_q4_0,
    quantize_q8_0,
    tensor_names,
    weight_tensor,
    workload,
)
