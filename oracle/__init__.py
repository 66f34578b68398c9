"""Float64 CPU oracle of one block-quantized Llama decode step.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import or run anything in
this package.  The CUDA library never calls it and shares no code with it: the
two meet only through the seeded input bytes of the ``synth`` module.

The oracle is the plain definition of the step, written in numpy float64 with
no blocking, fusion or reordering:

  tokens -> embedding -> [RMSNorm -> Q/K/V -> RoPE -> K/V append -> GQA
  attention -> Wo + residual -> RMSNorm -> SwiGLU FFN + residual] x N ->
  RMSNorm -> LM head -> logits -> greedy argmax

(the pipeline of "EdgeRunner Core Architecture", Overview and section 5.1).
Each function cites the passage it follows.  The KV cache holds fp16, as the
pages' default cache precision does; every other value is float64.

Pins (tests/test_oracle_pins.py) tie each function to something other than
itself: hand-built blocks with hand-derived values (tests/golden/), closed
forms, invariants, torch float64 library routines, and cached-vs-uncached
decoding.  The whole step is checked against a composition of torch float64
routines (rms_norm, scaled_dot_product_attention with GQA, silu, RoPE as a
complex rotation, struct-decoded blocks) on four small shapes.  No pin
compares with output values the pages print: they print no logits for any
model.
"""

from .blocks import (BLOCK_BYTES, dequant, dequant_kv_q8_0, dequant_q4_0, dequant_q8_0, dequant_rows,  # noqa: F401
                     quantize_kv_q8_0)
from .ops import attention_gqa, matvec, rmsnorm, rope, silu, softmax, swiglu  # noqa: F401
from .decode import OracleCache, OracleConfig, OracleModel, decode_step, greedy, uncached_logits  # noqa: F401
