"""Writes the stored expected values of the full-size parity tests, from the oracle alone.

    python tests/golden/make_fullsize.py [llama2_7b_q4] [llama3_8b_q8_b16]

For each workload it draws the seeded weights and KV prefill (``synth``), runs
the float64 oracle's greedy chain (``oracle.greedy``) over the workload's
chained steps for the sequences listed in SEQS, and stores in
``tests/golden/fullsize_<workload>.npz``:

  seqs         the sequences computed (sequences are independent: each has
               its own cache and position, so a subset gives the same values)
  fed          int64 [steps, len(seqs)]: the token fed at every step
  logit_steps  the steps whose logits are stored
  logits       float64 [len(logit_steps), len(seqs), vocab]
  top2         float64 [steps, len(seqs)]: the gap between the two largest
               logits at every step (how close each greedy choice was)

Nothing here comes from the CUDA library.  The oracle keeps its dequantised
matrices as float32, which is exact for every Q8_0 / Q4_0 value and for the
fp16 embedding, and widens them to float64 in every product.  A whole chain
takes several minutes per workload on 8 host cores and about 32 GB of memory.
"""

from __future__ import annotations

import dataclasses
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

# sequences of each workload whose chains are stored, and the steps whose logits are kept
SEQS = {"llama2_7b_q4": [0], "llama3_8b_q8_b16": [0, 15]}
LOGIT_STEPS = {"llama2_7b_q4": [0, 31, 63], "llama3_8b_q8_b16": [0, 31]}


def path_of(name: str) -> str:
    return os.path.join(HERE, f"fullsize_{name}.npz")


class _Tensors:
    """Tensor source for the oracle: each quantised matrix is drawn when first asked for and not kept (the
    oracle caches its dequantised copy); gains and the fp16 embedding are drawn once and kept."""

    def __init__(self, shape: synth.ModelShape):
        self.shape = shape
        self.small: dict[str, np.ndarray] = {}

    def __call__(self, name: str) -> np.ndarray:
        kind, _ = synth.gen.tensor_kind(self.shape, name)
        if kind in ("q8_0", "q4_0") and not (self.shape.tied and name == "token_embd.weight"):
            return synth.weight_tensor(self.shape, name)
        if name not in self.small:
            self.small[name] = synth.weight_tensor(self.shape, name)
        return self.small[name]


def make(name: str) -> str:
    wl = synth.workload(name)
    s = wl.shape
    seqs = SEQS[name]
    cfg = oracle.OracleConfig(**{f.name: getattr(s, f.name) for f in dataclasses.fields(oracle.OracleConfig)})
    model = oracle.OracleModel(cfg, _Tensors(s), cache_dequant=True, cache_dtype=np.float32)
    cache = oracle.OracleCache(cfg, wl.batch, wl.capacity)
    for b in seqs:
        for l in range(s.n_layers):
            k, v = synth.kv_prefill(wl, b, l)
            cache.fill(b, l, k, v)
    t0 = time.time()
    fed, logits = oracle.greedy(model, cache, wl.tokens0(), wl.positions0(), wl.steps, seqs=seqs)
    srt = np.sort(logits, axis=-1)
    top2 = srt[..., -1] - srt[..., -2]
    steps = LOGIT_STEPS[name]
    out = path_of(name)
    np.savez_compressed(out, seqs=np.array(seqs, np.int64), fed=fed.astype(np.int64),
                        logit_steps=np.array(steps, np.int64), logits=logits[steps].astype(np.float64),
                        top2=top2.astype(np.float64))
    print(f"{name}: {wl.steps} steps of sequences {seqs} in {time.time() - t0:.0f} s; "
          f"smallest top-2 gap {top2.min():.3e}; wrote {out}", flush=True)
    return out


if __name__ == "__main__":
    for n in (sys.argv[1:] or list(SEQS)):
        make(n)
