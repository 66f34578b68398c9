"""bench.py's oracle baseline: whole-model timing when it fits the budget, else the 1- and 2-layer extrapolation."""
import os
import sys

import pytest

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
import synth  # noqa: E402


def _fake_run(a, b, calls):
    """A model whose step costs a + b * layers seconds per sequence."""
    def run(wl, n_layers, steps, budget_s, seqs):
        calls.append(n_layers)
        per = (a + b * n_layers) * len(seqs)
        return per, steps
    return run


@pytest.mark.parametrize("budget", [1e6, 1.0])
def test_oracle_sample_rate(monkeypatch, budget):
    wl = synth.workload("smollm_q8")  # 30 layers
    a, b = 0.4, 0.05
    calls = []
    monkeypatch.setattr(bench, "_oracle_run", _fake_run(a, b, calls))
    rate, steps, info = bench.oracle_sample(wl, steps=8, budget_s=budget)
    assert rate == pytest.approx(1.0 / (a + b * wl.shape.n_layers), rel=1e-12)
    if budget > 100:  # the whole model fits: timed directly
        assert calls == [1, wl.shape.n_layers] and steps == 8 and "whole model" in info["how"]
    else:  # extrapolated from the model cut to 1 and 2 layers
        assert calls == [1, 1, 2] and steps == 4 and "extrapolated" in info["how"]
