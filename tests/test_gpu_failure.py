"""GPU: failure detection without a GPU fault, through the C ABI.

* A bounded wait that runs out: the persistent step's first grid barrier is told to wait for one more arrival
  than its grid supplies (a host argument), with the wait limit lowered to 5 ms.  The kernel returns, the
  give-up flag (bit 2) is reported, and the next normal step is clean and bit-identical to one before it.
* Allocation failure: the library's n-th device allocation is made to fail, for every n a model, a decode
  state and a stand-alone matrix make.  Each call returns ER_ENOMEM and frees everything it had taken.
* The recorded-graph cache stays bounded when a caller rotates buffers, and device memory stays flat.

These mirror the pages' command-buffer status and timeout checks ("llama.cpp Metal (MPS) End-to-End Inference
Path", step table) and their memory-budget refusal ("alpaca.swift", Highlights).
"""

from __future__ import annotations

import time

import numpy as np
import pytest

import synth
from helpers import gpu_model, gpu_state

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _er():
    from block_quantized_token_gb300 import er
    return er


def _step(state, wl, logits=None):
    dev = state.model.device
    t = torch.tensor(wl.tokens0(), dtype=torch.int32, device=dev)
    p = torch.tensor(wl.positions0(), dtype=torch.int32, device=dev)
    lg = torch.full((wl.batch, wl.shape.vocab), float("nan"), device=dev) if logits is None else logits
    am = torch.empty(wl.batch, dtype=torch.int32, device=dev)
    state.step(t, p, lg, am)
    return lg, am


def test_wait_gives_up_and_next_step_is_clean():
    er = _er()
    wl = synth.workload("tiny")
    model = gpu_model(wl.shape, synth.model_weights(wl.shape))
    state = gpu_state(model, wl)
    try:
        assert state.schedule == er.ER_SCHEDULE_PERSISTENT
        ref, ref_am = _step(state, wl)
        torch.cuda.synchronize()
        ref = ref.cpu().numpy()
        assert state.device_error()[1] == 0
        er.er_set_wait_limit_ns(5_000_000)
        er.er_kv_inject_wait_shortfall(state.handle, 1)
        try:
            t0 = time.perf_counter()
            _step(state, wl)
            torch.cuda.synchronize()  # every CTA returned
            elapsed = time.perf_counter() - t0
            st, code, _ = state.device_error()
            assert st == er.ER_EDEVICE and code & 4, (st, code)
            assert elapsed < 0.5, f"gave up after {elapsed:.3f} s with a 5 ms limit"
        finally:
            er.er_kv_inject_wait_shortfall(state.handle, 0)
            er.er_set_wait_limit_ns(0)
        got, am = _step(state, wl)
        torch.cuda.synchronize()
        st, code, nf = state.device_error()
        assert st == er.ER_OK and code == 0 and nf == 0
        np.testing.assert_array_equal(got.cpu().numpy(), ref)
        assert torch.equal(am, ref_am)
    finally:
        state.close()
        model.close()


def _count_allocs(fn):
    er = _er()
    before = er.er_debug_live_allocations()
    obj = fn()
    return obj, er.er_debug_live_allocations() - before


def test_allocation_failure_frees_everything():
    er = _er()
    from block_quantized_token_gb300 import runtime
    wl = synth.workload("tiny")
    weights = synth.model_weights(wl.shape)
    base = er.er_debug_live_allocations()
    model, n_model = _count_allocs(lambda: runtime.DecodeModel(wl.shape, weights))
    state, n_kv = _count_allocs(lambda: runtime.DecodeState(model, 1, wl.capacity))
    assert n_model > 5 and n_kv > 5
    state.close()
    assert er.er_debug_live_allocations() == base + n_model
    try:
        for n in range(n_kv):
            er.er_debug_fail_allocation(n)
            with pytest.raises(er.ErError) as e:
                runtime.DecodeState(model, 1, wl.capacity)
            er.er_debug_fail_allocation(-1)
            assert e.value.status == er.ER_ENOMEM, (n, e.value)
            assert er.er_debug_live_allocations() == base + n_model, f"decode state, allocation {n} leaked"
        model.close()
        assert er.er_debug_live_allocations() == base
        for n in range(n_model):
            er.er_debug_fail_allocation(n)
            with pytest.raises(er.ErError) as e:
                runtime.DecodeModel(wl.shape, weights)
            er.er_debug_fail_allocation(-1)
            assert e.value.status == er.ER_ENOMEM, (n, e.value)
            assert er.er_debug_live_allocations() == base, f"model, allocation {n} leaked"
        raw = synth.quantize(np.zeros((64, 64), np.float32), "q8_0")
        dev = torch.from_numpy(raw).cuda()
        for n in range(4):
            er.er_debug_fail_allocation(n)
            with pytest.raises(er.ErError) as e:
                er.er_matrix_create(er.ER_Q8_0, 64, 64, dev.data_ptr())
            er.er_debug_fail_allocation(-1)
            assert e.value.status == er.ER_ENOMEM
            assert er.er_debug_live_allocations() == base
        # the hook is off again: everything builds
        m = er.er_matrix_create(er.ER_Q8_0, 64, 64, dev.data_ptr())
        er.er_matrix_destroy(m)
        assert er.er_debug_live_allocations() == base
    finally:
        er.er_debug_fail_allocation(-1)
        model.close()


def test_graph_cache_is_bounded():
    er = _er()
    wl = synth.workload("tiny")
    model = gpu_model(wl.shape, synth.model_weights(wl.shape))
    state = gpu_state(model, wl)
    try:
        bufs = [torch.empty((1, wl.shape.vocab), device="cuda") for _ in range(40)]
        ref, _ = _step(state, wl, bufs[0])
        torch.cuda.synchronize()
        ref = ref.clone()
        for i in range(1, 9):
            _step(state, wl, bufs[i])
        torch.cuda.synchronize()
        assert er.er_kv_cached_graphs(state.handle) == 8
        free0 = torch.cuda.mem_get_info()[0]
        for i in range(9, 40):
            _step(state, wl, bufs[i])
            assert er.er_kv_cached_graphs(state.handle) == 8
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        assert free0 - free1 < (32 << 20), f"device memory fell by {(free0 - free1) >> 20} MiB"
        for b in bufs[1:]:
            assert torch.equal(b, ref)
        # the first pointer set was dropped long ago: recorded again, same result
        _step(state, wl, bufs[0])
        torch.cuda.synchronize()
        assert torch.equal(bufs[0], ref)
    finally:
        state.close()
        model.close()
