"""The C ABI without a GPU: every declared symbol is exported and bound; host-side checks."""

from __future__ import annotations

import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def er():
    from block_quantized_token_gb300 import build
    build.build()
    from block_quantized_token_gb300 import er as mod
    return mod


def declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^ER_API\s+[\w\s\*]*?\b(er_\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_step_api():
    names = declared_functions()
    for n in ("er_model_create", "er_kv_create", "er_decode_step"):
        assert n in names


def test_every_declared_symbol_is_exported(er):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(er.lib(), n), n
        assert n in er.EXPORTED, n
        assert callable(getattr(er, n)), n


def test_dtype_codes_match_gguf_table(er):
    # "EdgeRunner Core Architecture" section 1.3: float32 = 0, float16 = 1, q4_0 = 2, q8_0 = 8
    from test_oracle_pins import _golden_formats
    fmts, _ = _golden_formats()
    assert (er.ER_F32, er.ER_F16, er.ER_Q4_0, er.ER_Q8_0) == (fmts["f32"][0], fmts["f16"][0], fmts["q4_0"][0],
                                                              fmts["q8_0"][0])


def test_status_strings(er):
    assert er.er_status_str(er.ER_OK) == "ok"
    assert er.er_status_str(er.ER_EINVAL) == "invalid argument"
    assert er.er_status_str(99) == "unknown status"


def test_config_checks_need_no_gpu(er):
    import synth
    from block_quantized_token_gb300 import runtime
    shape = synth.workload("tiny").shape
    cases = [("head_dim", 96, er.ER_EUNSUPPORTED), ("n_kv_heads", 4, er.ER_EINVAL), ("max_batch", 0, er.ER_EINVAL),
             ("dim", 560, er.ER_EINVAL), ("w_type", er.ER_F16, er.ER_EINVAL), ("vocab", 0, er.ER_EINVAL),
             ("tied", 2, er.ER_EINVAL), ("rope_base", -1.0, er.ER_EINVAL)]
    for field, val, status in cases:
        cfg = runtime.make_config(shape)
        setattr(cfg, field, val)
        with pytest.raises(er.ErError) as e:
            er.er_model_create(cfg, er.er_weights(), 0)
        assert e.value.status == status, (field, str(e.value))
        assert er.er_last_error()


def test_null_arguments_rejected(er):
    with pytest.raises(er.ErError) as e:
        er.er_decode_step(0, 0, 0, None, None, 0)
    assert e.value.status == er.ER_EINVAL
    with pytest.raises(er.ErError) as e:
        er.er_positions_increment(0, 1, 0)
    assert e.value.status == er.ER_EINVAL
    with pytest.raises(er.ErError) as e:
        er.er_matrix_create(er.ER_Q8_0, 16, 48, 1234, 0)
    assert e.value.status == er.ER_EINVAL
    with pytest.raises(er.ErError) as e:
        er.er_kv_create(0, 1, 16)
    assert e.value.status == er.ER_EINVAL
    with pytest.raises(er.ErError) as e:
        er.er_kv_set_wide_gemv(0, er.ER_WIDE_TCGEN05)
    assert e.value.status == er.ER_EINVAL
    with pytest.raises(er.ErError) as e:
        er.er_kv_create_typed(0, 1, 16, er.ER_Q8_0)
    assert e.value.status == er.ER_EINVAL
    with pytest.raises(er.ErError) as e:
        er.er_kv_read_blocks(0, 0, 0, 0, 1, 0, 0, 0)
    assert e.value.status == er.ER_EINVAL
    assert er.er_kv_type(None) == -1
    with pytest.raises(er.ErError) as e:
        er.er_prefill(0, 0, 0, 1, 0, None, 0)
    assert e.value.status == er.ER_EINVAL
