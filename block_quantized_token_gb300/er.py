"""ctypes binding of liber.so: the same names as include/er.h, argument marshalling only.

Every function raises ErError when the C call returns a status other than
ER_OK.  Device pointers are plain integers (e.g. ``tensor.data_ptr()``) and
streams are ``cudaStream_t`` values as integers (e.g.
``torch.cuda.current_stream().cuda_stream``).  Importing this module loads the
library; it fails loudly when the library has not been built.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liber.so")

ER_OK, ER_EINVAL, ER_ENOMEM, ER_ECUDA, ER_EUNSUPPORTED, ER_EDEVICE = range(6)
ER_F32, ER_F16, ER_Q4_0, ER_Q8_0 = 0, 1, 2, 8
DTYPES = {"f32": ER_F32, "f16": ER_F16, "q4_0": ER_Q4_0, "q8_0": ER_Q8_0}
ER_SCHEDULE_AUTO, ER_SCHEDULE_PERSISTENT, ER_SCHEDULE_KERNELS = 0, 1, 2
ER_WIDE_AUTO, ER_WIDE_MMA_SYNC, ER_WIDE_TCGEN05 = 0, 1, 2
(ER_STAGE_EMBED, ER_STAGE_QKV, ER_STAGE_ATTN, ER_STAGE_WO, ER_STAGE_GATEUP, ER_STAGE_DOWN,
 ER_STAGE_HEAD) = range(7)


class ErError(RuntimeError):
    def __init__(self, msg: str, status: int):
        super().__init__(msg)
        self.status = status


class er_config(ctypes.Structure):
    _fields_ = [("dim", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn_dim", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rope_base", ctypes.c_double), ("rms_eps", ctypes.c_double),
                ("w_type", ctypes.c_int32), ("tied", ctypes.c_int32), ("max_batch", ctypes.c_int32)]


class er_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")]


class er_weights(ctypes.Structure):
    _fields_ = [("tok_embd", ctypes.c_void_p), ("output_norm", ctypes.c_void_p), ("output", ctypes.c_void_p),
                ("layers", ctypes.POINTER(er_layer_weights))]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with block_quantized_token_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_void_p
    sigs = {
        "er_model_create": (I32, [P(er_config), P(er_weights), VP, P(VP)]),
        "er_model_destroy": (None, [VP]),
        "er_model_device_bytes": (ctypes.c_size_t, [VP]),
        "er_kv_create": (I32, [VP, I32, I32, P(VP)]),
        "er_kv_create_typed": (I32, [VP, I32, I32, I32, P(VP)]),
        "er_kv_type": (I32, [VP]),
        "er_kv_read_blocks": (I32, [VP, I32, I32, I32, I32, VP, VP, VP]),
        "er_prefill": (I32, [VP, I32, VP, I32, I32, VP, VP]),
        "er_kv_destroy": (None, [VP]),
        "er_kv_layer_ptrs": (I32, [VP, I32, I32, P(VP), P(VP)]),
        "er_kv_write": (I32, [VP, I32, I32, I32, I32, VP, VP, VP]),
        "er_kv_read": (I32, [VP, I32, I32, I32, I32, VP, VP, VP]),
        "er_decode_step": (I32, [VP, VP, VP, VP, VP, VP]),
        "er_decode_step_eager": (I32, [VP, VP, VP, VP, VP, VP]),
        "er_positions_increment": (I32, [VP, I32, VP]),
        "er_kv_set_schedule": (I32, [VP, I32]),
        "er_kv_get_schedule": (I32, [VP]),
        "er_kv_set_wide_gemv": (I32, [VP, I32]),
        "er_kv_launches_per_step": (I32, [VP]),
        "er_get_device_error": (I32, [VP, P(I32), P(I32)]),
        "er_launch_stage": (I32, [VP, I32, I32, VP, VP, VP, VP, VP]),
        "er_matrix_create": (I32, [I32, I32, I32, VP, VP, P(VP)]),
        "er_matrix_destroy": (None, [VP]),
        "er_matrix_dequant": (I32, [VP, VP, VP]),
        "er_matrix_gemv": (I32, [VP, VP, I32, VP, VP]),
        "er_matrix_gemv_noalloc": (I32, [VP, VP, I32, VP, VP]),
        "er_matrix_gemv_noalloc_error": (I32, [P(I32)]),
        "er_kv_cached_graphs": (I32, [VP]),
        "er_kv_inject_wait_shortfall": (I32, [VP, I32]),
        "er_set_wait_limit_ns": (I32, [ctypes.c_uint64]),
        "er_debug_fail_allocation": (I32, [ctypes.c_int64]),
        "er_debug_live_allocations": (ctypes.c_int64, []),
        "er_gguf_open": (I32, [ctypes.c_char_p, P(VP)]),
        "er_gguf_close": (None, [VP]),
        "er_gguf_tensor_count": (ctypes.c_int64, [VP]),
        "er_gguf_tensor_info": (I32, [VP, ctypes.c_int64, P(ctypes.c_char_p), P(I32), P(I32),
                                      P(ctypes.c_int64), P(VP), P(ctypes.c_uint64)]),
        "er_gguf_find": (I32, [VP, ctypes.c_char_p, P(ctypes.c_int64)]),
        "er_gguf_config": (I32, [VP, I32, P(er_config)]),
        "er_model_create_from_gguf": (I32, [VP, I32, VP, P(VP)]),
        "er_status_str": (ctypes.c_char_p, [I32]),
        "er_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


_lib = _load()
EXPORTED = ("er_model_create", "er_model_destroy", "er_model_device_bytes", "er_kv_create", "er_kv_destroy",
            "er_kv_layer_ptrs", "er_kv_write", "er_kv_read", "er_decode_step", "er_decode_step_eager", "er_positions_increment",
            "er_kv_set_schedule", "er_kv_get_schedule", "er_kv_set_wide_gemv",
            "er_get_device_error", "er_launch_stage", "er_matrix_create", "er_matrix_destroy",
            "er_matrix_dequant", "er_matrix_gemv", "er_matrix_gemv_noalloc", "er_matrix_gemv_noalloc_error",
            "er_kv_launches_per_step", "er_kv_cached_graphs", "er_kv_inject_wait_shortfall", "er_set_wait_limit_ns",
            "er_debug_fail_allocation", "er_debug_live_allocations", "er_gguf_open", "er_gguf_close",
            "er_gguf_tensor_count", "er_gguf_tensor_info", "er_gguf_find", "er_gguf_config",
            "er_model_create_from_gguf", "er_kv_create_typed", "er_kv_type", "er_kv_read_blocks", "er_prefill", "er_status_str",
            "er_last_error")


def lib() -> ctypes.CDLL:
    return _lib


def _check(status: int, what: str) -> None:
    if status != ER_OK:
        raise ErError(f"{what}: {er_status_str(status)}: {er_last_error()}", status)


def er_status_str(status: int) -> str:
    return _lib.er_status_str(status).decode()


def er_last_error() -> str:
    return _lib.er_last_error().decode(errors="replace")


def er_model_create(cfg: er_config, weights: er_weights, stream: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(_lib.er_model_create(ctypes.byref(cfg), ctypes.byref(weights), stream, ctypes.byref(out)),
           "er_model_create")
    return out.value


def er_model_destroy(model: int) -> None:
    _lib.er_model_destroy(model)


def er_model_device_bytes(model: int) -> int:
    return _lib.er_model_device_bytes(model)


def er_kv_create(model: int, batch: int, capacity: int) -> int:
    out = ctypes.c_void_p()
    _check(_lib.er_kv_create(model, batch, capacity, ctypes.byref(out)), "er_kv_create")
    return out.value


def er_kv_create_typed(model: int, batch: int, capacity: int, kv_type: int) -> int:
    out = ctypes.c_void_p()
    _check(_lib.er_kv_create_typed(model, batch, capacity, kv_type, ctypes.byref(out)), "er_kv_create_typed")
    return out.value


def er_kv_type(kv: int | None) -> int:
    return _lib.er_kv_type(kv)


def er_kv_read_blocks(kv: int, seq: int, layer: int, start: int, n: int, k_blocks: int, v_blocks: int,
                      stream: int = 0) -> None:
    _check(_lib.er_kv_read_blocks(kv, seq, layer, start, n, k_blocks, v_blocks, stream), "er_kv_read_blocks")


def er_prefill(kv: int, seq: int, tokens: int | None, n: int, start: int, logits: int | None,
               stream: int = 0) -> None:
    _check(_lib.er_prefill(kv, seq, tokens, n, start, logits, stream), "er_prefill")


def er_kv_destroy(kv: int) -> None:
    _lib.er_kv_destroy(kv)


def er_kv_layer_ptrs(kv: int, seq: int, layer: int) -> tuple[int, int]:
    k, v = ctypes.c_void_p(), ctypes.c_void_p()
    _check(_lib.er_kv_layer_ptrs(kv, seq, layer, ctypes.byref(k), ctypes.byref(v)), "er_kv_layer_ptrs")
    return k.value, v.value


def er_kv_write(kv: int, seq: int, layer: int, start: int, n: int, k_rows: int, v_rows: int,
                stream: int = 0) -> None:
    _check(_lib.er_kv_write(kv, seq, layer, start, n, k_rows, v_rows, stream), "er_kv_write")


def er_kv_read(kv: int, seq: int, layer: int, start: int, n: int, k_rows: int, v_rows: int,
               stream: int = 0) -> None:
    _check(_lib.er_kv_read(kv, seq, layer, start, n, k_rows, v_rows, stream), "er_kv_read")


def er_decode_step(tokens: int, positions: int, kv: int, logits: int | None, argmax: int | None,
                   stream: int = 0) -> None:
    _check(_lib.er_decode_step(tokens, positions, kv, logits, argmax, stream), "er_decode_step")


def er_decode_step_eager(tokens: int, positions: int, kv: int, logits: int | None, argmax: int | None,
                         stream: int = 0) -> None:
    _check(_lib.er_decode_step_eager(tokens, positions, kv, logits, argmax, stream), "er_decode_step_eager")


def er_positions_increment(positions: int, batch: int, stream: int = 0) -> None:
    _check(_lib.er_positions_increment(positions, batch, stream), "er_positions_increment")


def er_kv_set_schedule(kv: int, schedule: int) -> None:
    _check(_lib.er_kv_set_schedule(kv, schedule), "er_kv_set_schedule")


def er_kv_set_wide_gemv(kv: int, variant: int) -> None:
    _check(_lib.er_kv_set_wide_gemv(kv, variant), "er_kv_set_wide_gemv")


def er_kv_get_schedule(kv: int) -> int:
    return _lib.er_kv_get_schedule(kv)


def er_kv_launches_per_step(kv: int) -> int:
    return int(_lib.er_kv_launches_per_step(kv))


def er_get_device_error(kv: int) -> tuple[int, int, int]:
    """Returns (status, code, non_finite) without raising on ER_EDEVICE."""
    code, nf = ctypes.c_int32(), ctypes.c_int32()
    st = _lib.er_get_device_error(kv, ctypes.byref(code), ctypes.byref(nf))
    if st not in (ER_OK, ER_EDEVICE):
        _check(st, "er_get_device_error")
    return st, code.value, nf.value


def er_launch_stage(kv: int, stage: int, layer: int, tokens: int, positions: int, logits: int | None,
                    argmax: int | None, stream: int = 0) -> None:
    _check(_lib.er_launch_stage(kv, stage, layer, tokens, positions, logits, argmax, stream), "er_launch_stage")


def er_matrix_create(w_type: int, rows: int, cols: int, blocks: int, stream: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(_lib.er_matrix_create(w_type, rows, cols, blocks, stream, ctypes.byref(out)), "er_matrix_create")
    return out.value


def er_matrix_destroy(mat: int) -> None:
    _lib.er_matrix_destroy(mat)


def er_matrix_dequant(mat: int, out: int, stream: int = 0) -> None:
    _check(_lib.er_matrix_dequant(mat, out, stream), "er_matrix_dequant")


def er_matrix_gemv(mat: int, x: int, batch: int, y: int, stream: int = 0) -> None:
    _check(_lib.er_matrix_gemv(mat, x, batch, y, stream), "er_matrix_gemv")


def er_matrix_gemv_noalloc(mat: int, x: int, batch: int, y: int, stream: int = 0) -> None:
    _check(_lib.er_matrix_gemv_noalloc(mat, x, batch, y, stream), "er_matrix_gemv_noalloc")


def er_matrix_gemv_noalloc_error() -> tuple[int, int]:
    """Returns (status, code) without raising on ER_EDEVICE."""
    code = ctypes.c_int32()
    st = _lib.er_matrix_gemv_noalloc_error(ctypes.byref(code))
    if st not in (ER_OK, ER_EDEVICE):
        _check(st, "er_matrix_gemv_noalloc_error")
    return st, code.value


def er_kv_cached_graphs(kv: int) -> int:
    return int(_lib.er_kv_cached_graphs(kv))


def er_kv_inject_wait_shortfall(kv: int, extra: int) -> None:
    _check(_lib.er_kv_inject_wait_shortfall(kv, extra), "er_kv_inject_wait_shortfall")


def er_set_wait_limit_ns(ns: int) -> None:
    _check(_lib.er_set_wait_limit_ns(ns), "er_set_wait_limit_ns")


def er_debug_fail_allocation(n: int) -> None:
    _check(_lib.er_debug_fail_allocation(n), "er_debug_fail_allocation")


def er_debug_live_allocations() -> int:
    return int(_lib.er_debug_live_allocations())


def er_gguf_open(path: str) -> int:
    out = ctypes.c_void_p()
    _check(_lib.er_gguf_open(os.fsencode(path), ctypes.byref(out)), "er_gguf_open")
    return out.value


def er_gguf_close(g: int) -> None:
    _lib.er_gguf_close(g)


def er_gguf_tensor_count(g: int) -> int:
    return int(_lib.er_gguf_tensor_count(g))


def er_gguf_tensor_info(g: int, i: int) -> tuple[str, int, list[int], int, int]:
    """(name, type, dims (innermost first, n_dims of them), host address of the data, bytes)."""
    name, typ, nd = ctypes.c_char_p(), ctypes.c_int32(), ctypes.c_int32()
    dims = (ctypes.c_int64 * 4)()
    data, nbytes = ctypes.c_void_p(), ctypes.c_uint64()
    _check(_lib.er_gguf_tensor_info(g, i, ctypes.byref(name), ctypes.byref(typ), ctypes.byref(nd), dims,
                                    ctypes.byref(data), ctypes.byref(nbytes)), "er_gguf_tensor_info")
    return name.value.decode(errors="replace"), typ.value, list(dims[:nd.value]), data.value or 0, nbytes.value


def er_gguf_find(g: int, name: str) -> int:
    idx = ctypes.c_int64()
    _check(_lib.er_gguf_find(g, name.encode(), ctypes.byref(idx)), "er_gguf_find")
    return idx.value


def er_gguf_config(g: int, max_batch: int = 1) -> er_config:
    cfg = er_config()
    _check(_lib.er_gguf_config(g, max_batch, ctypes.byref(cfg)), "er_gguf_config")
    return cfg


def er_model_create_from_gguf(g: int, max_batch: int = 1, stream: int = 0) -> int:
    out = ctypes.c_void_p()
    _check(_lib.er_model_create_from_gguf(g, max_batch, stream, ctypes.byref(out)), "er_model_create_from_gguf")
    return out.value
