"""Thin Python owners of er_model / er_kv handles, with torch as the device allocator.

Weights arrive as host arrays in GGUF layout (uint8 block bytes, float32 gains,
float16 embedding) keyed by GGUF tensor name; they are staged on the device,
handed to er_model_create (which repacks them into model-owned memory) and
released.  All compute happens in liber.so.
"""

from __future__ import annotations

import ctypes
from typing import Callable, Mapping

import numpy as np
import torch

from . import er

_LAYER_FIELDS = (("attn_norm", "attn_norm"), ("wq", "attn_q"), ("wk", "attn_k"), ("wv", "attn_v"),
                 ("wo", "attn_output"), ("ffn_norm", "ffn_norm"), ("w_gate", "ffn_gate"), ("w_up", "ffn_up"),
                 ("w_down", "ffn_down"))


KV_TYPES = {"f16": er.DTYPES["f16"], "q8_0": er.DTYPES["q8_0"]}  # er_kv_create_typed storage codes


def make_config(shape, max_batch: int = 1) -> er.er_config:
    """er_config from any object with the ModelShape fields."""
    return er.er_config(dim=shape.dim, n_layers=shape.n_layers, n_heads=shape.n_heads, n_kv_heads=shape.n_kv_heads,
                        head_dim=shape.head_dim, ffn_dim=shape.ffn_dim, vocab=shape.vocab,
                        rope_base=float(shape.rope_base), rms_eps=float(shape.rms_eps),
                        w_type=er.DTYPES[shape.w_type], tied=1 if shape.tied else 0, max_batch=max_batch)


def _to_device(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


class DecodeModel:
    """Owns an er_model built from host tensors (name -> array or a callable name -> array)."""

    def __init__(self, shape, tensors: Mapping[str, np.ndarray] | Callable[[str], np.ndarray],
                 max_batch: int = 1, device: str = "cuda"):
        get = tensors if callable(tensors) else tensors.__getitem__
        self.shape = shape
        self.device = torch.device(device)
        keep = []

        def dev(name):
            t = _to_device(get(name), self.device)
            keep.append(t)
            return t.data_ptr()

        layers = (er.er_layer_weights * shape.n_layers)()
        for l in range(shape.n_layers):
            for field, leaf in _LAYER_FIELDS:
                setattr(layers[l], field, dev(f"blk.{l}.{leaf}.weight"))
        w = er.er_weights(tok_embd=dev("token_embd.weight"), output_norm=dev("output_norm.weight"),
                          output=None if shape.tied else dev("output.weight"),
                          layers=ctypes.cast(layers, ctypes.POINTER(er.er_layer_weights)))
        self.cfg = make_config(shape, max_batch)
        stream = torch.cuda.current_stream(self.device).cuda_stream
        self.handle = er.er_model_create(self.cfg, w, stream)
        del keep

    @property
    def device_bytes(self) -> int:
        return er.er_model_device_bytes(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            er.er_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()


class DecodeState:
    """Owns an er_kv (KV cache + scratch of `batch` sequences) of a DecodeModel."""

    def __init__(self, model: DecodeModel, batch: int, capacity: int, kv_type: str = "f16"):
        """kv_type "f16" (fp16 rows) or "q8_0" (packed Q8_0 blocks, quantised as rows are written)."""
        self.model, self.batch, self.capacity = model, batch, capacity
        if kv_type not in KV_TYPES:
            raise ValueError(f"kv_type must be one of {sorted(KV_TYPES)}")
        self.kv_type = kv_type
        self.handle = er.er_kv_create_typed(model.handle, batch, capacity, KV_TYPES[kv_type])

    def write_rows(self, seq: int, layer: int, k_rows: np.ndarray | torch.Tensor, v_rows, start: int = 0,
                   stream: int | None = None) -> None:
        """Copy token-major fp16 rows [n, n_kv_heads*head_dim] into cache rows start..start+n-1."""
        dev = self.model.device
        k = k_rows if isinstance(k_rows, torch.Tensor) else _to_device(np.asarray(k_rows, np.float16), dev)
        v = v_rows if isinstance(v_rows, torch.Tensor) else _to_device(np.asarray(v_rows, np.float16), dev)
        k, v = k.contiguous(), v.contiguous()
        st = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream
        er.er_kv_write(self.handle, seq, layer, start, k.shape[0], k.data_ptr(), v.data_ptr(), st)
        torch.cuda.current_stream(dev).synchronize()

    def read_rows(self, seq: int, layer: int, start: int, n: int) -> tuple[torch.Tensor, torch.Tensor]:
        s = self.model.shape
        k = torch.empty((n, s.n_kv_heads * s.head_dim), dtype=torch.float16, device=self.model.device)
        v = torch.empty_like(k)
        st = torch.cuda.current_stream(self.model.device).cuda_stream
        er.er_kv_read(self.handle, seq, layer, start, n, k.data_ptr(), v.data_ptr(), st)
        torch.cuda.current_stream(self.model.device).synchronize()
        return k, v

    def read_blocks(self, seq: int, layer: int, start: int, n: int) -> tuple[np.ndarray, np.ndarray]:
        """Q8_0 cache rows start..start+n-1 as GGUF blocks: (d fp16, q int8) per side, shaped
        [n, n_kv_heads*head_dim/32] and [n, n_kv_heads*head_dim]."""
        s = self.model.shape
        nb = s.n_kv_heads * s.head_dim // 32
        k = torch.empty((n, nb, 34), dtype=torch.uint8, device=self.model.device)
        v = torch.empty_like(k)
        st = torch.cuda.current_stream(self.model.device).cuda_stream
        er.er_kv_read_blocks(self.handle, seq, layer, start, n, k.data_ptr(), v.data_ptr(), st)
        torch.cuda.current_stream(self.model.device).synchronize()
        out = []
        for t in (k, v):
            a = t.cpu().numpy()
            d = np.ascontiguousarray(a[:, :, :2]).view(np.float16).reshape(n, nb)
            q = np.ascontiguousarray(a[:, :, 2:]).view(np.int8).reshape(n, nb * 32)
            out += [d, q]
        return tuple(out)

    def prefill(self, seq: int, tokens: torch.Tensor, start: int, logits: torch.Tensor | None = None,
                stream: int | None = None) -> None:
        """Run the decoder over device int32 `tokens` of sequence `seq` at positions start.., writing the cache."""
        st = torch.cuda.current_stream(self.model.device).cuda_stream if stream is None else stream
        er.er_prefill(self.handle, seq, tokens.data_ptr() if tokens.numel() else None, int(tokens.numel()), start,
                      None if logits is None else logits.data_ptr(), st)

    def step(self, tokens: torch.Tensor, positions: torch.Tensor, logits: torch.Tensor | None,
             argmax: torch.Tensor | None, graph: bool = True, stream: int | None = None) -> None:
        st = torch.cuda.current_stream(self.model.device).cuda_stream if stream is None else stream
        fn = er.er_decode_step if graph else er.er_decode_step_eager
        fn(tokens.data_ptr(), positions.data_ptr(), self.handle, None if logits is None else logits.data_ptr(),
           None if argmax is None else argmax.data_ptr(), st)

    def set_schedule(self, schedule: int) -> None:
        er.er_kv_set_schedule(self.handle, schedule)

    def set_wide_gemv(self, variant: int) -> None:
        er.er_kv_set_wide_gemv(self.handle, variant)

    @property
    def schedule(self) -> int:
        return er.er_kv_get_schedule(self.handle)

    def device_error(self) -> tuple[int, int, int]:
        return er.er_get_device_error(self.handle)

    def close(self) -> None:
        if getattr(self, "handle", None):
            er.er_kv_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()
