"""GPU parity of the stand-alone kernels: dequantisation and block-quantized GEMV (C ABI)."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _er():
    from block_quantized_token_gb300 import er
    return er


def _mat(w_type, rows, cols, seed):
    rng = np.random.default_rng(seed)
    x = (0.02 * rng.standard_normal((rows, cols))).astype(np.float32)
    if seed % 3 == 0:  # include an all-zero block and a wide dynamic range
        x[0, :32] = 0
        x[-1, -32:] *= 1000
    return synth.quantize(x, w_type)


SHAPES = [(16, 64), (48, 96), (100, 160), (576, 576), (1536, 576), (576, 1536), (1000, 4096), (24, 32)]


@pytest.mark.parametrize("w_type", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_dequant_bit_exact(w_type, rows, cols):
    """Every element of the repacked matrix decodes to exactly d*q (the oracle's float64 value)."""
    er = _er()
    raw = _mat(w_type, rows, cols, rows + cols)
    dev = torch.from_numpy(raw).cuda()
    m = er.er_matrix_create(er.DTYPES[w_type], rows, cols, dev.data_ptr())
    try:
        out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
        er.er_matrix_dequant(m, out.data_ptr())
        torch.cuda.synchronize()
        want = oracle.dequant(raw, w_type, rows, cols)
        np.testing.assert_array_equal(out.cpu().numpy().astype(np.float64), want)
    finally:
        er.er_matrix_destroy(m)


def gemv_bound(w, x):
    """Element-wise error bound of the GEMV: (blocks + 8) * 2^-23 * sum_k |w_k x_k|.

    fp32 accumulation over K/32 block sums (each scaled once), the hi/lo fp16
    split of x (relative error <= 2^-22) and the tensor-core block sums
    (fp32 accumulate) each contribute at most a few units of 2^-24 per term.
    """
    nb = w.shape[1] // 32
    return (nb + 8) * 2.0 ** -23 * (np.abs(x) @ np.abs(w).T)


@pytest.mark.parametrize("w_type", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols,batch", [
    (576, 576, 1), (1536, 576, 1), (49152, 576, 1),      # the Q4_0 sweep of the 135M shape
    (4096, 4096, 1), (4096, 11008, 1), (100, 160, 3), (48, 96, 4), (1000, 1536, 5), (576, 576, 16),
    (24, 32, 2), (16, 64, 1)])
def test_gemv_parity(w_type, rows, cols, batch):
    er = _er()
    raw = _mat(w_type, rows, cols, 7 * rows + cols)
    rng = np.random.default_rng(rows * cols + batch)
    x = rng.standard_normal((batch, cols)).astype(np.float32)
    x[:, ::7] *= 30.0  # mixed magnitudes
    dev = torch.from_numpy(raw).cuda()
    m = er.er_matrix_create(er.DTYPES[w_type], rows, cols, dev.data_ptr())
    try:
        xd = torch.from_numpy(x).cuda()
        y = torch.empty((batch, rows), dtype=torch.float32, device="cuda")
        er.er_matrix_gemv(m, xd.data_ptr(), batch, y.data_ptr())
        y2 = torch.empty_like(y)
        er.er_matrix_gemv(m, xd.data_ptr(), batch, y2.data_ptr())
        torch.cuda.synchronize()
        w = oracle.dequant(raw, w_type, rows, cols)
        want = oracle.matvec(w, x.astype(np.float64))
        got = y.cpu().numpy().astype(np.float64)
        bound = gemv_bound(w, x.astype(np.float64))
        ratio = np.abs(got - want) / bound
        assert ratio.max() <= 1.0, f"worst error {ratio.max():.3f} of the bound"
        # deterministic: the same launch gives the same bits
        assert torch.equal(y, y2)
    finally:
        er.er_matrix_destroy(m)


# fp16 scale bit patterns at the format's edges: 1, -0.5, the largest finite (65504), the smallest normal
# (2^-14), the smallest subnormal (2^-24), -0, an inexact third, -3 (the same list the oracle's pins use)
EDGE_SCALES = [0x3C00, 0xB800, 0x7BFF, 0x0400, 0x0001, 0x8000, 0x3555, 0xC200]


def _edge_matrix(w_type, rows, cols):
    """GGUF bytes whose blocks cycle through EDGE_SCALES and, over every 8 consecutive blocks, through every
    int8 value (Q8_0) or every nibble in both positions of a byte (Q4_0)."""
    nb = rows * cols // 32
    bpb = {"q8_0": 34, "q4_0": 18}[w_type]
    out = np.zeros((nb, bpb), np.uint8)
    for i in range(nb):
        out[i, 0:2] = np.frombuffer(np.uint16(EDGE_SCALES[i % len(EDGE_SCALES)]).tobytes(), np.uint8)
        if w_type == "q8_0":
            out[i, 2:] = (np.arange(32) + 32 * (i % 8)) % 256  # int8 bytes 0..255 over 8 blocks
        else:
            j = np.arange(16)
            out[i, 2:] = ((j + i) % 16) | (((j + 3 * i + 5) % 16) << 4)
    return out.reshape(rows, cols // 32 * bpb)


@pytest.mark.parametrize("w_type", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols", [(48, 256), (40, 544)])
def test_edge_scales(w_type, rows, cols):
    """Blocks with subnormal, largest, zero-signed and negative fp16 scales and every quantised value: the
    dequantisation is bit-exact and the GEMV stays under its bound, on the GPU through the C ABI."""
    er = _er()
    raw = _edge_matrix(w_type, rows, cols)
    dev = torch.from_numpy(raw).cuda()
    m = er.er_matrix_create(er.DTYPES[w_type], rows, cols, dev.data_ptr())
    try:
        out = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
        er.er_matrix_dequant(m, out.data_ptr())
        w = oracle.dequant(raw, w_type, rows, cols)
        rng = np.random.default_rng(rows + cols)
        x = rng.standard_normal((3, cols)).astype(np.float32)
        xd = torch.from_numpy(x).cuda()
        y = torch.empty((3, rows), dtype=torch.float32, device="cuda")
        er.er_matrix_gemv(m, xd.data_ptr(), 3, y.data_ptr())
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        np.testing.assert_array_equal(got, w)
        assert np.array_equal(np.signbit(got), np.signbit(w)), "sign of zero differs"
        want = oracle.matvec(w, x.astype(np.float64))
        ratio = np.abs(y.cpu().numpy().astype(np.float64) - want) / gemv_bound(w, x.astype(np.float64))
        assert ratio.max() <= 1.0, f"worst error {ratio.max():.3f} of the bound"
    finally:
        er.er_matrix_destroy(m)


def test_matrix_create_rejects_bad_args():
    er = _er()
    dev = torch.zeros(34 * 4, dtype=torch.uint8, device="cuda")
    for args in [(er.ER_Q8_0, 0, 64), (er.ER_Q8_0, 4, 48), (5, 4, 64)]:
        with pytest.raises(er.ErError) as e:
            er.er_matrix_create(args[0], args[1], args[2], dev.data_ptr())
        assert e.value.status == er.ER_EINVAL
