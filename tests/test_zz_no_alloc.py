"""GPU: er_matrix_gemv_noalloc, the GEMV whose scratch is an array compiled into the library.

It must give what er_matrix_gemv gives (the same kernel, only the scratch
differs), call after call, since every call reuses the same array.  The file
name sorts last so that the test also runs after everything else in a session.
"""

from __future__ import annotations

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def gemv_bound(w, x):
    """Element-wise error bound of either GEMV against the exact product: (blocks + 8) * 2^-23 * sum |w x|."""
    nb = w.shape[1] // 32
    return (nb + 8) * 2.0 ** -23 * (np.abs(x) @ np.abs(w).T)


@pytest.mark.parametrize("w_type", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols,batch", [(576, 576, 1), (1000, 1536, 5), (4096, 4096, 1), (49152, 576, 2)])
def test_noalloc_matches_gemv(w_type, rows, cols, batch):
    from block_quantized_token_gb300 import er
    import oracle

    rng = np.random.default_rng(rows + 3 * cols + batch)
    w = (0.02 * rng.standard_normal((rows, cols))).astype(np.float32)
    raw = synth.quantize(w, w_type)
    x = rng.standard_normal((batch, cols)).astype(np.float32)
    dev = torch.from_numpy(raw).cuda()
    m = er.er_matrix_create(er.DTYPES[w_type], rows, cols, dev.data_ptr())
    try:
        xd = torch.from_numpy(x).cuda()
        want = torch.empty((batch, rows), dtype=torch.float32, device="cuda")
        er.er_matrix_gemv(m, xd.data_ptr(), batch, want.data_ptr())
        torch.cuda.synchronize()
        want = want.cpu().numpy().astype(np.float64)
        tol = gemv_bound(oracle.dequant(raw, w_type, rows, cols), x.astype(np.float64))
        for _ in range(2):  # two calls in a row on the same shared array
            got = torch.full((batch, rows), float("nan"), dtype=torch.float32, device="cuda")
            er.er_matrix_gemv_noalloc(m, xd.data_ptr(), batch, got.data_ptr())
            torch.cuda.synchronize()
            diff = np.abs(got.cpu().numpy().astype(np.float64) - want)
            assert np.all(diff <= tol), float(np.max(diff - tol))
    finally:
        er.er_matrix_destroy(m)


def test_noalloc_rejects_oversize():
    """More row groups than the fixed array holds: ER_EINVAL before any launch."""
    from block_quantized_token_gb300 import er

    rows, cols = 16 * 16384 + 1, 32
    raw = synth.quantize(np.zeros((rows, cols), np.float32), "q8_0")
    dev = torch.from_numpy(raw).cuda()
    m = er.er_matrix_create(er.DTYPES["q8_0"], rows, cols, dev.data_ptr())
    try:
        xd = torch.zeros((1, cols), dtype=torch.float32, device="cuda")
        y = torch.empty((1, rows), dtype=torch.float32, device="cuda")
        with pytest.raises(er.ErError) as err:
            er.er_matrix_gemv_noalloc(m, xd.data_ptr(), 1, y.data_ptr())
        assert err.value.status == er.ER_EINVAL
    finally:
        er.er_matrix_destroy(m)
