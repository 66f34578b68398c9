"""GPU: er_matrix_gemv_noalloc, the GEMV whose scratch is an array compiled into the library.

It runs the same deterministic kernel as er_matrix_gemv with only the scratch moved, so its output must be
bit-identical to er_matrix_gemv's (which its own parity test bounds against the oracle), call after call, since
every call reuses the same array.  Alternating a 49152-row and a 576-row matrix checks that a call after one
with more row groups still starts from clean counters.  The file name sorts last so that the test also runs
after everything else in a session.
"""

from __future__ import annotations

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


class _Mat:
    def __init__(self, w_type, rows, cols, batch, seed):
        from block_quantized_token_gb300 import er
        self.er = er
        rng = np.random.default_rng(seed)
        w = (0.02 * rng.standard_normal((rows, cols))).astype(np.float32)
        self.raw = torch.from_numpy(synth.quantize(w, w_type)).cuda()
        self.h = er.er_matrix_create(er.DTYPES[w_type], rows, cols, self.raw.data_ptr())
        self.x = torch.from_numpy(rng.standard_normal((batch, cols)).astype(np.float32)).cuda()
        self.rows, self.batch = rows, batch
        self.want = torch.empty((batch, rows), dtype=torch.float32, device="cuda")
        er.er_matrix_gemv(self.h, self.x.data_ptr(), batch, self.want.data_ptr())

    def noalloc(self):
        got = torch.full((self.batch, self.rows), float("nan"), dtype=torch.float32, device="cuda")
        self.er.er_matrix_gemv_noalloc(self.h, self.x.data_ptr(), self.batch, got.data_ptr())
        st, code = self.er.er_matrix_gemv_noalloc_error()  # synchronises
        assert st == self.er.ER_OK and code == 0
        return got

    def close(self):
        self.er.er_matrix_destroy(self.h)


@pytest.mark.parametrize("w_type", ["q8_0", "q4_0"])
@pytest.mark.parametrize("rows,cols,batch", [(576, 576, 1), (1000, 1536, 5), (4096, 4096, 1), (49152, 576, 2)])
def test_noalloc_matches_gemv(w_type, rows, cols, batch):
    m = _Mat(w_type, rows, cols, batch, rows + 3 * cols + batch)
    try:
        for _ in range(2):  # two calls in a row on the same shared array
            assert torch.equal(m.noalloc(), m.want)
    finally:
        m.close()


@pytest.mark.parametrize("w_type", ["q8_0", "q4_0"])
def test_noalloc_alternating_shapes(w_type):
    """A large matrix (3072 row groups, cross-CTA sums) and a small one take turns on the shared array."""
    big = _Mat(w_type, 49152, 576, 3, 11)
    small = _Mat(w_type, 576, 576, 2, 12)
    try:
        for _ in range(3):
            assert torch.equal(big.noalloc(), big.want)
            assert torch.equal(small.noalloc(), small.want)
    finally:
        big.close()
        small.close()


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
