"""Glue between the seeded generator and the oracle (tests only)."""

from __future__ import annotations

import dataclasses

import numpy as np

import oracle
import synth


def oracle_config(shape: synth.ModelShape) -> oracle.OracleConfig:
    return oracle.OracleConfig(**{f.name: getattr(shape, f.name) for f in dataclasses.fields(oracle.OracleConfig)})


def oracle_model(shape: synth.ModelShape, weights=None, cache_dequant=True) -> oracle.OracleModel:
    if weights is None:
        weights = synth.gen.model_weights(shape)
    return oracle.OracleModel(oracle_config(shape), weights, cache_dequant=cache_dequant)


def oracle_cache(wl: synth.Workload, seqs=None, kv_type: str = "f16") -> oracle.OracleCache:
    cfg = oracle_config(wl.shape)
    cache = oracle.OracleCache(cfg, wl.batch, wl.capacity, kv_type=kv_type)
    for b in (range(wl.batch) if seqs is None else seqs):
        for l in range(wl.shape.n_layers):
            k, v = synth.kv_prefill(wl, b, l)
            cache.fill(b, l, k, v)
    return cache


TINY = synth.ModelShape(n_layers=2, dim=64, n_heads=4, n_kv_heads=2, head_dim=16, ffn_dim=96, vocab=128,
                        rope_base=10000.0, rms_eps=1e-5, w_type="q8_0", tied=False)


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# ------------------------------------------------------------------------------------------
# GPU side (imports the CUDA binding lazily; only GPU tests call these)
# ------------------------------------------------------------------------------------------
def gpu_model(shape, weights, max_batch=1):
    from block_quantized_token_gb300 import runtime
    return runtime.DecodeModel(shape, weights, max_batch=max_batch)


def gpu_state(model, wl, seqs=None, kv_type: str = "f16"):
    from block_quantized_token_gb300 import runtime
    st = runtime.DecodeState(model, wl.batch, wl.capacity, kv_type=kv_type)
    for b in (range(wl.batch) if seqs is None else seqs):
        for l in range(wl.shape.n_layers):
            k, v = synth.kv_prefill(wl, b, l)
            st.write_rows(b, l, k, v)
    return st


def gpu_chain(state, wl, steps, tokens0=None, positions0=None, graph=True):
    """Run `steps` greedy steps chained on the device; returns (tokens fed [steps, B], logits [steps, B, V])."""
    import torch
    dev = state.model.device
    tok = torch.tensor(wl.tokens0() if tokens0 is None else tokens0, dtype=torch.int32, device=dev)
    pos = torch.tensor(wl.positions0() if positions0 is None else positions0, dtype=torch.int32, device=dev)
    logits = torch.empty((wl.batch, wl.shape.vocab), dtype=torch.float32, device=dev)
    fed = torch.empty((steps, wl.batch), dtype=torch.int32, device=dev)
    hist = torch.empty((steps, wl.batch, wl.shape.vocab), dtype=torch.float32, device=dev)
    from block_quantized_token_gb300 import er
    stream = torch.cuda.current_stream(dev).cuda_stream
    for s in range(steps):
        fed[s].copy_(tok)
        state.step(tok, pos, logits, tok, graph=graph)
        hist[s].copy_(logits)
        er.er_positions_increment(pos.data_ptr(), wl.batch, stream)
    torch.cuda.synchronize()
    return fed.cpu().numpy(), hist.cpu().numpy().astype(np.float64)


def logits_close(got, want, max_abs=2e-3, rel=1e-4):
    """The logits gate: max |got - want| <= 2e-3 and ||got - want|| / ||want|| <= 1e-4 per row."""
    got = np.asarray(got, np.float64).reshape(-1, np.shape(want)[-1])
    want = np.asarray(want, np.float64).reshape(got.shape)
    for g, w in zip(got, want):
        e = np.abs(g - w).max()
        r = rel_l2(g, w)
        assert e <= max_abs and r <= rel, f"max abs {e:.3e} (<= {max_abs}), rel L2 {r:.3e} (<= {rel})"


def top2_gap(logits):
    s = np.sort(np.asarray(logits, np.float64))
    return float(s[-1] - s[-2])


# ------------------------------------------------------------------------------------------
# derived tolerance of the new layer-0 K/V cache rows
# ------------------------------------------------------------------------------------------
U32 = 2.0 ** -24  # unit roundoff of fp32


def layer0_kv_exact(model, shape, token: int, pos: int):
    """The layer-0 K row (after RoPE) and V row that `token` at `pos` appends, in float64, with the element-wise
    bound on the GPU's fp32 values before any rounding to the cache type (layer0_kv_tolerance derives it).
    Returns (k, v, delta_k, delta_v), each [n_kv_heads * hd]."""
    s = shape
    x = model.embedding_rows([token])[0]
    g = model.gain("blk.0.attn_norm.weight")
    K = s.dim
    f = 1.0 / np.sqrt(np.mean(x * x) + s.rms_eps)
    u = x * g

    def pre(name):
        w = model.matrix(name)
        y = f * (w.astype(np.float64) @ u)
        gb = (K // 32 + 9) * 2.0 ** -23 * (np.abs(w.astype(np.float64)) @ np.abs(u))
        return y, f * gb + np.abs(y) * ((K / 64 + 15) * U32 + 2 * U32)

    yk, dk = pre("blk.0.attn_k.weight")
    yv, dv = pre("blk.0.attn_v.weight")
    dpair = dk[0::2] + dk[1::2] + (np.abs(yk[0::2]) + np.abs(yk[1::2])) * 4 * U32
    kr = oracle.rope(yk.reshape(s.n_kv_heads, s.head_dim), pos, s.rope_base).reshape(-1)
    return kr, yv, np.repeat(dpair, 2), dv


def layer0_kv_tolerance(model, shape, token: int, pos: int):
    """Element-wise bound on |GPU fp16 row - oracle fp16 row| for the K and V rows that layer 0 appends for
    `token` at `pos`, derived from the GPU's fp32 arithmetic.

    Layer 0's input x is the embedding row, exact on both sides.  Before the fp16 rounding the GPU's value of
    element i of y = f * (W (g * x)) (f = 1 / sqrt(mean(x^2) + eps), the RMSNorm factor) differs from the exact
    one by at most
      delta_i = f * (blocks + 9) * 2^-23 * sum_k |w_ik g_k x_k|   (the GEMV bound, with one more 2^-24 per
                                                                  term for the fp32 product g * x)
              + |y_i| * ((K/64 + 15) * 2^-24 + 2^-23)            (f: a sum of K positive squares at depth at
                                                                  most K/32 + 24, /K, + eps, sqrt and 1/x each
                                                                  rounded once; the product f * sum)
    and a rotated K pair (a, b) by at most delta_a + delta_b + (|y_a| + |y_b|) * 2^-22 (fp32 cos/sin and the
    rotation's two products and one sum).  Two values within delta round to fp16 values at most
    delta + one fp16 ulp (at the larger magnitude) apart.  Returns (tol_k, tol_v), each [n_kv_heads * hd].
    """
    kr, yv, dk_rot, dv = layer0_kv_exact(model, shape, token, pos)

    def tol(y, d):
        big = np.abs(y) + d
        return np.abs(np.spacing(big.astype(np.float16))).astype(np.float64) + d

    return tol(kr, dk_rot), tol(yv, dv)


def check_q8_blocks(d_got, q_got, x, delta):
    """GPU Q8_0 blocks (d [n/32] fp16, q [n] int8) of a row whose exact value is x (float64 [n]) and whose GPU
    fp32 value before quantising lies within delta of it.  The codes are the quantiser's (float32, see
    oracle.quantize_kv_q8_0) for some row within delta of x: d equals the oracle's d unless amax / 127 lies
    within reach of an fp16 rounding boundary, and each q equals the oracle's code unless x / d lies within
    reach of a half-integer, where it may be one off.  Returns the number of such one-off codes."""
    x = np.asarray(x, np.float64)
    d_ref, q_ref = oracle.quantize_kv_q8_0(x.astype(np.float32))
    d_got = np.asarray(d_got, np.float16).reshape(d_ref.shape)
    q_got = np.asarray(q_got, np.int8).reshape(q_ref.shape)
    delta = 2.0 * np.asarray(delta, np.float64) + 2.0 ** -22 * np.abs(x)  # margin for the float32 steps
    xb, db = x.reshape(-1, 32), delta.reshape(-1, 32)
    amax, amax_d = np.abs(xb).max(axis=1), db.max(axis=1)
    d_lo = ((amax - amax_d) / 127).astype(np.float32).astype(np.float16)
    d_hi = ((amax + amax_d) / 127).astype(np.float32).astype(np.float16)
    d_diff = d_got.reshape(-1) != d_ref.reshape(-1)
    assert not (d_diff & (d_lo == d_hi)).any(), "a block scale differs where no rounding boundary is near"
    assert (d_got.reshape(-1) >= d_lo).all() and (d_got.reshape(-1) <= d_hi).all(), "a block scale out of reach"
    same = ~d_diff
    qg, qr = q_got.reshape(-1, 32)[same].astype(np.int64), q_ref.reshape(-1, 32)[same].astype(np.int64)
    dd = d_ref.reshape(-1)[same].astype(np.float64)[:, None]
    r, rd = xb[same] / np.where(dd > 0, dd, 1), db[same] / np.where(dd > 0, dd, 1)
    frac = np.abs(np.abs(r) - np.floor(np.abs(r)) - 0.5)  # distance of |x / d| from a half-integer
    off = qg != qr
    assert (np.abs(qg - qr) <= 1).all(), "a code more than one step from the oracle's"
    assert not (off & (frac > rd)).any(), "a code differs where x / d is not near a half-integer"
    return int(off.sum())


# ------------------------------------------------------------------------------------------
# Q8_0 cache: the quantiser's legitimate one-step alternatives, and an oracle cache that takes one
# ------------------------------------------------------------------------------------------
def q8_codes(xb, d):
    """The quantiser's codes of one block for a given fp16 scale d (float32 quotient, half away from zero)."""
    d32 = np.float32(d)
    r = np.zeros_like(xb, dtype=np.float32) if d32 == 0 else (xb.astype(np.float32) / d32).astype(np.float64)
    return np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -127, 127).astype(np.int8)


def q8_alternatives(x, delta):
    """Each way the quantiser may code a block of the row x (float64 [n]) differently from the oracle for some
    row within delta of x: (block, d, q) with one code one step off where x / d lies within reach of a
    half-integer, or the whole block under the other fp16 scale where amax / 127 lies within reach of an
    fp16 rounding boundary.  Same margin as helpers.check_q8_blocks."""
    x = np.asarray(x, np.float64)
    d_ref, q_ref = oracle.quantize_kv_q8_0(x.astype(np.float32))
    delta = 2.0 * np.asarray(delta, np.float64) + 2.0 ** -22 * np.abs(x)
    out = []
    for blk in range(x.size // 32):
        xb, db, qb = x[32 * blk:32 * blk + 32], delta[32 * blk:32 * blk + 32], q_ref[32 * blk:32 * blk + 32]
        amax, amd = np.abs(xb).max(), db.max()
        for d2 in {np.float16(np.float32((amax - amd) / 127)), np.float16(np.float32((amax + amd) / 127))}:
            if d2 != d_ref[blk]:
                out.append((blk, d2, q8_codes(xb.astype(np.float32), d2)))
        d = float(d_ref[blk])
        if d == 0:
            continue
        r = np.abs(xb) / d
        near = np.abs(r - np.floor(r) - 0.5) <= db / d
        for e in np.nonzero(near)[0]:
            k = int(np.floor(r[e]))
            cur = abs(int(qb[e]))
            alt = min(k if cur == k + 1 else k + 1, 127)
            if alt != cur:
                q2 = qb.copy()
                q2[e] = np.int8(np.sign(xb[e]) * alt)
                out.append((blk, d_ref[blk], q2))
    return out


class OverrideCache(oracle.OracleCache):
    """The oracle's Q8_0 cache with one block of one new layer-0 row replaced after it is quantised."""

    def __init__(self, cfg, batch, capacity, override):
        super().__init__(cfg, batch, capacity, kv_type="q8_0")
        self.override = override  # (b, position, "k" | "v", block, d, q)

    def put(self, b, layer, rows, k, v):
        super().put(b, layer, rows, k, v)
        ob, op, side, blk, d2, q2 = self.override
        if layer != 0 or not isinstance(rows, (int, np.integer)) or (b, int(rows)) != (ob, op):
            return
        hd = self.cfg.head_dim
        h, j = divmod(blk, hd // 32)
        ds, qs, full = (self.kd, self.kq, self.k) if side == "k" else (self.vd, self.vq, self.v)
        ds[b][0][op][h, j] = d2
        qs[b][0][op][h, 32 * j:32 * j + 32] = q2
        full[b][0][op][h] = oracle.dequant_kv_q8_0(ds[b][0][op][h], qs[b][0][op][h]).astype(np.float32)
