// Block-quantized GEMV core shared by the stand-alone GEMV kernel and the
// persistent decode-step kernel: the operand prologue (RMSNorm statistics,
// power-of-two rescale, hi/lo fp16 split into MMA B fragments), the per-unit
// tensor-core dot products, the consumption of a warp's weight ring, the
// CTA-level and grid-level sums of shared row groups, and the fused epilogues.
//
// Work split (two-level "stream-K"): a matrix is a list of U = R * UPR units
// (16 rows x 64 columns, contiguous in memory).  CTA c of the C CTAs working on
// the matrix takes the contiguous range [c U / C, (c+1) U / C) and splits it
// evenly over its warps, so every warp streams the same number of bytes
// whatever the matrix shape.  A row group inside one warp's range is finished
// by that warp; one shared by warps of a CTA is summed in shared memory in warp
// order; one shared by CTAs (at most the first and last of each CTA) is
// finished by the last CTA to arrive (an acquire-release counter), which sums
// the CTAs' partials in CTA order.  The result does not depend on timing.
//
// Dot products: the unit's int8 / int4 values are turned into exact fp16 in
// registers and multiplied on the tensor cores (mma m16n8k16, fp32 accumulate)
// with the activations split as x = hi + lo (two fp16 columns per batch
// column, |x - hi - lo| <= 2^-22 |x|), each 32-element block of x rescaled by
// its own power of two 2^e so its largest element lies in [2^14, 2^15); one MMA
// pair per block, whose fp32 sum is multiplied by d * 2^-e (d the weight
// block's fp16 scale).  RMSNorm's 1/rms is a per-column factor applied in the
// epilogue, so the operand needs no reduction over the whole vector.  The
// tensor cores here are a way to keep the per-weight instruction count below
// the HBM byte rate, not a contraction in their own right: the GEMV is bound
// by HBM bandwidth.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "layout.cuh"

namespace er {

constexpr int GV_WARPS = 16;
constexpr int GV_SLOTS = 3;
constexpr int GV_MAXB = 4;

template <int QT>
struct GvCfg {
    static constexpr int UB = QTraits<QT>::unit_bytes;
    static constexpr int QB = QTraits<QT>::quant_bytes;
    static constexpr int SU = QT == Q8_0 ? 2 : 4;  // units per ring slot
    static constexpr int SLOT = SU * UB;            // 2176 / 2304 bytes
    static constexpr int RING = GV_WARPS * GV_SLOTS * SLOT;
};

__host__ __device__ inline int gv_nbp(int K) { return ((K / 32) + 1) & ~1; }
// operand: B fragments [kb][g < 2B][t] x 16 bytes, then block factors [kb/2][b][2] fp32
__host__ __device__ inline size_t gv_xs_bytes(int K, int B) { return (size_t)gv_nbp(K) * B * 132; }

// CTAs working on a matrix: one per row group when there are no more row
// groups than CTAs and rows are short (no cross-CTA sums); otherwise all.
__host__ __device__ inline int gv_ctas(int R, int UPR, int max_ctas) {
    if (R <= max_ctas && UPR <= 32) return R;
    long long U = (long long)R * UPR;
    return (int)(U < max_ctas ? U : max_ctas);
}

// Shared-memory scratch of one GEMV pass (the operand area xs follows it).
struct GvScratch {
    float *fac;    // [16]: fac[8] = abort flag
    float *red;    // [GV_WARPS][GV_MAXB][2]: per-warp sum of squares of x
    float *wpart;  // [GV_WARPS][2 slots][64]: partial sums of shared row groups
    int *wrg;      // [GV_WARPS][2]: their row groups (-1: none)
    uint8_t *xs;   // operand (gv_xs_bytes)
};
constexpr int GV_SCRATCH_BYTES = 64 + 512 + GV_WARPS * 2 * 64 * 4 + 128;

__device__ inline GvScratch gv_scratch(uint8_t *base) {
    GvScratch s;
    s.fac = reinterpret_cast<float *>(base);
    s.red = reinterpret_cast<float *>(base + 64);
    s.wpart = reinterpret_cast<float *>(base + 64 + 512);
    s.wrg = reinterpret_cast<int *>(base + 64 + 512 + GV_WARPS * 2 * 64 * 4);
    s.xs = base + GV_SCRATCH_BYTES;
    return s;
}

// This CTA's and this warp's unit ranges of a matrix (empty when idle).  With
// `aligned`, CTAs take whole row groups (C = min(R, max_ctas) CTAs, R/C or
// R/C + 1 row groups each): no row group is shared by CTAs, at the price of
// at most one row group of imbalance.
// Unit indices are 32-bit: the launchers require R * UPR * max_ctas < 2^31.
struct GvRange {
    int ca, cb, wa, wb;  // CTA range, warp range
    int n, nw;           // CTA units, working warps
    int rgf, j0;         // row group of unit wa, and wa's position in it
    bool cta_active, working;
};

__host__ __device__ inline bool gv_index_ok(long long R, long long UPR, long long max_ctas) {
    return R * UPR * (max_ctas + 1) < (1ll << 31);
}

__device__ inline GvRange gv_range(int R, int UPR, int cta, int max_ctas, int warp, bool aligned = false) {
    GvRange r;
    const int U = R * UPR;
    const int nC = aligned ? (R < max_ctas ? R : max_ctas) : gv_ctas(R, UPR, max_ctas);
    r.cta_active = cta < nC;
    if (!r.cta_active) {
        r.ca = r.cb = r.wa = r.wb = U;
        r.n = r.nw = 0;
        r.rgf = R;
        r.j0 = 0;
        r.working = false;
        return r;
    }
    if (aligned) {
        r.ca = cta * R / nC * UPR;
        r.cb = (cta + 1) * R / nC * UPR;
    } else {
        r.ca = (int)((long long)cta * U / nC);
        r.cb = (int)((long long)(cta + 1) * U / nC);
    }
    r.n = r.cb - r.ca;
    r.nw = r.n < GV_WARPS ? r.n : GV_WARPS;
    r.working = warp < r.nw;
    r.wa = r.working ? r.ca + warp * r.n / r.nw : r.cb;
    r.wb = r.working ? r.ca + (warp + 1) * r.n / r.nw : r.cb;
    r.rgf = r.wa / UPR;
    r.j0 = r.wa - r.rgf * UPR;
    return r;
}

// Value of element (row, col) of an IDENT-mapped repacked matrix, decoded with
// the same register conversions the GEMV uses.
__device__ inline float repacked_value(const uint8_t *W, int qt, int UPR, int row, int col) {
    int rg = row >> 4, r = row & 15;
    int unit = col >> 6, c = col & 63;
    const uint8_t *ub = W + ((size_t)rg * UPR + unit) * unit_bytes_of(qt);
    FragPos p = frag_pos(r, c);
    __half dh = *reinterpret_cast<const __half *>(ub + scale_offset(qt, r, p.b));
    uint32_t h2;
    if (qt == Q8_0) {
        int off = q8_byte_offset(p);
        uint32_t w = *reinterpret_cast<const uint32_t *>(ub + (off & ~3));
        uint32_t lo, hi;
        q8_word_to_h2(w, lo, hi);
        h2 = (off & 2) ? hi : lo;
        return __half2float(dh) * ((off & 1) ? h2f_hi(h2) : h2f_lo(h2));
    }
    int word = 2 * p.b + p.h;
    uint32_t w = *reinterpret_cast<const uint32_t *>(ub + p.lane * 16 + word * 4);
    uint32_t rr[4];
    q4_word_to_h2(w, rr);
    h2 = rr[p.reg];
    return __half2float(dh) * (p.e ? h2f_hi(h2) : h2f_lo(h2));
}

// ---------------------------------------------------------------------------
// epilogues: lane (g, t) holds rows g and g+8 of row group rg for batch t.
// Activations written inside a kernel are read with ld.global.cg (L2), since
// another SM may have written them after this SM cached the line in L1.
// ---------------------------------------------------------------------------
template <int EPI>
__device__ inline void gv_epilogue(const GemvArgs &a, int rg, float v0, float v1, float f, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const bool bok = t < a.B;
    const int bt = a.b0 + t;  // column of the whole batch
    if (EPI == EPI_STORE || EPI == EPI_RESID) {
        if (!bok) return;
        v0 *= f;
        v1 *= f;
        int r0 = 16 * rg + g, r1 = r0 + 8;
        float *y = a.y + (size_t)bt * a.N;
        if (EPI == EPI_STORE) {
            if (r0 < a.N) y[r0] = v0;
            if (r1 < a.N) y[r1] = v1;
        } else {
            const int lr = rg - a.resid_rg0;
            if (a.resid_s && lr >= 0 && lr < a.resid_nrg) {  // rows staged at the start of the phase
                if (r0 < a.N) y[r0] = a.resid_s[(lr * 16 + g) * GV_MAXB + bt] + v0;
                if (r1 < a.N) y[r1] = a.resid_s[(lr * 16 + g + 8) * GV_MAXB + bt] + v1;
            } else {
                if (r0 < a.N) y[r0] = __ldcg(y + r0) + v0;
                if (r1 < a.N) y[r1] = __ldcg(y + r1) + v1;
            }
        }
    } else if (EPI == EPI_QKV) {
        if (!bok) return;
        v0 *= f;
        v1 *= f;
        const int pos = a.pos_s ? a.pos_s[bt] : a.positions[bt];
        if (pos < 0 || pos >= a.cap) return;
        const int sq = a.seqmap ? a.seqmap[bt] : bt;  // the column's sequence in the cache
        int r0 = 16 * rg + 2 * g;  // RoPE pair (r0, r0 + 1)
        if (r0 >= a.qd + 2 * a.kvd) return;
        if (r0 < a.qd + a.kvd) {  // q or k: rotate
            int base = r0 < a.qd ? r0 : r0 - a.qd;
            int dd = base % a.hd;
            const float2 cs = a.rope_s ? a.rope_s[bt * (a.hd / 2) + dd / 2] : a.rope[(size_t)pos * (a.hd / 2) + dd / 2];
            float o0 = v0 * cs.x - v1 * cs.y;
            float o1 = v1 * cs.x + v0 * cs.y;
            if (r0 < a.qd) {
                float2 *q = reinterpret_cast<float2 *>(a.q_out + (size_t)bt * a.qd + r0);
                *q = make_float2(o0, o1);
            } else {
                if (a.k_stage) {
                    *reinterpret_cast<float2 *>(a.k_stage + (size_t)bt * a.kvd + base) = make_float2(o0, o1);
                } else {
                    int kvh = base / a.hd;
                    size_t off = ((((size_t)sq * a.L + a.layer) * a.KV + kvh) * a.cap + pos) * a.hd + dd;
                    *reinterpret_cast<__half2 *>(a.kc + off) = __floats2half2_rn(o0, o1);
                }
            }
        } else {
            int base = r0 - a.qd - a.kvd;
            if (a.v_stage) {
                *reinterpret_cast<float2 *>(a.v_stage + (size_t)bt * a.kvd + base) = make_float2(v0, v1);
            } else {
                int kvh = base / a.hd, dd = base % a.hd;
                size_t off = ((((size_t)sq * a.L + a.layer) * a.KV + kvh) * a.cap + pos) * a.hd + dd;
                *reinterpret_cast<__half2 *>(a.vc + off) = __floats2half2_rn(v0, v1);
            }
        }
    } else if (EPI == EPI_SWIGLU) {
        if (!bok) return;
        int n = 8 * rg + g;
        if (n >= a.N) return;
        float gt = v0 * f, up = v1 * f;
        a.a_out[(size_t)bt * a.N + n] = gt / (1.f + expf(-gt)) * up;
    } else {  // EPI_LOGITS
        unsigned long long key = 0;
        if (bok) {
            v0 *= f;
            v1 *= f;
            int r0 = 16 * rg + g, r1 = r0 + 8;
            float *y = a.y ? a.y + (size_t)bt * a.N : nullptr;
            bool bad = false;
            if (r0 < a.N) {
                if (y) y[r0] = v0;
                bad |= !isfinite(v0);
                float kv = isnan(v0) ? -INFINITY : v0;
                key = ((unsigned long long)float_order_key(kv) << 32) | (0xFFFFFFFFu - (uint32_t)r0);
            }
            if (r1 < a.N) {
                if (y) y[r1] = v1;
                bad |= !isfinite(v1);
                float kv = isnan(v1) ? -INFINITY : v1;
                unsigned long long k1 = ((unsigned long long)float_order_key(kv) << 32) | (0xFFFFFFFFu - (uint32_t)r1);
                key = k1 > key ? k1 : key;
            }
            if (bad) atomicOr(a.flags, ER_FLAG_NONFINITE);
        }
        // max over the 8 lanes of the same batch column (lanes t, t+4, ..., t+28)
        for (int off = 4; off < 32; off <<= 1) {
            unsigned long long o = __shfl_xor_sync(0xffffffffu, key, off);
            key = o > key ? o : key;
        }
        if (bok && g == 0 && key) atomicMax(a.amax + bt, key);
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atom_add_acq_rel_gpu(a.done, 1) == a.R - 1;  // releases this warp's maxima
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();
        if (last) {
            if (lane < a.B) {
                unsigned long long k = atomicExch(a.amax + a.b0 + lane, 0ull);
                int idx = k ? (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu)) : 0;
                if (a.argmax_out) a.argmax_out[a.b0 + lane] = idx;
            }
            if (lane == 0) *a.done = 0;
        }
    }
}

// ---------------------------------------------------------------------------
// operand prologue (all threads; the caller synchronises the CTA after it).
// Four lanes per (block kb, column b): each loads 8 elements of x (and of the
// RMSNorm gain), the four agree on the block's largest |x * gain| and scale
// 2^e, and each writes its 8 hi/lo fp16 pairs straight into the MMA B-fragment
// layout [g = 2b (hi), 2b+1 (lo)][t][16 bytes] plus, once, the block factor
// 2^-e.  The per-warp sums of x^2 (for RMSNorm) go to red.
// ---------------------------------------------------------------------------
// Default source of the operand: 8 consecutive elements k.. of column b of x.
struct GvLoadX {
    __device__ void operator()(const GemvArgs &a, int b, int k, float (&v)[8]) const {
        const float4 *xp = reinterpret_cast<const float4 *>(a.x + (size_t)(a.b0 + b) * a.K + k);
        const float4 x0 = __ldcg(xp), x1 = __ldcg(xp + 1);
        v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
        v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
    }
};

template <class Load>
__device__ inline void gv_operand(const GemvArgs &a, const GvScratch &s, int tid, int nthreads, const Load &load) {
    const int K = a.K, B = a.B, nbp = gv_nbp(K), nb = K / 32;
    const int lane = tid & 31, warp = tid >> 5;
    float *sx = reinterpret_cast<float *>(s.xs + (size_t)nbp * B * 128);
    float ssq[GV_MAXB];
#pragma unroll
    for (int b = 0; b < GV_MAXB; ++b) ssq[b] = 0.f;
    const int nq = nbp * B * 4;
    for (int base = warp * 32; base < nq; base += nthreads) {  // warp-uniform trip count
        const int idx = base + lane;
        const bool ok = idx < nq;
        const int item = idx >> 2, q = idx & 3;
        const int kb = item / B, b = item - kb * B;
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 0.f;
        if (ok && kb < nb) {
            const int k = kb * 32 + q * 8;
            float4 g0 = make_float4(1.f, 1.f, 1.f, 1.f), g1 = g0;
            if (a.gain) {  // constant data: requested ahead of x
                const float4 *gp = reinterpret_cast<const float4 *>(a.gain + k);
                g0 = __ldg(gp);
                g1 = __ldg(gp + 1);
            }
            load(a, b, k, v);
            float sq = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) sq = fmaf(v[i], v[i], sq);
#pragma unroll
            for (int bb = 0; bb < GV_MAXB; ++bb)
                if (bb == b) ssq[bb] += sq;
            if (a.gain) {
                v[0] *= g0.x; v[1] *= g0.y; v[2] *= g0.z; v[3] *= g0.w;
                v[4] *= g1.x; v[5] *= g1.y; v[6] *= g1.z; v[7] *= g1.w;
            }
        }
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
        int e = 0;
        if (m > 0.f && isfinite(m)) {
            int E;
            frexpf(m, &E);
            e = 15 - E;  // block max * 2^e in [2^14, 2^15)
        }
        if (ok) {
            const float sc = ldexpf(1.f, e);
            uint8_t *area = s.xs + (size_t)item * 128;
#pragma unroll
            for (int p = 0; p < 4; ++p) {  // element pair (2j, 2j+1) of the block, j = 4q + p
                const int j = 4 * q + p;
                const int h = j >> 3, w8 = j & 7, reg = w8 >> 2, tt = w8 & 3;
                const float v0 = v[2 * p] * sc, v1 = v[2 * p + 1] * sc;
                const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                const __half l0 = __float2half_rn(v0 - __half2float(h0));
                const __half l1 = __float2half_rn(v1 - __half2float(h1));
                const int off = tt * 16 + (h * 2 + reg) * 4;
                *reinterpret_cast<__half2 *>(area + off) = __halves2half2(h0, h1);
                *reinterpret_cast<__half2 *>(area + 64 + off) = __halves2half2(l0, l1);
            }
            if (q == 0) sx[((kb >> 1) * B + b) * 2 + (kb & 1)] = ldexpf(1.f, -e);
        }
    }
    for (int b = 0; b < B; ++b) {
        float sm = ssq[0];
#pragma unroll
        for (int bb = 1; bb < GV_MAXB; ++bb)
            if (bb == b) sm = ssq[bb];
        for (int off = 16; off; off >>= 1) sm += __shfl_xor_sync(0xffffffffu, sm, off);
        if (lane == 0) s.red[(warp * GV_MAXB + b) * 2] = sm;
    }
}

__device__ inline void gv_operand(const GemvArgs &a, const GvScratch &s, int tid, int nthreads) {
    gv_operand(a, s, tid, nthreads, GvLoadX{});
}

// RMSNorm factor 1 / sqrt(mean(x^2) + eps) of column b (1 without a gain)
__device__ inline float gv_rstd(const GemvArgs &a, const GvScratch &s, int b, int nwarps) {
    if (!a.gain) return 1.f;
    float sm = 0.f;
    for (int w = 0; w < nwarps; ++w) sm += s.red[(w * GV_MAXB + b) * 2];
    return 1.f / sqrtf(sm / (float)a.K + a.eps);
}

// ---------------------------------------------------------------------------
// one unit (2 blocks x 16 rows) from shared memory at `ub`
// ---------------------------------------------------------------------------
template <int QT>
__device__ inline void gv_unit(uint32_t ub, uint32_t xa, uint32_t kb_stride, uint32_t sxa, bool has_b, int lane,
                               float &acc0, float &acc1) {
    const int g = lane >> 2;
    const uint2 bf = lds64(sxa);  // 2^-e of the unit's two activation blocks
    const float f0 = __uint_as_float(bf.x), f1 = __uint_as_float(bf.y);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = make_uint4(0, 0, 0, 0);
    if (has_b) {
        xb0 = lds128(xa);
        xb1 = lds128(xa + kb_stride);
    }
    const uint2 sc = lds64(ub + GvCfg<QT>::QB + g * 8);
    float c[4];
    uint32_t fa[4];
    if (QT == Q8_0) {
        const uint4 q0 = lds128(ub + lane * 16);
        const uint4 q1 = lds128(ub + 512 + lane * 16);
        q8_word_to_h2(q0.x, fa[0], fa[1]);
        q8_word_to_h2(q0.y, fa[2], fa[3]);
        mma_16816(c, fa, xb0.x, xb0.y, zero4);
        q8_word_to_h2(q0.z, fa[0], fa[1]);
        q8_word_to_h2(q0.w, fa[2], fa[3]);
        mma_16816(c, fa, xb0.z, xb0.w, c);
        acc0 = fmaf(h2f_lo(sc.x) * f0, c[0] + c[1], acc0);
        acc1 = fmaf(h2f_hi(sc.x) * f0, c[2] + c[3], acc1);
        q8_word_to_h2(q1.x, fa[0], fa[1]);
        q8_word_to_h2(q1.y, fa[2], fa[3]);
        mma_16816(c, fa, xb1.x, xb1.y, zero4);
        q8_word_to_h2(q1.z, fa[0], fa[1]);
        q8_word_to_h2(q1.w, fa[2], fa[3]);
        mma_16816(c, fa, xb1.z, xb1.w, c);
        acc0 = fmaf(h2f_lo(sc.y) * f1, c[0] + c[1], acc0);
        acc1 = fmaf(h2f_hi(sc.y) * f1, c[2] + c[3], acc1);
    } else {
        const uint4 q = lds128(ub + lane * 16);
        q4_word_to_h2(q.x, fa);
        mma_16816(c, fa, xb0.x, xb0.y, zero4);
        q4_word_to_h2(q.y, fa);
        mma_16816(c, fa, xb0.z, xb0.w, c);
        acc0 = fmaf(h2f_lo(sc.x) * f0, c[0] + c[1], acc0);
        acc1 = fmaf(h2f_hi(sc.x) * f0, c[2] + c[3], acc1);
        q4_word_to_h2(q.z, fa);
        mma_16816(c, fa, xb1.x, xb1.y, zero4);
        q4_word_to_h2(q.w, fa);
        mma_16816(c, fa, xb1.z, xb1.w, c);
        acc0 = fmaf(h2f_lo(sc.y) * f1, c[0] + c[1], acc0);
        acc1 = fmaf(h2f_hi(sc.y) * f1, c[2] + c[3], acc1);
    }
}

// ---------------------------------------------------------------------------
// Consume this warp's units [r.wa, r.wb) from its ring: global ring slots
// k0, k0+1, ... (slot k % GV_SLOTS, phase parity (k / GV_SLOTS) & 1).  After
// each slot, refill(k) lets lane 0 request the warp's next slot.  Row groups the
// warp covers completely are finished here; partial ones go to s.wpart/s.wrg
// (which the caller reset to -1 before).  Returns the number of slots consumed,
// or -1 after a wait that gave up (flag set).
// ---------------------------------------------------------------------------
template <int QT, int EPI, class Refill>
__device__ inline int gv_consume(const GemvArgs &a, const GvScratch &s, const GvRange &r, uint8_t *ring,
                                 uint64_t *wbar, unsigned k0, Refill refill, int lane, int warp) {
    using C = GvCfg<QT>;
    const int UPR = a.UPR;
    const int g = lane >> 2, t = lane & 3;
    const int nunits = r.wb - r.wa;
    const int nslots = (nunits + C::SU - 1) / C::SU;
    if (nslots == 0) return 0;
    const bool has_b = g < 2 * a.B;
    const uint32_t xs_lane = smem_u32(s.xs) + (uint32_t)((g * 4 + t) * 16);
    const uint32_t kb_stride = (uint32_t)(2 * a.B * 64);
    const int tb = t < a.B ? t : a.B - 1;  // lanes past the batch read column B-1 (results unused)
    const uint32_t sx_lane = smem_u32(s.xs) + (uint32_t)(gv_nbp(a.K) * a.B * 128 + tb * 8);
    const uint32_t sx_stride = (uint32_t)(a.B * 8);  // per unit
    const float f = gv_rstd(a, s, tb, GV_WARPS);
    const int rg_first = r.rgf;

    auto leave = [&](int rgf, float v0, float v1) {
        const int r_lo = rgf * UPR, r_hi = r_lo + UPR;
        if (r_lo >= r.wa && r_hi <= r.wb) {
            gv_epilogue<EPI>(a, rgf, v0, v1, f, lane);
            return;
        }
        const int slot = (rgf == rg_first) ? 0 : 1;
        *reinterpret_cast<float2 *>(s.wpart + (warp * 2 + slot) * 64 + lane * 2) = make_float2(v0, v1);
        if (lane == 0) s.wrg[warp * 2 + slot] = rgf;
    };

    float acc0 = 0.f, acc1 = 0.f, accb0 = 0.f, accb1 = 0.f;
    int rg = rg_first;
    int j = r.j0;
    for (int k = 0; k < nslots; ++k) {
        const unsigned kg = k0 + (unsigned)k;
        const unsigned sidx = kg % GV_SLOTS;
        if (!mbar_wait(wbar + sidx, (kg / GV_SLOTS) & 1u)) {
            if (lane == 0) atomicOr(a.flags, ER_FLAG_WAIT);
            return -1;
        }
        const int cnt = min(C::SU, nunits - k * C::SU);
        const uint32_t slot_base = smem_u32(ring + sidx * C::SLOT);
        for (int i = 0; i < cnt;) {
            if (j == UPR) {
                leave(rg, acc0 + accb0, acc1 + accb1);
                acc0 = acc1 = accb0 = accb1 = 0.f;
                ++rg;
                j = 0;
            }
            const uint32_t xa = xs_lane + (uint32_t)(2 * j) * kb_stride;
            const uint32_t sxa = sx_lane + (uint32_t)j * sx_stride;
            if (i + 1 < cnt && j + 1 < UPR) {  // two independent units in flight
                gv_unit<QT>(slot_base + i * C::UB, xa, kb_stride, sxa, has_b, lane, acc0, acc1);
                gv_unit<QT>(slot_base + (i + 1) * C::UB, xa + 2 * kb_stride, kb_stride, sxa + sx_stride, has_b, lane,
                            accb0, accb1);
                i += 2;
                j += 2;
            } else {
                gv_unit<QT>(slot_base + i * C::UB, xa, kb_stride, sxa, has_b, lane, acc0, acc1);
                i += 1;
                j += 1;
            }
        }
        __syncwarp();
        refill(kg);
    }
    leave(rg, acc0 + accb0, acc1 + accb1);
    return nslots;
}

// ---------------------------------------------------------------------------
// After gv_consume and a CTA barrier: row groups shared by warps of this CTA
// (the lowest warp sums them in warp order), then those shared by CTAs (the
// last CTA to arrive sums them in CTA order).
// ---------------------------------------------------------------------------
template <int EPI>
__device__ inline void gv_finish_shared(const GemvArgs &a, const GvScratch &s, const GvRange &r, int cta,
                                        int max_ctas, int lane, int warp) {
    if (!r.working) return;
    const int UPR = a.UPR;
    const int U = a.R * UPR;
    const int nC = gv_ctas(a.R, UPR, max_ctas);
    const int cfirst = r.ca / UPR;
    const int t = lane & 3;
    const float f = gv_rstd(a, s, t < a.B ? t : a.B - 1, GV_WARPS);
    for (int slot = 0; slot < 2; ++slot) {
        const int rgf = s.wrg[warp * 2 + slot];
        if (rgf < 0) continue;
        const int r_lo = rgf * UPR, r_hi = r_lo + UPR;
        const int lo_local = (r_lo > r.ca ? r_lo : r.ca) - r.ca;
        const int hi_local = (r_hi < r.cb ? r_hi : r.cb) - r.ca;
        const int w_first = ((lo_local + 1) * r.nw - 1) / r.n;
        if (w_first != warp) continue;
        const int w_last = (hi_local * r.nw - 1) / r.n;
        float2 v = *reinterpret_cast<const float2 *>(s.wpart + (warp * 2 + slot) * 64 + lane * 2);
        for (int w = warp + 1; w <= w_last; ++w) {
            float2 o = *reinterpret_cast<const float2 *>(s.wpart + (w * 2) * 64 + lane * 2);
            v.x += o.x;
            v.y += o.y;
        }
        if (r_lo >= r.ca && r_hi <= r.cb) {
            gv_epilogue<EPI>(a, rgf, v.x, v.y, f, lane);
            continue;
        }
        const int cslot = (rgf == cfirst) ? 0 : 1;
        *reinterpret_cast<float2 *>(a.part + ((size_t)cta * 2 + cslot) * 64 + lane * 2) = v;
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atom_add_acq_rel_gpu(a.cnt + rgf, 1);  // releases the partial
        old = __shfl_sync(0xffffffffu, old, 0);
        __syncwarp();
        const int c_first = ((r_lo + 1) * nC - 1) / U, c_last = (r_hi * nC - 1) / U;
        if (old == (int)(c_last - c_first)) {  // the acquire above orders these loads after every partial
            float s0 = 0.f, s1 = 0.f;
            for (int c = c_first; c <= c_last; ++c) {
                const int sl = ((c * U / nC) / UPR == rgf) ? 0 : 1;
                const float *q = a.part + ((size_t)c * 2 + sl) * 64 + lane * 2;
                s0 += __ldcg(q);
                s1 += __ldcg(q + 1);
            }
            gv_epilogue<EPI>(a, rgf, s0, s1, f, lane);
            if (lane == 0) a.cnt[rgf] = 0;
        }
    }
}

}  // namespace er
