// Persistent decode step: one cooperative grid, one CTA per SM, runs the whole
// step -- embedding, every layer's five phases, LM head and argmax -- with
// grid-wide barriers between phases instead of kernel launches.
//
// Why: at decode batch 1 each phase moves 0.3-50 MB, so a kernel per phase
// spends much of its life ramping up and draining.  Here the weights, which
// do not depend on the activations, stream continuously: every warp owns a
// ring of shared-memory slots that a bulk async copy refills as soon as a slot
// is consumed, walking the warp's units of every GEMV of the step in order
// (QKV, Wo, gate/up, down of each layer, then the head).  While a CTA waits at
// a barrier or runs attention, its rings already hold the next GEMV's first
// slots.
//
// Phases ("EdgeRunner Core Architecture" section 5.1, one token per sequence):
//   EMBED   x = token_embd[token]
//   QKV     RMSNorm + [Wq;Wk;Wv] + RoPE, q -> scratch, fp16 K/V -> cache row pos
//   ATT     GQA attention over cache rows 0..pos (rows split evenly over the
//           CTAs, then over their warps; a CTA merges its warps' softmax
//           states; heads split over CTAs leave one state per CTA)
//   WO      x += Wo o, the operand merging the CTAs' states of split heads
//   GATEUP  a = silu(Wgate h2) * (Wup h2), h2 = RMSNorm(x)
//   DOWN    x += Wdown a
//   HEAD    logits = Wout RMSNorm(x); argmax
// Every barrier wait is bounded (a second of %globaltimer by default); a wait
// that gives up sets a device flag and every CTA returns after draining its
// copies.
#pragma once

#include "gemv_core.cuh"

namespace er {

constexpr int MK_OFF_RING = 512;  // after the mbarriers
template <int QT>
constexpr int mk_off_scratch() { return MK_OFF_RING + GvCfg<QT>::RING; }

__host__ __device__ inline size_t mk_att_smem_bytes(int hd, int G);

// operand area: the largest GEMV operand or the attention phase's parked states
template <int QT>
__host__ __device__ inline size_t mk_smem_bytes(int max_k, int B, int hd, int G) {
    const size_t xs = gv_xs_bytes(max_k, B), att = mk_att_smem_bytes(hd, G);
    return (size_t)mk_off_scratch<QT>() + GV_SCRATCH_BYTES + (xs > att ? xs : att);
}

// Grid barrier number `gen` (1, 2, ...): every CTA adds 1 to *bar, then waits
// until *bar reaches gen * gridDim.x + extra (extra > 0 only when a test
// injects a shortfall: then no CTA can pass and every wait gives up).  Returns
// false (all threads) if the wait gave up or another CTA flagged an error.
__device__ inline bool mk_barrier(unsigned *bar, int *flags, unsigned gen, int *ok_smem, unsigned extra = 0) {
    __syncthreads();
    if (threadIdx.x == 0) {
        red_add_release_gpu(bar, 1);
        const unsigned target = gen * gridDim.x + extra;
        bool ok = true;
        if (ld_acquire_gpu(bar) < target) {
            const uint64_t t0 = globaltimer_ns();
            const unsigned long long lim = wait_limit_ns();
            for (uint32_t i = 1;; ++i) {
                if (ld_acquire_gpu(bar) >= target) break;
                if ((i & 31) == 0) {
                    if (*reinterpret_cast<volatile int *>(flags) & ER_FLAG_WAIT) {
                        ok = false;
                        break;
                    }
                    if (globaltimer_ns() - t0 > lim) {
                        atomicOr(flags, ER_FLAG_WAIT);
                        ok = false;
                        break;
                    }
                }
                if (i > 64) __nanosleep(32);
            }
        }
        if (ok && (*reinterpret_cast<volatile int *>(flags) & ER_FLAG_WAIT)) ok = false;
        *ok_smem = ok ? 1 : 0;
    }
    __syncthreads();
    return *ok_smem != 0;
}

// ---------------------------------------------------------------------------
// attention phase of layer l
//
// The rows of all (sequence, KV head) pairs, rows 0..pos each, form one list of
// NR rows.  CTA c of C takes the contiguous range [c NR / C, (c+1) NR / C)
// (at least MK_ATT_MIN_ROWS rows per CTA) and splits it evenly over its warps.
// A warp keeps, per query head of the group, the online-softmax state (max m,
// sum l, o = sum e^(s - m) v, scores in log2 units) of each head it covers.  A
// head one warp covers completely is finished by that warp.  Otherwise the
// warp parks its state in shared memory and the CTA merges its warps' states
// of the head (one thread per output element, warp order): a head inside the
// CTA is finished there; a head shared by CTAs leaves the CTA's merged state in
// global memory (slot 0: the CTA's first segment, slot 1: its last), and the
// Wo phase merges those states, in CTA order, while it builds its operand.
// ---------------------------------------------------------------------------
constexpr int MK_ATT_MIN_ROWS = 256;
constexpr int MK_RESID_RG = 4;  // row groups of residual rows a CTA stages in shared memory

// shared memory (it reuses the GEMV operand area): parked states [GV_WARPS][2][G (HD + 2)]
__host__ __device__ inline size_t mk_att_smem_bytes(int hd, int G) { return (size_t)GV_WARPS * 2 * G * (hd + 2) * 4; }

// merge state (m2, l2, o2) into (m, l, o)
__device__ inline void mk_merge(float &m, float &l, float *acc, float m2, float l2, const float *acc2) {
    const float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;
    const float c1 = exp2f(m - mn), c2 = exp2f(m2 - mn);
    l = l * c1 + l2 * c2;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = acc[i] * c1 + acc2[i] * c2;
    m = mn;
}

// Row indices are 32-bit: the launcher requires B * KV * cap * (CTAs + 1) < 2^31.
struct AttGeom {  // where (sequence b, KV head kvh) lies in the row list, and its split
    int NR, C;
    int T[ER_MK_MAXB];
    int base[ER_MK_MAXB + 1];
};

__device__ inline AttGeom att_geom(const StepArgs &p, const int *pos_s, int nctas) {
    AttGeom g;
    g.NR = 0;
    for (int b = 0; b < p.B; ++b) {
        const int pos = pos_s[b];
        g.T[b] = (pos >= 0 && pos < p.cap) ? pos + 1 : 0;
        g.base[b] = g.NR;
        g.NR += p.KV * g.T[b];
    }
    g.base[p.B] = g.NR;
    g.C = (g.NR + MK_ATT_MIN_ROWS - 1) / MK_ATT_MIN_ROWS;
    if (g.C > nctas) g.C = nctas;
    return g;
}

// (b, kvh, segment) holding row u of the list
__device__ inline void att_locate(const StepArgs &p, const AttGeom &g, int u, int &b, int &kvh, int &seg_start,
                                  int &seg_end) {
    b = 0;
    while (b + 1 < p.B && u >= g.base[b + 1]) ++b;
    kvh = (u - g.base[b]) / g.T[b];
    seg_start = g.base[b] + kvh * g.T[b];
    seg_end = seg_start + g.T[b];
}

// This warp's rows [wa, wb) of the list (empty for idle warps and CTAs)
__device__ inline void att_warp_range(const AttGeom &g, int cta, int warp, int &ca, int &cb, int &n, int &nw,
                                      int &wa, int &wb) {
    const bool cta_active = cta < g.C;
    ca = cta_active ? cta * g.NR / g.C : g.NR;
    cb = cta_active ? (cta + 1) * g.NR / g.C : g.NR;
    n = cb - ca;
    nw = n < GV_WARPS ? n : GV_WARPS;
    wa = warp < nw ? ca + warp * n / nw : cb;
    wb = warp < nw ? ca + (warp + 1) * n / nw : cb;
}

// Per segment s = b * KV + kvh: the CTAs c_first..c_last whose ranges hold its
// rows, and the state slot of c_first (0 if the segment starts at or before
// c_first's range, else 1; every later CTA uses slot 0).
constexpr int MK_MAX_SEGS = 256;
struct SegTable {
    unsigned char cf[MK_MAX_SEGS], cl[MK_MAX_SEGS], s0[MK_MAX_SEGS];
};

__device__ inline void seg_table_fill(const StepArgs &p, const AttGeom &g, SegTable &t, int tid, int nthreads) {
    for (int sgi = tid; sgi < p.B * p.KV; sgi += nthreads) {
        const int b = sgi / p.KV, kvh = sgi - b * p.KV;
        int cf = 0, cl = 0, s0 = 0;
        if (g.T[b] > 0) {
            const int seg_start = g.base[b] + kvh * g.T[b], seg_end = seg_start + g.T[b];
            cf = ((seg_start + 1) * g.C - 1) / g.NR;
            cl = (seg_end * g.C - 1) / g.NR;
            s0 = (cf * g.NR / g.C >= seg_start) ? 0 : 1;
        }
        t.cf[sgi] = (unsigned char)cf;
        t.cl[sgi] = (unsigned char)cl;
        t.s0[sgi] = (unsigned char)s0;
    }
}

template <int HD, int G>
__device__ void mk_attention(const StepArgs &p, const AttGeom &geo, int l, int cta, int warp, int lane,
                             float *att_smem) {
    constexpr int LPR = HD / 8, RPW = 32 / LPR;
    constexpr int U = G == 1 ? 4 : (G == 2 ? 2 : 1);  // rows per lane and buffer
    constexpr int SF = G * (HD + 2);                   // floats per parked warp state
    const int tid = threadIdx.x;
    const int rw = lane / LPR, dl = (lane % LPR) * 8;
    const int KV = p.KV, qd = p.H * HD;
    int ca, cb, wa, wb, n, nw;
    att_warp_range(geo, cta, warp, ca, cb, n, nw, wa, wb);
    const bool cta_active = cta < geo.C;
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);

    int u = wa;
    while (u < wb) {
        int b, kvh, seg_start, seg_end;
        att_locate(p, geo, u, b, kvh, seg_start, seg_end);
        const int r0 = u - seg_start, r1 = (wb < seg_end ? wb : seg_end) - seg_start;
        const bool first_seg = (u == wa);
        u = wb < seg_end ? wb : seg_end;

        const size_t head_off = (((size_t)b * p.L + l) * KV + kvh) * (size_t)p.cap * HD;
        const __half *Kb = p.kc + head_off + dl;
        const __half *Vb = p.vc + head_off + dl;
        float qv[G][8], m[G], ls[G], acc[G][8];
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            const float4 *qp = reinterpret_cast<const float4 *>(p.q + (size_t)b * qd + (kvh * G + gi) * HD + dl);
            const float4 x0 = __ldcg(qp), x1 = __ldcg(qp + 1);
            qv[gi][0] = x0.x * qscale; qv[gi][1] = x0.y * qscale; qv[gi][2] = x0.z * qscale; qv[gi][3] = x0.w * qscale;
            qv[gi][4] = x1.x * qscale; qv[gi][5] = x1.y * qscale; qv[gi][6] = x1.z * qscale; qv[gi][7] = x1.w * qscale;
            m[gi] = -INFINITY;
            ls[gi] = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[gi][i] = 0.f;
        }
        // two register buffers of U rows per lane: one batch loads while the
        // previous one is scored and accumulated
        uint4 kA[U], vA[U], kB[U], vB[U];
        auto load = [&](uint4 (&kr)[U], uint4 (&vr)[U], int rb) {
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                const int row = rb + uu * RPW + rw;
                kr[uu] = vr[uu] = make_uint4(0, 0, 0, 0);
                if (row < r1) {
                    kr[uu] = __ldcg(reinterpret_cast<const uint4 *>(Kb + (size_t)row * HD));
                    vr[uu] = __ldcg(reinterpret_cast<const uint4 *>(Vb + (size_t)row * HD));
                }
            }
        };
        auto consume = [&](const uint4 (&kr)[U], const uint4 (&vr)[U], int rb) {
            float sc[U][G];
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                const bool ok = rb + uu * RPW + rw < r1;
                const __half2 *kh = reinterpret_cast<const __half2 *>(&kr[uu]);
                float kf[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = __half22float2(kh[i]);
                    kf[2 * i] = f.x;
                    kf[2 * i + 1] = f.y;
                }
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    float d = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) d = fmaf(qv[gi][i], kf[i], d);
#pragma unroll
                    for (int off = 1; off < LPR; off <<= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                    sc[uu][gi] = ok ? d : -INFINITY;
                }
            }
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                float mn = m[gi];
#pragma unroll
                for (int uu = 0; uu < U; ++uu) mn = fmaxf(mn, sc[uu][gi]);
                if (mn == -INFINITY) continue;
                const float corr = exp2f(m[gi] - mn);
                ls[gi] *= corr;
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[gi][i] *= corr;
                m[gi] = mn;
#pragma unroll
                for (int uu = 0; uu < U; ++uu) {
                    const float pr = exp2f(sc[uu][gi] - mn);
                    ls[gi] += pr;
                    const __half2 *vh = reinterpret_cast<const __half2 *>(&vr[uu]);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = __half22float2(vh[i]);
                        acc[gi][2 * i] = fmaf(pr, f.x, acc[gi][2 * i]);
                        acc[gi][2 * i + 1] = fmaf(pr, f.y, acc[gi][2 * i + 1]);
                    }
                }
            }
        };
        constexpr int STEP = RPW * U;
        load(kA, vA, r0);
        for (int rb = r0; rb < r1; rb += 2 * STEP) {  // warp-uniform bounds
            if (rb + STEP < r1) load(kB, vB, rb + STEP);
            consume(kA, vA, rb);
            if (rb + STEP >= r1) break;
            if (rb + 2 * STEP < r1) load(kA, vA, rb + 2 * STEP);
            consume(kB, vB, rb + STEP);
        }
        // merge the RPW row slots of the warp (lanes with the same dl)
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                const float m2 = __shfl_xor_sync(0xffffffffu, m[gi], off);
                const float l2 = __shfl_xor_sync(0xffffffffu, ls[gi], off);
                float a2[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) a2[i] = __shfl_xor_sync(0xffffffffu, acc[gi][i], off);
                mk_merge(m[gi], ls[gi], acc[gi], m2, l2, a2);
            }
        }
        if (rw != 0) continue;
        if (seg_start >= wa && seg_end <= wb) {  // the whole head: finish here
            float *o_head = p.o + (size_t)b * qd + (size_t)kvh * G * HD + dl;
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                const float inv = ls[gi] > 0.f ? 1.f / ls[gi] : 0.f;
                float4 *op = reinterpret_cast<float4 *>(o_head + gi * HD);
                op[0] = make_float4(acc[gi][0] * inv, acc[gi][1] * inv, acc[gi][2] * inv, acc[gi][3] * inv);
                op[1] = make_float4(acc[gi][4] * inv, acc[gi][5] * inv, acc[gi][6] * inv, acc[gi][7] * inv);
            }
            continue;
        }
        // shared with other warps: park the state [gi][m, l, o[HD]] in shared memory
        float *st = att_smem + (warp * 2 + (first_seg ? 0 : 1)) * SF;
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            if (dl == 0) {
                st[gi * (HD + 2)] = m[gi];
                st[gi * (HD + 2) + 1] = ls[gi];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) st[gi * (HD + 2) + 2 + dl + i] = acc[gi][i];
        }
    }
    __syncthreads();  // every warp's states are parked (CTA-uniform from here)
    if (!cta_active) return;

    // ---- the CTA's heads that no single warp covered (one thread per output element)
    const int gi = tid / HD, d = tid % HD;
    if (tid >= G * HD) return;
    int v = ca;
    while (v < cb) {
        int b, kvh, seg_start, seg_end;
        att_locate(p, geo, v, b, kvh, seg_start, seg_end);
        v = cb < seg_end ? cb : seg_end;
        const int lo_local = (seg_start > ca ? seg_start : ca) - ca;
        const int hi_local = (seg_end < cb ? seg_end : cb) - ca;
        const int w_first = ((lo_local + 1) * nw - 1) / n, w_last = (hi_local * nw - 1) / n;
        const bool in_cta = seg_start >= ca && seg_end <= cb;
        if (in_cta && w_first == w_last) continue;  // one warp covered it: finished there
        const int w_first_a = ca + w_first * n / nw;
        const int first_slot = (w_first_a >= seg_start) ? 0 : 1;
        // merge the covering warps' states (warp order)
        float M = -INFINITY, L = 0.f, O = 0.f;
        for (int w = w_first; w <= w_last; ++w)
            M = fmaxf(M, att_smem[(w * 2 + (w == w_first ? first_slot : 0)) * SF + gi * (HD + 2)]);
        if (M != -INFINITY)
            for (int w = w_first; w <= w_last; ++w) {
                const float *st = att_smem + (w * 2 + (w == w_first ? first_slot : 0)) * SF + gi * (HD + 2);
                const float e = exp2f(st[0] - M);
                L = fmaf(st[1], e, L);
                O = fmaf(st[2 + d], e, O);
            }
        if (in_cta) {
            p.o[(size_t)b * qd + (size_t)(kvh * G + gi) * HD + d] = L > 0.f ? O / L : 0.f;
            continue;
        }
        // shared with other CTAs: leave the CTA's state for the Wo operand
        const int cslot = (seg_start <= ca) ? 0 : 1;
        float *gst = p.apart + ((size_t)(cta * 2 + cslot) * G + gi) * (HD + 4);
        gst[4 + d] = O;
        if (d == 0) {
            gst[0] = M;
            gst[1] = L;
        }
    }
}

// Operand source of the Wo phase: element k.. of column b of the attention
// output, merging (CTA order) the states of a head split over CTAs.
template <int HD, int G>
struct MkLoadAttn {
    const StepArgs *p;
    const SegTable *t;  // in shared memory
    __device__ void operator()(const GemvArgs &a, int b, int k, float (&v)[8]) const {
        const int h = k / HD, kvh = h / G, gi = h - kvh * G, d = k - h * HD;
        const int sgi = b * p->KV + kvh;
        const int cf = t->cf[sgi], cl = t->cl[sgi];
        if (cf == cl) {  // finished inside one CTA (or empty: zeros were written)
            const float4 *op = reinterpret_cast<const float4 *>(p->o + (size_t)b * p->qd + k);
            const float4 x0 = __ldcg(op), x1 = __ldcg(op + 1);
            v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w;
            v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
            return;
        }
        float M = -INFINITY, L = 0.f, O[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) O[i] = 0.f;
        for (int c0 = cf; c0 <= cl; c0 += 4) {  // four CTAs' states in flight
            float mm[4], ll[4];
            float4 o0[4], o1[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = c0 + j;
                mm[j] = -INFINITY;
                ll[j] = 0.f;
                o0[j] = o1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c <= cl) {
                    const int slot = c == cf ? t->s0[sgi] : 0;
                    const float *st = p->apart + ((size_t)(c * 2 + slot) * G + gi) * (HD + 4);
                    const float2 ml = __ldcg(reinterpret_cast<const float2 *>(st));
                    mm[j] = ml.x;
                    ll[j] = ml.y;
                    o0[j] = __ldcg(reinterpret_cast<const float4 *>(st + 4 + d));
                    o1[j] = __ldcg(reinterpret_cast<const float4 *>(st + 8 + d));
                }
            }
            float mc = M;
#pragma unroll
            for (int j = 0; j < 4; ++j) mc = fmaxf(mc, mm[j]);
            if (mc == -INFINITY) continue;
            const float corr = exp2f(M - mc);
            L *= corr;
#pragma unroll
            for (int i = 0; i < 8; ++i) O[i] *= corr;
            M = mc;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float e = exp2f(mm[j] - mc);
                L = fmaf(ll[j], e, L);
                O[0] = fmaf(o0[j].x, e, O[0]); O[1] = fmaf(o0[j].y, e, O[1]);
                O[2] = fmaf(o0[j].z, e, O[2]); O[3] = fmaf(o0[j].w, e, O[3]);
                O[4] = fmaf(o1[j].x, e, O[4]); O[5] = fmaf(o1[j].y, e, O[5]);
                O[6] = fmaf(o1[j].z, e, O[6]); O[7] = fmaf(o1[j].w, e, O[7]);
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = O[i] * inv;
    }
};

// ---------------------------------------------------------------------------
template <int QT, int HD, int G>
__global__ void __launch_bounds__(GV_WARPS * 32, 1) step_kernel(const StepArgs p) {
    using C = GvCfg<QT>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    const GvScratch s = gv_scratch(smem + mk_off_scratch<QT>());
    __shared__ int ok_smem;
    __shared__ GvRange rr_smem[GV_WARPS][5];  // this warp's ranges of the five matrix shapes
    __shared__ int pos_s[ER_MK_MAXB];                     // the step's positions
    __shared__ float2 rope_s[ER_MK_MAXB * (HD / 2)];      // their RoPE rows (cos, sin)
    __shared__ float resid_s[MK_RESID_RG * 16 * GV_MAXB];  // residual rows of a Wo / down phase
    __shared__ AttGeom geo_s;                             // the attention split of this step
    __shared__ SegTable seg_s;                            // and where its heads' states lie

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x, nctas = gridDim.x;
    const int L = p.L;
    const int ngp = 4 * L + 1;  // GEMV phases: (QKV, WO, GATEUP, DOWN) per layer, then HEAD
    GvRange *rr = rr_smem[warp];
    if (lane < 5) rr[lane] = gv_range(p.R[lane], p.UPR[lane], cta, nctas, warp, true);
    __syncwarp();
    uint64_t *wbar = bars + warp * GV_SLOTS;
    uint8_t *ring = smem + MK_OFF_RING + warp * GV_SLOTS * C::SLOT;

    // ---- producer (lane 0): the warp's slots of every GEMV of the step, in order
    int pg = 0, pk = 0;
    unsigned issued = 0, consumed = 0;
    auto issue_next = [&]() {
        while (pg < ngp) {
            const int type = pg == 4 * L ? 4 : (pg & 3);
            const GvRange &r = rr[type];
            const int nun = (int)(r.wb - r.wa);
            if (pk * C::SU < nun) {
                const uint8_t *w = type == 4 ? p.head : p.layers[pg >> 2].w[type];
                const int cnt = min(C::SU, nun - pk * C::SU);
                const uint32_t bytes = (uint32_t)cnt * C::UB;
                const unsigned sidx = issued % GV_SLOTS;
                mbar_arrive_expect_tx(wbar + sidx, bytes);
                bulk_g2s(ring + sidx * C::SLOT, w + (size_t)(r.wa + pk * C::SU) * C::UB, bytes, wbar + sidx);
                ++issued;
                ++pk;
                return;
            }
            ++pg;
            pk = 0;
        }
    };
    if (lane == 0) {
        for (int i = 0; i < GV_SLOTS; ++i) mbar_init(wbar + i, 1);
        fence_mbar_init();
        for (int i = 0; i < GV_SLOTS; ++i) issue_next();
    }
    __syncwarp();
    auto refill = [&](unsigned kg) {  // slot kg consumed
        if (lane == 0) {
            fence_proxy_async_smem();
            issue_next();
        }
        consumed = kg + 1;
    };

    unsigned gen = 0;
    bool ok = true;

    // ---- per-step constants: positions, RoPE rows, attention split
    if (tid < p.B) pos_s[tid] = p.positions[tid];
    __syncthreads();
    if (tid == 0) geo_s = att_geom(p, pos_s, nctas);
    __syncthreads();
    seg_table_fill(p, geo_s, seg_s, tid, blockDim.x);
    for (int i = tid; i < p.B * (HD / 2); i += blockDim.x) {
        const int b = i / (HD / 2), j = i - b * (HD / 2);
        const int pos = pos_s[b];
        rope_s[i] = (pos >= 0 && pos < p.cap) ? p.rope[(size_t)pos * (HD / 2) + j] : make_float2(1.f, 0.f);
    }

    // ---- EMBED
    {
        if (cta == 0 && tid < p.B) {
            const int tok = p.tokens[tid], pos = p.positions[tid];
            if (tok < 0 || tok >= p.V) atomicOr(p.flags, ER_FLAG_TOKEN);
            if (pos < 0 || pos >= p.cap) atomicOr(p.flags, ER_FLAG_POS);
        }
        for (int idx = cta * blockDim.x + tid; idx < p.B * p.D; idx += nctas * blockDim.x) {
            const int b = idx / p.D, k = idx - b * p.D;
            const int tok = p.tokens[b];
            float v = 0.f;
            if (tok >= 0 && tok < p.V)
                v = p.embd_f16 ? __half2float(p.embd_f16[(size_t)tok * p.D + k])
                               : repacked_value(p.head, QT, p.UPR[4], tok, k);
            p.x[(size_t)b * p.D + k] = v;
        }
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem, p.bar_extra);
    }

    // one GEMV phase; every thread of the CTA takes the same path through the
    // CTA barriers.  A failed ring wait (flag set) only skips this warp's shared
    // sums; the grid barrier after the phase sees the flag and stops every CTA.
    auto gemv = [&](GemvArgs &a, const GvRange &r, auto epi_tag, const auto &load) {
        constexpr int EPI = decltype(epi_tag)::value;
        bool good = true;
        a.resid_s = nullptr;
        if (lane == 0) s.wrg[warp * 2] = s.wrg[warp * 2 + 1] = -1;
        if (r.cta_active) {
            if (EPI == EPI_RESID) {
                // the residual rows this CTA finishes (whole row groups), read once up front
                const int rg0 = (int)(r.ca / a.UPR);
                const int nrg = min((int)((r.cb - r.ca) / a.UPR), MK_RESID_RG);
                for (int i = tid; i < nrg * 16 * a.B; i += blockDim.x) {
                    const int b = i % a.B, rr = i / a.B, row = rg0 * 16 + rr;
                    resid_s[rr * GV_MAXB + b] = row < a.N ? __ldcg(a.y + (size_t)b * a.N + row) : 0.f;
                }
                a.resid_s = resid_s;
                a.resid_rg0 = rg0;
                a.resid_nrg = nrg;
            }
            gv_operand(a, s, tid, blockDim.x, load);
            __syncthreads();
            if (r.working) good = gv_consume<QT, EPI>(a, s, r, ring, wbar, consumed, refill, lane, warp) >= 0;
            __syncthreads();
            if (good) gv_finish_shared<EPI>(a, s, r, cta, nctas, lane, warp);
        }
    };

    GemvArgs a = {};
    a.qt = QT;
    a.B = p.B;
    a.b0 = 0;
    a.eps = p.eps;
    a.part = p.part;
    a.cnt = p.cnt;
    a.flags = p.flags;
    a.positions = p.positions;
    a.qd = p.qd;
    a.kvd = p.kvd;
    a.hd = HD;
    a.KV = p.KV;
    a.L = L;
    a.cap = p.cap;
    a.kc = p.kc;
    a.vc = p.vc;
    a.rope = p.rope;
    a.q_out = p.q;
    a.a_out = p.a;
    a.amax = p.amax;
    a.done = p.done;
    a.argmax_out = p.argmax;
    a.pos_s = pos_s;
    a.rope_s = rope_s;
    const GvLoadX load_x{};
    const MkLoadAttn<HD, G> load_o{&p, &seg_s};

    for (int l = 0; l < L && ok; ++l) {
        const StepLayer &ly = p.layers[l];
        // QKV
        a.W = ly.w[0]; a.R = p.R[0]; a.UPR = p.UPR[0]; a.N = p.qd + 2 * p.kvd; a.K = p.D;
        a.x = p.x; a.gain = ly.attn_norm; a.layer = l;
        gemv(a, rr[0], std::integral_constant<int, EPI_QKV>(), load_x);
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
        if (!ok) break;
        // ATT (its shared-memory states reuse the GEMV operand area)
        mk_attention<HD, G>(p, geo_s, l, cta, warp, lane, reinterpret_cast<float *>(s.xs));
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
        if (!ok) break;
        // WO
        a.W = ly.w[1]; a.R = p.R[1]; a.UPR = p.UPR[1]; a.N = p.D; a.K = p.qd;
        a.x = p.o; a.gain = nullptr; a.y = p.x;
        gemv(a, rr[1], std::integral_constant<int, EPI_RESID>(), load_o);
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
        if (!ok) break;
        // GATEUP
        a.W = ly.w[2]; a.R = p.R[2]; a.UPR = p.UPR[2]; a.N = p.F; a.K = p.D;
        a.x = p.x; a.gain = ly.ffn_norm;
        gemv(a, rr[2], std::integral_constant<int, EPI_SWIGLU>(), load_x);
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
        if (!ok) break;
        // DOWN
        a.W = ly.w[3]; a.R = p.R[3]; a.UPR = p.UPR[3]; a.N = p.D; a.K = p.F;
        a.x = p.a; a.gain = nullptr; a.y = p.x;
        gemv(a, rr[3], std::integral_constant<int, EPI_RESID>(), load_x);
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
    }
    if (ok) {
        // HEAD
        a.W = p.head; a.R = p.R[4]; a.UPR = p.UPR[4]; a.N = p.V; a.K = p.D;
        a.x = p.x; a.gain = p.out_norm; a.y = p.logits;
        gemv(a, rr[4], std::integral_constant<int, EPI_LOGITS>(), load_x);
    }
    // copies still in flight (only after an error) must land before the CTA exits
    if (lane == 0)
        for (unsigned k = consumed; k < issued; ++k) mbar_wait(wbar + k % GV_SLOTS, (k / GV_SLOTS) & 1u);
}

}  // namespace er
