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
//   ATT     GQA attention over cache rows 0..pos (rows split evenly over all
//           warps of the grid; partial softmax states merged per KV head by
//           the last warp to finish it)
//   WO      x += Wo o
//   GATEUP  a = silu(Wgate h2) * (Wup h2), h2 = RMSNorm(x)
//   DOWN    x += Wdown a
//   HEAD    logits = Wout RMSNorm(x); argmax
// Every barrier wait is bounded (about a second of %globaltimer); a wait that
// gives up sets a device flag and every CTA returns after draining its copies.
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
// until *bar reaches gen * gridDim.x.  Returns false (all threads) if the wait
// gave up or another CTA flagged an error.
__device__ inline bool mk_barrier(unsigned *bar, int *flags, unsigned gen, int *ok_smem) {
    __syncthreads();
    if (threadIdx.x == 0) {
        red_add_release_gpu(bar, 1);
        const unsigned target = gen * gridDim.x;
        bool ok = true;
        if (ld_acquire_gpu(bar) < target) {
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t i = 1;; ++i) {
                if (ld_acquire_gpu(bar) >= target) break;
                if ((i & 31) == 0) {
                    if (*reinterpret_cast<volatile int *>(flags) & ER_FLAG_WAIT) {
                        ok = false;
                        break;
                    }
                    if (globaltimer_ns() - t0 > ER_WAIT_NS) {
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
// warp parks its state in shared memory; the CTA merges its warps' states of a
// head (one thread per output element, warp order); a head shared by CTAs has
// each CTA's merged state parked in global memory and merged, in CTA order, by
// the last CTA to arrive (a counter per head).
// ---------------------------------------------------------------------------
constexpr int MK_ATT_MIN_ROWS = 64;

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

struct AttGeom {  // where (sequence b, KV head kvh) lies in the row list, and its split
    long long NR, C;
    int T[ER_MK_MAXB];
    long long base[ER_MK_MAXB + 1];
};

__device__ inline AttGeom att_geom(const StepArgs &p, int nctas) {
    AttGeom g;
    g.NR = 0;
    for (int b = 0; b < p.B; ++b) {
        const int pos = p.positions[b];
        g.T[b] = (pos >= 0 && pos < p.cap) ? pos + 1 : 0;
        g.base[b] = g.NR;
        g.NR += (long long)p.KV * g.T[b];
    }
    g.base[p.B] = g.NR;
    g.C = (g.NR + MK_ATT_MIN_ROWS - 1) / MK_ATT_MIN_ROWS;
    if (g.C > nctas) g.C = nctas;
    return g;
}

// (b, kvh, segment) holding row u of the list
__device__ inline void att_locate(const StepArgs &p, const AttGeom &g, long long u, int &b, int &kvh,
                                  long long &seg_start, long long &seg_end) {
    b = 0;
    while (b + 1 < p.B && u >= g.base[b + 1]) ++b;
    kvh = (int)((u - g.base[b]) / g.T[b]);
    seg_start = g.base[b] + (long long)kvh * g.T[b];
    seg_end = seg_start + g.T[b];
}

template <int HD, int G>
__device__ void mk_attention(const StepArgs &p, int l, int cta, int nctas, int warp, int lane, float *att_smem) {
    constexpr int LPR = HD / 8, RPW = 32 / LPR;
    constexpr int U = G == 1 ? 8 : (G == 2 ? 4 : 2);  // rows in flight per lane
    constexpr int SF = G * (HD + 2);                   // floats per state
    __shared__ int last_s;
    __shared__ unsigned char slot_s[256];              // contributing CTAs' slots (cross-CTA merge)
    const int tid = threadIdx.x;
    const int rw = lane / LPR, dl = (lane % LPR) * 8;
    const int KV = p.KV, qd = p.H * HD;
    const AttGeom geo = att_geom(p, nctas);
    const long long NR = geo.NR, C = geo.C;
    const bool cta_active = cta < C;
    const long long ca = cta_active ? cta * NR / C : NR, cb = cta_active ? (cta + 1) * NR / C : NR;
    const int n = (int)(cb - ca), nw = n < GV_WARPS ? n : GV_WARPS;
    const long long wa = warp < nw ? ca + (long long)warp * n / nw : cb;
    const long long wb = warp < nw ? ca + (long long)(warp + 1) * n / nw : cb;
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);

    long long u = wa;
    while (u < wb) {
        int b, kvh;
        long long seg_start, seg_end;
        att_locate(p, geo, u, b, kvh, seg_start, seg_end);
        const int r0 = (int)(u - seg_start), r1 = (int)((wb < seg_end ? wb : seg_end) - seg_start);
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
        for (int rb = r0; rb < r1; rb += RPW * U) {  // warp-uniform bound
            uint4 kr[U], vr[U];
#pragma unroll
            for (int uu = 0; uu < U; ++uu) {
                const int row = rb + uu * RPW + rw;
                kr[uu] = vr[uu] = make_uint4(0, 0, 0, 0);
                if (row < r1) {
                    kr[uu] = __ldcg(reinterpret_cast<const uint4 *>(Kb + (size_t)row * HD));
                    vr[uu] = __ldcg(reinterpret_cast<const uint4 *>(Vb + (size_t)row * HD));
                }
            }
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

    // ---- the CTA's heads that no single warp covered (loop is CTA-uniform)
    const int gi = tid / HD, d = tid % HD;  // one thread per output element
    const bool elem = tid < G * HD;
    long long v = ca;
    while (v < cb) {
        int b, kvh;
        long long seg_start, seg_end;
        att_locate(p, geo, v, b, kvh, seg_start, seg_end);
        v = cb < seg_end ? cb : seg_end;
        const int lo_local = (int)((seg_start > ca ? seg_start : ca) - ca);
        const int hi_local = (int)((seg_end < cb ? seg_end : cb) - ca);
        const int w_first = ((lo_local + 1) * nw - 1) / n, w_last = (hi_local * nw - 1) / n;
        const bool in_cta = seg_start >= ca && seg_end <= cb;
        if (in_cta && w_first == w_last) continue;  // one warp covered it: finished there
        const long long w_first_a = ca + (long long)w_first * n / nw;
        const int first_slot = (w_first_a >= seg_start) ? 0 : 1;
        // merge the covering warps' states (warp order)
        float M = -INFINITY, L = 0.f, O = 0.f;
        if (elem) {
            for (int w = w_first; w <= w_last; ++w)
                M = fmaxf(M, att_smem[(w * 2 + (w == w_first ? first_slot : 0)) * SF + gi * (HD + 2)]);
            if (M != -INFINITY)
                for (int w = w_first; w <= w_last; ++w) {
                    const float *st = att_smem + (w * 2 + (w == w_first ? first_slot : 0)) * SF + gi * (HD + 2);
                    const float e = exp2f(st[0] - M);
                    L = fmaf(st[1], e, L);
                    O = fmaf(st[2 + d], e, O);
                }
        }
        float *o_group = p.o + (size_t)b * qd + (size_t)kvh * G * HD;
        if (in_cta) {
            if (elem) o_group[gi * HD + d] = L > 0.f ? O / L : 0.f;
            continue;
        }
        // shared with other CTAs: park the CTA's state; the last CTA to arrive merges
        const int cslot = (seg_start <= ca) ? 0 : 1;
        float *gst = p.apart + ((size_t)cta * 2 + cslot) * SF + gi * (HD + 2);
        if (elem) {
            gst[2 + d] = O;
            if (d == 0) {
                gst[0] = M;
                gst[1] = L;
            }
        }
        const long long c_first = ((seg_start + 1) * C - 1) / NR, c_last = (seg_end * C - 1) / NR;
        const int F = (int)(c_last - c_first + 1);
        __syncthreads();
        if (tid == 0) {
            const int grp = b * KV + kvh;
            last_s = atom_add_acq_rel_gpu(p.acnt + grp, 1) == F - 1;  // releases the CTA's state
            if (last_s) p.acnt[grp] = 0;
        }
        for (int j = tid; j < F && j < 256; j += blockDim.x)
            slot_s[j] = ((c_first + j) * NR / C >= seg_start) ? 0 : 1;
        __syncthreads();
        if (last_s && elem) {
            // online merge in CTA order, eight contributors' loads in flight at a time
            float Mg = -INFINITY, Lg = 0.f, Og = 0.f;
            for (int j0 = 0; j0 < F; j0 += 8) {
                float mm[8], ll[8], oo[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const bool ok = j0 + q < F;
                    const float *cs = p.apart + ((size_t)(c_first + (ok ? j0 + q : 0)) * 2 + slot_s[ok ? j0 + q : 0]) * SF +
                                      gi * (HD + 2);
                    mm[q] = ok ? __ldcg(cs) : -INFINITY;
                    ll[q] = ok ? __ldcg(cs + 1) : 0.f;
                    oo[q] = ok ? __ldcg(cs + 2 + d) : 0.f;
                }
                float mc = Mg;
#pragma unroll
                for (int q = 0; q < 8; ++q) mc = fmaxf(mc, mm[q]);
                if (mc == -INFINITY) continue;
                const float corr = exp2f(Mg - mc);
                Lg *= corr;
                Og *= corr;
                Mg = mc;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float e = exp2f(mm[q] - mc);
                    Lg = fmaf(ll[q], e, Lg);
                    Og = fmaf(oo[q], e, Og);
                }
            }
            o_group[gi * HD + d] = Lg > 0.f ? Og / Lg : 0.f;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
template <int QT, int HD, int G>
__global__ void __launch_bounds__(GV_WARPS * 32, 1) step_kernel(const StepArgs p) {
    using C = GvCfg<QT>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    const GvScratch s = gv_scratch(smem + mk_off_scratch<QT>());
    __shared__ int ok_smem;
    __shared__ GvRange rr_smem[GV_WARPS][5];  // this warp's ranges of the five matrix shapes

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
    long long issued = 0, consumed = 0;
    auto issue_next = [&]() {
        while (pg < ngp) {
            const int type = pg == 4 * L ? 4 : (pg & 3);
            const GvRange &r = rr[type];
            const int nun = (int)(r.wb - r.wa);
            if (pk * C::SU < nun) {
                const uint8_t *w = type == 4 ? p.head : p.layers[pg >> 2].w[type];
                const int cnt = min(C::SU, nun - pk * C::SU);
                const uint32_t bytes = (uint32_t)cnt * C::UB;
                const int sidx = (int)(issued % GV_SLOTS);
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
    auto refill = [&](long long kg) {  // slot kg consumed
        if (lane == 0) {
            fence_proxy_async_smem();
            issue_next();
        }
        consumed = kg + 1;
    };

    unsigned gen = 0;
    bool ok = true;

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
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
    }

    // one GEMV phase; every thread of the CTA takes the same path through the
    // CTA barriers.  A failed ring wait (flag set) only skips this warp's shared
    // sums; the grid barrier after the phase sees the flag and stops every CTA.
    auto gemv = [&](const GemvArgs &a, const GvRange &r, auto epi_tag) {
        constexpr int EPI = decltype(epi_tag)::value;
        bool good = true;
        if (lane == 0) s.wrg[warp * 2] = s.wrg[warp * 2 + 1] = -1;
        if (r.cta_active) {
            gv_operand(a, s, tid, blockDim.x);
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

    for (int l = 0; l < L && ok; ++l) {
        const StepLayer &ly = p.layers[l];
        // QKV
        a.W = ly.w[0]; a.R = p.R[0]; a.UPR = p.UPR[0]; a.N = p.qd + 2 * p.kvd; a.K = p.D;
        a.x = p.x; a.gain = ly.attn_norm; a.layer = l;
        gemv(a, rr[0], std::integral_constant<int, EPI_QKV>());
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
        if (!ok) break;
        // ATT (its shared-memory states reuse the GEMV operand area)
        mk_attention<HD, G>(p, l, cta, nctas, warp, lane, reinterpret_cast<float *>(s.xs));
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
        if (!ok) break;
        // WO
        a.W = ly.w[1]; a.R = p.R[1]; a.UPR = p.UPR[1]; a.N = p.D; a.K = p.qd;
        a.x = p.o; a.gain = nullptr; a.y = p.x;
        gemv(a, rr[1], std::integral_constant<int, EPI_RESID>());
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
        if (!ok) break;
        // GATEUP
        a.W = ly.w[2]; a.R = p.R[2]; a.UPR = p.UPR[2]; a.N = p.F; a.K = p.D;
        a.x = p.x; a.gain = ly.ffn_norm;
        gemv(a, rr[2], std::integral_constant<int, EPI_SWIGLU>());
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
        if (!ok) break;
        // DOWN
        a.W = ly.w[3]; a.R = p.R[3]; a.UPR = p.UPR[3]; a.N = p.D; a.K = p.F;
        a.x = p.a; a.gain = nullptr; a.y = p.x;
        gemv(a, rr[3], std::integral_constant<int, EPI_RESID>());
        ok = mk_barrier(p.bar, p.flags, ++gen, &ok_smem);
    }
    if (ok) {
        // HEAD
        a.W = p.head; a.R = p.R[4]; a.UPR = p.UPR[4]; a.N = p.V; a.K = p.D;
        a.x = p.x; a.gain = p.out_norm; a.y = p.logits;
        gemv(a, rr[4], std::integral_constant<int, EPI_LOGITS>());
    }
    // copies still in flight (only after an error) must land before the CTA exits
    if (lane == 0)
        for (long long k = consumed; k < issued; ++k) mbar_wait(wbar + k % GV_SLOTS, (uint32_t)((k / GV_SLOTS) & 1));
}

}  // namespace er
