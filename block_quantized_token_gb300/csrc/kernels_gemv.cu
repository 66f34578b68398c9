// Block-quantized GEMV (batch 1..4) with fused prologue and epilogues.
//
// y_b = W x_b for every batch column b, W a repacked Q8_0 / Q4_0 matrix.  One
// weight pass serves all columns; every weight byte is read from HBM once.
//
// Work split (two-level "stream-K"): the matrix is a list of U = R * UPR units
// (16 rows x 64 columns, contiguous in memory).  CTA c takes the contiguous
// range [c U / C, (c+1) U / C) and splits it evenly over its warps, so every
// warp streams the same number of bytes whatever the matrix shape.  A row group
// inside one warp's range is finished by that warp; one shared by warps of a
// CTA is summed in shared memory in warp order; one shared by CTAs (at most the
// first and last of each CTA) is finished by the last CTA to arrive (an
// acquire-release counter), which sums the CTAs' partials in CTA order.  The
// result does not depend on timing.  When the matrix has no more row groups
// than SMs and short rows, C = R: every CTA owns whole row groups.
//
// Streaming: each warp owns a ring of shared-memory slots filled by bulk async
// copies (cp.async.bulk, completion on an mbarrier).  The first slots are
// requested before griddepcontrol.wait, so the weight traffic of this kernel
// overlaps the tail of the previous one.
//
// Dot products: the unit's int8 / int4 values are turned into exact fp16 in
// registers and multiplied on the tensor cores (mma m16n8k16, fp32 accumulate)
// with the activations split as x = hi + lo (two fp16 columns per batch
// column, |x - hi - lo| <= 2^-22 |x| after a power-of-two rescale), one MMA pair
// per 32-block; the block's fp16 scale d multiplies the fp32 block sum.  The
// tensor cores here are a way to keep the per-weight instruction count below
// the HBM byte rate, not a contraction in their own right: the kernel is
// bound by HBM bandwidth.
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
    static constexpr int SU = QT == Q8_0 ? 2 : 4;  // units per slot
    static constexpr int SLOT = SU * UB;            // 2176 / 2304 bytes
    static constexpr int RING = GV_WARPS * GV_SLOTS * SLOT;
};

// shared-memory map:
//   [mbarriers 512][rings][factors 64][reduce 512][warp partials][warp row groups 128][operand]
constexpr int GV_OFF_RING = 512;
template <int QT>
constexpr int gv_off_fac() { return GV_OFF_RING + GvCfg<QT>::RING; }
template <int QT>
constexpr int gv_off_red() { return gv_off_fac<QT>() + 64; }
template <int QT>
constexpr int gv_off_wpart() { return gv_off_red<QT>() + 512; }
template <int QT>
constexpr int gv_off_wrg() { return gv_off_wpart<QT>() + GV_WARPS * 2 * 64 * 4; }
template <int QT>
constexpr int gv_off_xs() { return gv_off_wrg<QT>() + 128; }

__host__ __device__ inline int gv_nbp(int K) { return ((K / 32) + 1) & ~1; }
__host__ __device__ inline size_t gv_xs_bytes(int K, int B) { return (size_t)gv_nbp(K) * B * 128; }

// ---------------------------------------------------------------------------
// epilogues: lane (g, t) holds rows g and g+8 of row group rg for batch t
// ---------------------------------------------------------------------------
template <int EPI>
__device__ inline void gv_epilogue(const GemvArgs &a, int rg, float v0, float v1, const float *fac, int lane) {
    const int g = lane >> 2, t = lane & 3;
    const bool bok = t < a.B;
    const int bt = a.b0 + t;  // column of the whole batch
    if (EPI == EPI_STORE || EPI == EPI_RESID) {
        if (!bok) return;
        v0 *= fac[t];
        v1 *= fac[t];
        int r0 = 16 * rg + g, r1 = r0 + 8;
        float *y = a.y + (size_t)bt * a.N;
        if (EPI == EPI_STORE) {
            if (r0 < a.N) y[r0] = v0;
            if (r1 < a.N) y[r1] = v1;
        } else {
            if (r0 < a.N) y[r0] += v0;
            if (r1 < a.N) y[r1] += v1;
        }
    } else if (EPI == EPI_QKV) {
        if (!bok) return;
        v0 *= fac[t];
        v1 *= fac[t];
        const int pos = a.positions[bt];
        if (pos < 0 || pos >= a.cap) return;
        int r0 = 16 * rg + 2 * g;  // RoPE pair (r0, r0 + 1)
        if (r0 >= a.qd + 2 * a.kvd) return;
        if (r0 < a.qd + a.kvd) {  // q or k: rotate
            int base = r0 < a.qd ? r0 : r0 - a.qd;
            int dd = base % a.hd;
            float2 cs = a.rope[(size_t)pos * (a.hd / 2) + dd / 2];
            float o0 = v0 * cs.x - v1 * cs.y;
            float o1 = v1 * cs.x + v0 * cs.y;
            if (r0 < a.qd) {
                float2 *q = reinterpret_cast<float2 *>(a.q_out + (size_t)bt * a.qd + r0);
                *q = make_float2(o0, o1);
            } else {
                int kvh = base / a.hd;
                size_t off = ((((size_t)bt * a.L + a.layer) * a.KV + kvh) * a.cap + pos) * a.hd + dd;
                *reinterpret_cast<__half2 *>(a.kc + off) = __floats2half2_rn(o0, o1);
            }
        } else {
            int base = r0 - a.qd - a.kvd;
            int kvh = base / a.hd, dd = base % a.hd;
            size_t off = ((((size_t)bt * a.L + a.layer) * a.KV + kvh) * a.cap + pos) * a.hd + dd;
            *reinterpret_cast<__half2 *>(a.vc + off) = __floats2half2_rn(v0, v1);
        }
    } else if (EPI == EPI_SWIGLU) {
        if (!bok) return;
        int n = 8 * rg + g;
        if (n >= a.N) return;
        float gt = v0 * fac[t], up = v1 * fac[t];
        a.a_out[(size_t)bt * a.N + n] = gt / (1.f + expf(-gt)) * up;
    } else {  // EPI_LOGITS
        unsigned long long key = 0;
        if (bok) {
            v0 *= fac[t];
            v1 *= fac[t];
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
template <int QT, int EPI>
__global__ void __launch_bounds__(GV_WARPS * 32, 1) gemv_kernel(const GemvArgs a) {
    using C = GvCfg<QT>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    float *fac = reinterpret_cast<float *>(smem + gv_off_fac<QT>());
    float *red = reinterpret_cast<float *>(smem + gv_off_red<QT>());
    float *wpart = reinterpret_cast<float *>(smem + gv_off_wpart<QT>());
    int *wrg = reinterpret_cast<int *>(smem + gv_off_wrg<QT>());
    uint8_t *xs = smem + gv_off_xs<QT>();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int UPR = a.UPR;
    const long long U = (long long)a.R * UPR;
    const int nC = gridDim.x, cta = blockIdx.x;
    const long long ca = (long long)cta * U / nC, cb = (long long)(cta + 1) * U / nC;
    const int n = (int)(cb - ca);  // units of this CTA (>= 1)
    const int nw = n < GV_WARPS ? n : GV_WARPS;
    const bool working = warp < nw;
    const long long wa = working ? ca + (long long)warp * n / nw : cb;
    const long long wb = working ? ca + (long long)(warp + 1) * n / nw : cb;
    const int nunits = (int)(wb - wa);
    const int nslots = (nunits + C::SU - 1) / C::SU;
    uint64_t *wbar = bars + warp * GV_SLOTS;
    uint8_t *ring = smem + GV_OFF_RING + warp * GV_SLOTS * C::SLOT;
    const uint8_t *wsrc = a.W + (size_t)wa * C::UB;

    auto issue = [&](int k) {  // lane 0 only
        int s = k % GV_SLOTS;
        int cnt = min(C::SU, nunits - k * C::SU);
        uint32_t bytes = (uint32_t)cnt * C::UB;
        mbar_arrive_expect_tx(wbar + s, bytes);
        bulk_g2s(ring + s * C::SLOT, wsrc + (size_t)k * C::SLOT, bytes, wbar + s);
    };

    int issued = min(GV_SLOTS, nslots);
    if (lane == 0) {
        for (int s = 0; s < GV_SLOTS; ++s) mbar_init(wbar + s, 1);
        fence_mbar_init();
        for (int k = 0; k < issued; ++k) issue(k);
        wrg[warp * 2] = wrg[warp * 2 + 1] = -1;
    }
    __syncwarp();

    // ---- everything above touches only constant weights; now wait for inputs
    pdl_wait();
    int flag_wait = 0;
    if (tid == 0) flag_wait = *reinterpret_cast<volatile int *>(a.flags) & ER_FLAG_WAIT;

    // ---- prologue, one pass over global memory: v = x * gain (fp32) into the
    // operand area as [kb][b][32 floats], with per-column sum of squares and max|v|
    const int K = a.K, B = a.B;
    const int nbp = gv_nbp(K);
    {
        float ss[GV_MAXB], mx[GV_MAXB];
#pragma unroll
        for (int b = 0; b < GV_MAXB; ++b) ss[b] = mx[b] = 0.f;
        const int k4n = K / 4;
        for (int idx = tid; idx < B * k4n; idx += blockDim.x) {
            const int b = idx / k4n, k = (idx - b * k4n) * 4;
            float4 v = *reinterpret_cast<const float4 *>(a.x + (size_t)(a.b0 + b) * K + k);
            float sq = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            if (a.gain) {
                float4 gn = *reinterpret_cast<const float4 *>(a.gain + k);
                v.x *= gn.x;
                v.y *= gn.y;
                v.z *= gn.z;
                v.w *= gn.w;
            }
            float m = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
            for (int bb = 0; bb < GV_MAXB; ++bb)
                if (bb == b) {
                    ss[bb] += sq;
                    mx[bb] = fmaxf(mx[bb], m);
                }
            *reinterpret_cast<float4 *>(xs + ((size_t)((k >> 5) * B + b) * 32 + (k & 31)) * 4) = v;
        }
        // zero the padding block (an odd number of blocks per row)
        for (int idx = tid; idx < (nbp * 32 - K) * B; idx += blockDim.x) {
            int b = idx / (nbp * 32 - K), k = K + idx % (nbp * 32 - K);
            *reinterpret_cast<float *>(xs + ((size_t)((k >> 5) * B + b) * 32 + (k & 31)) * 4) = 0.f;
        }
        for (int b = 0; b < B; ++b) {
            float s = ss[0], m = mx[0];
#pragma unroll
            for (int bb = 1; bb < GV_MAXB; ++bb)
                if (bb == b) {
                    s = ss[bb];
                    m = mx[bb];
                }
            for (int off = 16; off; off >>= 1) {
                s += __shfl_xor_sync(0xffffffffu, s, off);
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            }
            if (lane == 0) {
                red[(warp * GV_MAXB + b) * 2] = s;
                red[(warp * GV_MAXB + b) * 2 + 1] = m;
            }
        }
        if (tid == 0) fac[8] = flag_wait ? 1.f : 0.f;  // red[] is full: 16 warps x 4 columns x 2
        __syncthreads();
    }
    // a kernel earlier in the stream gave up on a wait: the state is already
    // invalid, so drain this warp's copies and stop (one read, shared by the CTA)
    if (fac[8] != 0.f) {
        if (lane == 0)
            for (int k = 0; k < issued; ++k) mbar_wait(wbar + k % GV_SLOTS, (k / GV_SLOTS) & 1);
        return;
    }
    pdl_launch_dependents();

    // per-column factors: fac[b] = rstd * 2^-e (epilogue), scale 2^e (operand)
    auto column_scale = [&](int b, float &rstd_unscale) -> float {
        float s = 0.f, m = 0.f;
        for (int w = 0; w < GV_WARPS; ++w) {
            s += red[(w * GV_MAXB + b) * 2];
            m = fmaxf(m, red[(w * GV_MAXB + b) * 2 + 1]);
        }
        int e = 0;
        if (m > 0.f && isfinite(m)) {
            int E;
            frexpf(m, &E);
            e = 15 - E;  // max |v| * 2^e in [2^14, 2^15)
        }
        float rstd = a.gain ? 1.f / sqrtf(s / (float)K + a.eps) : 1.f;
        rstd_unscale = ldexpf(rstd, -e);
        return ldexpf(1.f, e);
    };
    if (tid < B) {
        float f;
        column_scale(tid, f);
        fac[tid] = f;
    }

    // ---- operand: each (block kb, column b) 128-byte area turns, in place, from
    // 32 fp32 values into the MMA B fragments [g = 2b (hi), 2b+1 (lo)][t][16 bytes];
    // four lanes per area, reads before writes within the warp
    {
        const int nq = nbp * B * 4;
        for (int base = warp * 32; base < nq; base += blockDim.x) {
            const int idx = base + lane;
            const bool ok = idx < nq;
            const int item = idx >> 2, q = idx & 3;
            uint8_t *area = xs + (size_t)item * 128;
            float v[8];
            if (ok) {
                float4 f0 = reinterpret_cast<const float4 *>(area)[2 * q];
                float4 f1 = reinterpret_cast<const float4 *>(area)[2 * q + 1];
                v[0] = f0.x; v[1] = f0.y; v[2] = f0.z; v[3] = f0.w;
                v[4] = f1.x; v[5] = f1.y; v[6] = f1.z; v[7] = f1.w;
            }
            __syncwarp();
            if (ok) {
                float unused;
                const float sc = column_scale(item % B, unused);
#pragma unroll
                for (int p = 0; p < 4; ++p) {  // element pair (2j, 2j+1), j = 4q + p
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
            }
        }
    }
    __syncthreads();

    // ---- main loop
    const bool has_b = g < 2 * B;
    const uint32_t xs_lane = smem_u32(xs) + (uint32_t)((g * 4 + t) * 16);
    const uint32_t xs_kb_stride = (uint32_t)(2 * B * 64);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    const long long wrg_first = wa / UPR;

    // one unit: 2 blocks x 16 rows, A fragments from shared memory
    auto unit = [&](uint32_t ub, int j, float &acc0, float &acc1) {
        const uint32_t xa = xs_lane + (uint32_t)(2 * j) * xs_kb_stride;
        uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = make_uint4(0, 0, 0, 0);
        if (has_b) {
            xb0 = lds128(xa);
            xb1 = lds128(xa + xs_kb_stride);
        }
        const uint2 sc = lds64(ub + C::QB + g * 8);
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
            acc0 = fmaf(h2f_lo(sc.x), c[0] + c[1], acc0);
            acc1 = fmaf(h2f_hi(sc.x), c[2] + c[3], acc1);
            q8_word_to_h2(q1.x, fa[0], fa[1]);
            q8_word_to_h2(q1.y, fa[2], fa[3]);
            mma_16816(c, fa, xb1.x, xb1.y, zero4);
            q8_word_to_h2(q1.z, fa[0], fa[1]);
            q8_word_to_h2(q1.w, fa[2], fa[3]);
            mma_16816(c, fa, xb1.z, xb1.w, c);
            acc0 = fmaf(h2f_lo(sc.y), c[0] + c[1], acc0);
            acc1 = fmaf(h2f_hi(sc.y), c[2] + c[3], acc1);
        } else {
            const uint4 q = lds128(ub + lane * 16);
            q4_word_to_h2(q.x, fa);
            mma_16816(c, fa, xb0.x, xb0.y, zero4);
            q4_word_to_h2(q.y, fa);
            mma_16816(c, fa, xb0.z, xb0.w, c);
            acc0 = fmaf(h2f_lo(sc.x), c[0] + c[1], acc0);
            acc1 = fmaf(h2f_hi(sc.x), c[2] + c[3], acc1);
            q4_word_to_h2(q.z, fa);
            mma_16816(c, fa, xb1.x, xb1.y, zero4);
            q4_word_to_h2(q.w, fa);
            mma_16816(c, fa, xb1.z, xb1.w, c);
            acc0 = fmaf(h2f_lo(sc.y), c[0] + c[1], acc0);
            acc1 = fmaf(h2f_hi(sc.y), c[2] + c[3], acc1);
        }
    };

    // a row group this warp leaves: finished here if the warp covered all of
    // it, otherwise parked in shared memory for the CTA-level sum
    auto leave = [&](int rgf, float v0, float v1) {
        const long long r_lo = (long long)rgf * UPR, r_hi = r_lo + UPR;
        if (r_lo >= wa && r_hi <= wb) {
            gv_epilogue<EPI>(a, rgf, v0, v1, fac, lane);
            return;
        }
        const int slot = (rgf == wrg_first) ? 0 : 1;
        *reinterpret_cast<float2 *>(wpart + (warp * 2 + slot) * 64 + lane * 2) = make_float2(v0, v1);
        if (lane == 0) wrg[warp * 2 + slot] = rgf;
    };

    float acc0 = 0.f, acc1 = 0.f, accb0 = 0.f, accb1 = 0.f;
    int rg = (int)wrg_first;
    int j = (int)(wa - (long long)rg * UPR);
    int aborted_at = -1;
    for (int k = 0; k < nslots; ++k) {
        const int s = k % GV_SLOTS;
        if (!mbar_wait(wbar + s, (k / GV_SLOTS) & 1)) {
            if (lane == 0) atomicOr(a.flags, ER_FLAG_WAIT);
            aborted_at = k;
            break;
        }
        const int cnt = min(C::SU, nunits - k * C::SU);
        const uint32_t slot_base = smem_u32(ring + s * C::SLOT);
        for (int i = 0; i < cnt;) {
            if (j == UPR) {
                leave(rg, acc0 + accb0, acc1 + accb1);
                acc0 = acc1 = accb0 = accb1 = 0.f;
                ++rg;
                j = 0;
            }
            if (i + 1 < cnt && j + 1 < UPR) {  // two independent units in flight
                unit(slot_base + i * C::UB, j, acc0, acc1);
                unit(slot_base + (i + 1) * C::UB, j + 1, accb0, accb1);
                i += 2;
                j += 2;
            } else {
                unit(slot_base + i * C::UB, j, acc0, acc1);
                i += 1;
                j += 1;
            }
        }
        __syncwarp();
        if (k + GV_SLOTS < nslots) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(k + GV_SLOTS);
            }
            ++issued;
        }
    }
    if (aborted_at >= 0) {
        // wait (bounded) for this warp's copies still in flight before the CTA exits
        if (lane == 0)
            for (int k = aborted_at; k < issued; ++k) mbar_wait(wbar + k % GV_SLOTS, (k / GV_SLOTS) & 1);
    } else if (nunits > 0) {
        leave(rg, acc0 + accb0, acc1 + accb1);
    }
    __syncthreads();

    // ---- CTA level: row groups shared by warps; the lowest warp sums them
    const long long cfirst = ca / UPR;
    for (int slot = 0; slot < 2; ++slot) {
        const int rgf = (working && aborted_at < 0) ? wrg[warp * 2 + slot] : -1;
        if (rgf < 0) continue;
        const long long r_lo = (long long)rgf * UPR, r_hi = r_lo + UPR;
        const int lo_local = (int)((r_lo > ca ? r_lo : ca) - ca);
        const int hi_local = (int)((r_hi < cb ? r_hi : cb) - ca);
        const int w_first = ((lo_local + 1) * nw - 1) / n;
        if (w_first != warp) continue;
        const int w_last = (hi_local * nw - 1) / n;
        float2 v = *reinterpret_cast<const float2 *>(wpart + (warp * 2 + slot) * 64 + lane * 2);
        for (int w = warp + 1; w <= w_last; ++w) {
            float2 o = *reinterpret_cast<const float2 *>(wpart + (w * 2) * 64 + lane * 2);
            v.x += o.x;
            v.y += o.y;
        }
        if (r_lo >= ca && r_hi <= cb) {
            gv_epilogue<EPI>(a, rgf, v.x, v.y, fac, lane);
            continue;
        }
        // ---- grid level: a row group shared by CTAs; the last CTA to arrive sums them
        const int cslot = (rgf == cfirst) ? 0 : 1;
        *reinterpret_cast<float2 *>(a.part + ((size_t)cta * 2 + cslot) * 64 + lane * 2) = v;
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atom_add_acq_rel_gpu(a.cnt + rgf, 1);  // releases the partial
        old = __shfl_sync(0xffffffffu, old, 0);
        __syncwarp();
        const long long c_first = ((r_lo + 1) * nC - 1) / U, c_last = (r_hi * nC - 1) / U;
        if (old == (int)(c_last - c_first)) {  // the acquire above orders these loads after every partial
            float s0 = 0.f, s1 = 0.f;
            for (long long c = c_first; c <= c_last; ++c) {
                const int sl = ((c * U / nC) / UPR == rgf) ? 0 : 1;
                const float *q = a.part + ((size_t)c * 2 + sl) * 64 + lane * 2;
                s0 += __ldcg(q);
                s1 += __ldcg(q + 1);
            }
            gv_epilogue<EPI>(a, rgf, s0, s1, fac, lane);
            if (lane == 0) a.cnt[rgf] = 0;
        }
    }
}

// ---------------------------------------------------------------------------
size_t gemv_part_floats(int num_sms) { return (size_t)num_sms * 2 * 64; }

template <int QT>
static size_t gv_smem(int K, int B) { return gv_off_xs<QT>() + gv_xs_bytes(K, B); }

template <int QT, int EPI>
static cudaError_t gv_attr() {
    cudaError_t e = cudaFuncSetAttribute(gemv_kernel<QT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    // one shared-memory carveout for every kernel of the step: no L1/shared
    // reconfiguration between consecutive launches
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_kernel<QT, EPI>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t gemv_prepare() {
    cudaError_t e = cudaSuccess;
    cudaError_t r[10] = {gv_attr<Q8_0, EPI_STORE>(), gv_attr<Q8_0, EPI_RESID>(), gv_attr<Q8_0, EPI_QKV>(),
                         gv_attr<Q8_0, EPI_SWIGLU>(), gv_attr<Q8_0, EPI_LOGITS>(), gv_attr<Q4_0, EPI_STORE>(),
                         gv_attr<Q4_0, EPI_RESID>(), gv_attr<Q4_0, EPI_QKV>(), gv_attr<Q4_0, EPI_SWIGLU>(),
                         gv_attr<Q4_0, EPI_LOGITS>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) e = x;
    if (e == cudaSuccess) e = attention_prepare();
    return e;
}

bool gemv_fits(int qt, int K, int B) {
    if (B < 1 || B > GV_MAXB || K % 32) return false;
    size_t need = qt == Q8_0 ? gv_smem<Q8_0>(K, B) : gv_smem<Q4_0>(K, B);
    return need <= 227 * 1024;
}

int gemv_max_cols(int qt, int K) {
    for (int b = GV_MAXB; b >= 1; --b)
        if (gemv_fits(qt, K, b)) return b;
    return 0;
}

// Grid size: one CTA per row group when there are no more row groups than SMs
// and rows are short (no cross-CTA sums at all); otherwise one CTA per SM.
int gemv_grid(int R, int UPR, int num_sms) {
    if (R <= num_sms && UPR <= 32) return R;
    long long U = (long long)R * UPR;
    return (int)(U < num_sms ? U : num_sms);
}

template <int QT, int EPI>
static cudaError_t gv_launch(const GemvArgs &a, int num_sms, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)gemv_grid(a.R, a.UPR, num_sms));
    cfg.blockDim = dim3(GV_WARPS * 32);
    cfg.dynamicSmemBytes = gv_smem<QT>(a.K, a.B);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_kernel<QT, EPI>, a);
}

cudaError_t launch_gemv(int epi, const GemvArgs &a, int num_sms, cudaStream_t st, bool pdl) {
    if (!gemv_fits(a.qt, a.K, a.B)) return cudaErrorInvalidValue;
    if (a.qt == Q8_0) {
        switch (epi) {
            case EPI_STORE: return gv_launch<Q8_0, EPI_STORE>(a, num_sms, st, pdl);
            case EPI_RESID: return gv_launch<Q8_0, EPI_RESID>(a, num_sms, st, pdl);
            case EPI_QKV: return gv_launch<Q8_0, EPI_QKV>(a, num_sms, st, pdl);
            case EPI_SWIGLU: return gv_launch<Q8_0, EPI_SWIGLU>(a, num_sms, st, pdl);
            case EPI_LOGITS: return gv_launch<Q8_0, EPI_LOGITS>(a, num_sms, st, pdl);
        }
    } else {
        switch (epi) {
            case EPI_STORE: return gv_launch<Q4_0, EPI_STORE>(a, num_sms, st, pdl);
            case EPI_RESID: return gv_launch<Q4_0, EPI_RESID>(a, num_sms, st, pdl);
            case EPI_QKV: return gv_launch<Q4_0, EPI_QKV>(a, num_sms, st, pdl);
            case EPI_SWIGLU: return gv_launch<Q4_0, EPI_SWIGLU>(a, num_sms, st, pdl);
            case EPI_LOGITS: return gv_launch<Q4_0, EPI_LOGITS>(a, num_sms, st, pdl);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace er
