// Block-quantized GEMV (batch 1..4) with fused prologue and epilogues.
//
// y_b = W x_b for every batch column b, W a repacked Q8_0 / Q4_0 matrix.  One
// weight pass serves all columns; every weight byte is read from HBM once.
//
// Work split ("stream-K"): the matrix is a list of U = R * UPR units (16 rows x
// 64 columns, contiguous in memory).  Warp w of the grid takes the contiguous
// unit range [w U / TW, (w+1) U / TW), so every warp streams the same number of
// bytes whatever the matrix shape.  A row group that lies inside one warp's
// range is finished by that warp; one shared by several warps is finished by
// the last of them to arrive (an atomic counter), which sums the warps'
// partial sums in warp order -- the result does not depend on timing.
//
// Streaming: each warp owns a ring of shared-memory slots filled by bulk async
// copies (cp.async.bulk, completion on an mbarrier).  The first slots are
// requested before griddepcontrol.wait, so weight traffic of this kernel
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

constexpr int GV_WARPS = 8;
constexpr int GV_SLOTS = 4;
constexpr int GV_MAXB = 4;

template <int QT>
struct GvCfg {
    static constexpr int UB = QTraits<QT>::unit_bytes;
    static constexpr int SU = QT == Q8_0 ? 4 : 8;  // units per slot
    static constexpr int SLOT = SU * UB;            // 4352 / 4608 bytes
    static constexpr int RING = GV_WARPS * GV_SLOTS * SLOT;
};

// shared-memory map: [mbarriers 256][rings][per-batch factors 64][reduce 256][operand]
constexpr int GV_OFF_RING = 256;
template <int QT>
constexpr int gv_off_fac() { return GV_OFF_RING + GvCfg<QT>::RING; }
template <int QT>
constexpr int gv_off_red() { return gv_off_fac<QT>() + 64; }
template <int QT>
constexpr int gv_off_xs() { return gv_off_red<QT>() + 256; }

__host__ __device__ inline int gv_nbp(int K) { return ((K / 32) + 1) & ~1; }
__host__ __device__ inline size_t gv_xs_bytes(int K, int B) { return (size_t)gv_nbp(K) * B * 128; }

// warp that owns unit u (U units over TW warps, every warp non-empty)
__device__ inline long long gv_owner(long long u, long long U, long long TW) { return ((u + 1) * TW - 1) / U; }
__device__ inline long long gv_start(long long w, long long U, long long TW) { return w * U / TW; }

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
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) last = atomicAdd(a.done, 1) == a.R - 1;
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
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
    uint8_t *xs = smem + gv_off_xs<QT>();

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long U = (long long)a.R * a.UPR;
    // working warps: at most one per unit, so every working warp's range is non-empty
    const long long TW = min((long long)gridDim.x * GV_WARPS, U);
    const long long gw = (long long)blockIdx.x * GV_WARPS + warp;
    const bool working = gw < TW;
    const long long ua = working ? gv_start(gw, U, TW) : U, ub = working ? gv_start(gw + 1, U, TW) : U;
    const int nunits = (int)(ub - ua);
    const int nslots = (nunits + C::SU - 1) / C::SU;
    uint64_t *wbar = bars + warp * GV_SLOTS;
    uint8_t *ring = smem + GV_OFF_RING + warp * GV_SLOTS * C::SLOT;
    const uint8_t *wsrc = a.W + (size_t)ua * C::UB;

    auto issue = [&](int k) {  // lane 0 only
        int s = k % GV_SLOTS;
        int n = min(C::SU, nunits - k * C::SU);
        uint32_t bytes = (uint32_t)n * C::UB;
        mbar_arrive_expect_tx(wbar + s, bytes);
        bulk_g2s(ring + s * C::SLOT, wsrc + (size_t)k * C::SLOT, bytes, wbar + s);
    };

    int issued = min(GV_SLOTS, nslots);
    if (lane == 0) {
        for (int s = 0; s < GV_SLOTS; ++s) mbar_init(wbar + s, 1);
        fence_mbar_init();
        for (int k = 0; k < issued; ++k) issue(k);
    }
    __syncwarp();

    // ---- everything above touches only constant weights; now wait for inputs
    pdl_wait();
    // a kernel earlier in the stream gave up on a wait: the state is already
    // invalid, so drain this warp's copies and stop (one read, shared by the CTA)
    if (tid == 0) red[63] = (*reinterpret_cast<volatile int *>(a.flags) & ER_FLAG_WAIT) ? 1.f : 0.f;
    __syncthreads();
    if (red[63] != 0.f) {
        if (lane == 0)
            for (int k = 0; k < issued; ++k) mbar_wait(wbar + k % GV_SLOTS, (k / GV_SLOTS) & 1);
        return;
    }
    pdl_launch_dependents();

    // ---- prologue: per batch column, sum of squares (norm) and max |x * gain|
    const int K = a.K, B = a.B;
    for (int b = 0; b < B; ++b) {
        float ss = 0.f, mx = 0.f;
        const float *x = a.x + (size_t)(a.b0 + b) * K;
        for (int k = tid; k < K; k += blockDim.x) {
            float v = x[k];
            ss += v * v;
            float w = a.gain ? v * a.gain[k] : v;
            mx = fmaxf(mx, fabsf(w));
        }
        for (int off = 16; off; off >>= 1) {
            ss += __shfl_xor_sync(0xffffffffu, ss, off);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        }
        if (lane == 0) {
            red[warp * 2] = ss;
            red[warp * 2 + 1] = mx;
        }
        __syncthreads();
        if (tid == 0) {
            float s = 0.f, m = 0.f;
            for (int w = 0; w < GV_WARPS; ++w) {
                s += red[w * 2];
                m = fmaxf(m, red[w * 2 + 1]);
            }
            int e = 0;
            if (m > 0.f && isfinite(m)) {
                int E;
                frexpf(m, &E);
                e = 15 - E;  // max |x| * 2^e in [2^14, 2^15)
            }
            float rstd = a.gain ? 1.f / sqrtf(s / (float)K + a.eps) : 1.f;
            fac[b] = ldexpf(rstd, -e);
            fac[GV_MAXB + b] = ldexpf(1.f, e);
        }
        __syncthreads();
    }
    // ---- operand: hi/lo fp16 in MMA B-fragment order, [kb][g < 2B][t] x 16 bytes
    {
        const int nbp = gv_nbp(K);
        const int npairs = nbp * 16;  // k pairs incl. padding block
        for (int b = 0; b < B; ++b) {
            const float sc = fac[GV_MAXB + b];
            const float *x = a.x + (size_t)(a.b0 + b) * K;
            for (int i = tid; i < npairs; i += blockDim.x) {
                int k = 2 * i;
                float v0 = 0.f, v1 = 0.f;
                if (k < K) {
                    v0 = x[k];
                    v1 = x[k + 1];
                    if (a.gain) {
                        v0 *= a.gain[k];
                        v1 *= a.gain[k + 1];
                    }
                    v0 *= sc;
                    v1 *= sc;
                }
                __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                __half l0 = __float2half_rn(v0 - __half2float(h0)), l1 = __float2half_rn(v1 - __half2float(h1));
                int kb = k >> 5, kk = k & 31, h = kk >> 4, kl = kk & 15;
                int t = (kl & 7) >> 1, reg = kl >> 3;
                size_t base = ((size_t)(kb * 2 * B + 2 * b) * 4 + t) * 16 + (h * 2 + reg) * 4;
                *reinterpret_cast<__half2 *>(xs + base) = __halves2half2(h0, h1);
                *reinterpret_cast<__half2 *>(xs + base + 64) = __halves2half2(l0, l1);  // g + 1: 4 t-slots of 16 B
            }
        }
    }
    __syncthreads();

    // ---- main loop
    const int g = lane >> 2, t = lane & 3;
    const bool has_b = g < 2 * B;
    const uint32_t xs_lane = smem_u32(xs) + (uint32_t)((g * 4 + t) * 16);
    const uint32_t xs_kb_stride = (uint32_t)(2 * B * 64);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

    float acc0 = 0.f, acc1 = 0.f;
    long long u = ua;
    int rg = (int)(ua / a.UPR);
    int j = (int)(ua - (long long)rg * a.UPR);
    int aborted_at = -1;

    auto finish = [&](int rgf, float v0, float v1) {
        long long r_lo = (long long)rgf * a.UPR, r_hi = r_lo + a.UPR;
        if (r_lo >= ua && r_hi <= ub) {
            gv_epilogue<EPI>(a, rgf, v0, v1, fac, lane);
            return;
        }
        // the warp's share is its first row group (slot 0) or its last (slot 1)
        const int slot = (ua >= r_lo) ? 0 : 1;
        float *p = a.part + ((size_t)gw * 2 + slot) * 64 + lane * 2;
        p[0] = v0;
        p[1] = v1;
        __threadfence();
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atomicAdd(a.cnt + rgf, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        long long wf = gv_owner(r_lo, U, TW), wl = gv_owner(r_hi - 1, U, TW);
        if (old == (int)(wl - wf)) {
            __threadfence();
            float s0 = 0.f, s1 = 0.f;
            for (long long w = wf; w <= wl; ++w) {
                const int sl = (gv_start(w, U, TW) >= r_lo) ? 0 : 1;
                const float *q = a.part + ((size_t)w * 2 + sl) * 64 + lane * 2;
                s0 += __ldcg(q);
                s1 += __ldcg(q + 1);
            }
            gv_epilogue<EPI>(a, rgf, s0, s1, fac, lane);
            if (lane == 0) a.cnt[rgf] = 0;
        }
    };

    for (int k = 0; k < nslots; ++k) {
        const int s = k % GV_SLOTS;
        if (!mbar_wait(wbar + s, (k / GV_SLOTS) & 1)) {
            if (lane == 0) atomicOr(a.flags, ER_FLAG_WAIT);
            aborted_at = k;
            break;
        }
        const int n = min(C::SU, nunits - k * C::SU);
        const uint32_t slot_base = smem_u32(ring + s * C::SLOT);
        for (int i = 0; i < n; ++i, ++u) {
            if (j == a.UPR) {
                finish(rg, acc0, acc1);
                acc0 = acc1 = 0.f;
                ++rg;
                j = 0;
            }
            const uint32_t unit_base = slot_base + i * C::UB;
            const uint32_t xa = xs_lane + (uint32_t)(2 * j) * xs_kb_stride;
            uint4 xb0 = make_uint4(0, 0, 0, 0), xb1 = make_uint4(0, 0, 0, 0);
            if (has_b) {
                xb0 = lds128(xa);
                xb1 = lds128(xa + xs_kb_stride);
            }
            uint2 sc = lds64(unit_base + QTraits<QT>::quant_bytes + g * 8);
            float c[4];
            uint32_t fa[4];
            if (QT == Q8_0) {
                uint4 q0 = lds128(unit_base + lane * 16);
                uint4 q1 = lds128(unit_base + 512 + lane * 16);
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
                uint4 q = lds128(unit_base + lane * 16);
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
            ++j;
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
        return;
    }
    if (nunits > 0) finish(rg, acc0, acc1);
}

// ---------------------------------------------------------------------------
size_t gemv_part_floats(int num_sms) { return (size_t)num_sms * GV_WARPS * 2 * 64; }

template <int QT>
static size_t gv_smem(int K, int B) { return gv_off_xs<QT>() + gv_xs_bytes(K, B); }

template <int QT, int EPI>
static cudaError_t gv_attr() {
    return cudaFuncSetAttribute(gemv_kernel<QT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

cudaError_t gemv_prepare() {
    cudaError_t e = cudaSuccess;
    cudaError_t r[10] = {gv_attr<Q8_0, EPI_STORE>(), gv_attr<Q8_0, EPI_RESID>(), gv_attr<Q8_0, EPI_QKV>(),
                         gv_attr<Q8_0, EPI_SWIGLU>(), gv_attr<Q8_0, EPI_LOGITS>(), gv_attr<Q4_0, EPI_STORE>(),
                         gv_attr<Q4_0, EPI_RESID>(), gv_attr<Q4_0, EPI_QKV>(), gv_attr<Q4_0, EPI_SWIGLU>(),
                         gv_attr<Q4_0, EPI_LOGITS>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) e = x;
    return e;
}

int gemv_max_cols(int qt, int K) {
    for (int b = GV_MAXB; b >= 1; --b)
        if (gemv_fits(qt, K, b)) return b;
    return 0;
}

bool gemv_fits(int qt, int K, int B) {
    if (B < 1 || B > GV_MAXB || K % 32) return false;
    size_t need = qt == Q8_0 ? gv_smem<Q8_0>(K, B) : gv_smem<Q4_0>(K, B);
    return need <= 227 * 1024;
}

template <int QT, int EPI>
static cudaError_t gv_launch(const GemvArgs &a, int num_sms, cudaStream_t st, bool pdl) {
    size_t smem = gv_smem<QT>(a.K, a.B);
    long long U = (long long)a.R * a.UPR;
    long long ctas = (U + GV_WARPS - 1) / GV_WARPS;
    if (ctas > num_sms) ctas = num_sms;
    if (ctas < 1) ctas = 1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(GV_WARPS * 32);
    cfg.dynamicSmemBytes = smem;
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
