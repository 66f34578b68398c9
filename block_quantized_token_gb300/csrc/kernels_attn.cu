// Split-K GQA decode attention over the fp16 KV cache, with the cross-chunk
// combine done by the last CTA to finish (no second launch, no spinning).
//
// CTA (chunk c, KV head kvh, sequence b) scores the G = H / KV query heads of
// the group against cache rows [c*CH, min((c+1)*CH, pos+1)) and keeps, per head,
// the running max m, the running sum l = sum exp(s - m) and o = sum exp(s - m) v
// (online softmax).  Rows of one head are contiguous ([head][position][dim]), so
// the four warps stream consecutive rows with 128-bit loads, one iteration
// ahead of the arithmetic.  Rows below `pos` were written by earlier steps, so
// the first iteration's rows are requested before griddepcontrol.wait; only the
// row at `pos` (written by the QKV kernel of this step) waits for it.  The CTA
// that completes a (b, kvh) group last merges the chunks:
//   M = max_c m_c,  o = sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c
// ("EdgeRunner Core Architecture" section 5.2: scale 1/sqrt(hd), causal, a
// query at position p attends rows 0..p; query head h reads KV head h / G).
#include "common.cuh"
#include "internal.h"

namespace er {

constexpr int AT_WARPS = 4;
constexpr int AT_UNROLL = 4;
constexpr int AT_COMBINE_SMEM = 48 * 1024;  // staging for the last CTA's merge

template <int HD>
struct AtCfg {
    static constexpr int LPR = HD / 8;    // lanes per row (8 halves each)
    static constexpr int RPW = 32 / LPR;  // rows per warp step
    static constexpr int RPI = AT_WARPS * RPW * AT_UNROLL;  // rows per CTA iteration
};

__device__ inline void merge_state(float &m, float &l, float *acc, float m2, float l2, const float *acc2) {
    float mn = fmaxf(m, m2);
    if (mn == -INFINITY) return;
    float c1 = exp2f(m - mn), c2 = exp2f(m2 - mn);
    l = l * c1 + l2 * c2;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = acc[i] * c1 + acc2[i] * c2;
    m = mn;
}

template <int HD, int G>
__global__ void __launch_bounds__(AT_WARPS * 32) attn_kernel(const AttnArgs a) {
    using C = AtCfg<HD>;
    extern __shared__ float stage[];  // S * G * (HD + 2) floats, used by the last CTA
    __shared__ float sm_m[AT_WARPS][G], sm_l[AT_WARPS][G];
    __shared__ float sm_o[AT_WARPS][G][HD];
    __shared__ int sm_last;

    const int c = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rw = lane / C::LPR, dl = (lane % C::LPR) * 8;

    // positions are inputs of the whole step: stable before the wait
    const int pos = a.positions[b];
    const int T = (pos >= 0 && pos < a.cap) ? pos + 1 : 0;
    const int r0 = c * a.CH, r1 = min(r0 + a.CH, T);
    const size_t head_off = (((size_t)b * a.L + a.layer) * a.KV + kvh) * (size_t)a.cap * HD;
    const __half *Kb = a.kc + head_off + dl;
    const __half *Vb = a.vc + head_off + dl;
    const int qd = a.H * HD;
    const int base0 = r0 + warp * C::RPW + rw;  // this lane's first row

    uint4 kr[AT_UNROLL], vr[AT_UNROLL];
#pragma unroll
    for (int u = 0; u < AT_UNROLL; ++u) {
        const int row = base0 + u * AT_WARPS * C::RPW;
        kr[u] = vr[u] = make_uint4(0, 0, 0, 0);
        if (row < r1 && row != pos) {
            kr[u] = *reinterpret_cast<const uint4 *>(Kb + (size_t)row * HD);
            vr[u] = *reinterpret_cast<const uint4 *>(Vb + (size_t)row * HD);
        }
    }

    pdl_wait();
    pdl_launch_dependents();

#pragma unroll
    for (int u = 0; u < AT_UNROLL; ++u) {
        const int row = base0 + u * AT_WARPS * C::RPW;
        if (row < r1 && row == pos) {
            kr[u] = *reinterpret_cast<const uint4 *>(Kb + (size_t)row * HD);
            vr[u] = *reinterpret_cast<const uint4 *>(Vb + (size_t)row * HD);
        }
    }

    // q of the group, pre-scaled so scores are in log2 units
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);
    float qv[G][8];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        const float4 *qp = reinterpret_cast<const float4 *>(a.q + (size_t)b * qd + (kvh * G + gi) * HD + dl);
        float4 x0 = qp[0], x1 = qp[1];
        qv[gi][0] = x0.x * qscale; qv[gi][1] = x0.y * qscale; qv[gi][2] = x0.z * qscale; qv[gi][3] = x0.w * qscale;
        qv[gi][4] = x1.x * qscale; qv[gi][5] = x1.y * qscale; qv[gi][6] = x1.z * qscale; qv[gi][7] = x1.w * qscale;
    }
    float m[G], l[G], acc[G][8];
#pragma unroll
    for (int gi = 0; gi < G; ++gi) {
        m[gi] = -INFINITY;
        l[gi] = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[gi][i] = 0.f;
    }

    for (int base = base0; base - rw < r1; base += C::RPI) {
        // next iteration's rows first, so their loads overlap this iteration's math
        uint4 kn[AT_UNROLL], vn[AT_UNROLL];
#pragma unroll
        for (int u = 0; u < AT_UNROLL; ++u) {
            const int row = base + C::RPI + u * AT_WARPS * C::RPW;
            kn[u] = vn[u] = make_uint4(0, 0, 0, 0);
            if (row < r1) {
                kn[u] = *reinterpret_cast<const uint4 *>(Kb + (size_t)row * HD);
                vn[u] = *reinterpret_cast<const uint4 *>(Vb + (size_t)row * HD);
            }
        }
        float s[AT_UNROLL][G];
#pragma unroll
        for (int u = 0; u < AT_UNROLL; ++u) {
            const bool ok = base + u * AT_WARPS * C::RPW < r1;
            const __half2 *kh = reinterpret_cast<const __half2 *>(&kr[u]);
            float kf[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float2 f = __half22float2(kh[i]);
                kf[2 * i] = f.x;
                kf[2 * i + 1] = f.y;
            }
#pragma unroll
            for (int gi = 0; gi < G; ++gi) {
                float d = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) d = fmaf(qv[gi][i], kf[i], d);
#pragma unroll
                for (int off = 1; off < C::LPR; off <<= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
                s[u][gi] = ok ? d : -INFINITY;
            }
        }
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            float mn = m[gi];
#pragma unroll
            for (int u = 0; u < AT_UNROLL; ++u) mn = fmaxf(mn, s[u][gi]);
            if (mn == -INFINITY) continue;
            const float corr = exp2f(m[gi] - mn);
            l[gi] *= corr;
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[gi][i] *= corr;
            m[gi] = mn;
#pragma unroll
            for (int u = 0; u < AT_UNROLL; ++u) {
                const float p = exp2f(s[u][gi] - mn);
                l[gi] += p;
                const __half2 *vh = reinterpret_cast<const __half2 *>(&vr[u]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float2 f = __half22float2(vh[i]);
                    acc[gi][2 * i] = fmaf(p, f.x, acc[gi][2 * i]);
                    acc[gi][2 * i + 1] = fmaf(p, f.y, acc[gi][2 * i + 1]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < AT_UNROLL; ++u) {
            kr[u] = kn[u];
            vr[u] = vn[u];
        }
    }

    // merge the RPW row slots of the warp (lanes with the same dl)
#pragma unroll
    for (int off = C::LPR; off < 32; off <<= 1) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            float m2 = __shfl_xor_sync(0xffffffffu, m[gi], off);
            float l2 = __shfl_xor_sync(0xffffffffu, l[gi], off);
            float a2[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a2[i] = __shfl_xor_sync(0xffffffffu, acc[gi][i], off);
            merge_state(m[gi], l[gi], acc[gi], m2, l2, a2);
        }
    }
    if (rw == 0) {
#pragma unroll
        for (int gi = 0; gi < G; ++gi) {
            if (dl == 0) {
                sm_m[warp][gi] = m[gi];
                sm_l[warp][gi] = l[gi];
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) sm_o[warp][gi][dl + i] = acc[gi][i];
        }
    }
    __syncthreads();

    // CTA partial -> scratch: per (b, kvh, c, gi): [m, l, o[HD]]
    const int group = b * a.KV + kvh;
    float *part = a.part + ((size_t)group * a.S + c) * G * (HD + 2);
    for (int idx = tid; idx < G * (HD + 2); idx += blockDim.x) {
        const int gi = idx / (HD + 2), j = idx % (HD + 2);
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < AT_WARPS; ++w) M = fmaxf(M, sm_m[w][gi]);
        float v = (j == 0) ? M : 0.f;
        if (j > 0 && M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < AT_WARPS; ++w) {
                const float e = exp2f(sm_m[w][gi] - M);
                v += (j == 1 ? sm_l[w][gi] : sm_o[w][gi][j - 2]) * e;
            }
        }
        part[idx] = v;
    }
    __syncthreads();
    if (tid == 0) sm_last = atom_add_acq_rel_gpu(a.cnt + group, 1) == a.S - 1;  // releases the CTA's partial
    __syncthreads();
    if (!sm_last) return;

    // last CTA of the group: stage every chunk's partial, then merge in chunk order
    const float *gp = a.part + (size_t)group * a.S * G * (HD + 2);
    const int nf = a.S * G * (HD + 2);
    for (int i = tid; i < nf; i += blockDim.x) stage[i] = __ldcg(gp + i);
    __syncthreads();
    for (int idx = tid; idx < G * HD; idx += blockDim.x) {
        const int gi = idx / HD, d = idx % HD;
        float M = -INFINITY;
        for (int cc = 0; cc < a.S; ++cc) M = fmaxf(M, stage[(cc * G + gi) * (HD + 2)]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int cc = 0; cc < a.S; ++cc) {
                const float *pc = stage + (cc * G + gi) * (HD + 2);
                const float e = exp2f(pc[0] - M);
                L += pc[1] * e;
                O += pc[2 + d] * e;
            }
        }
        a.o[(size_t)b * qd + (kvh * G + gi) * HD + d] = (L > 0.f) ? O / L : 0.f;
    }
    if (tid == 0) a.cnt[group] = 0;
}

void attention_plan(int hd, int KV, int B, int cap, int num_sms, int *S, int *CH) {
    const int per_iter = AT_WARPS * (32 / (hd / 8)) * AT_UNROLL;  // rows one CTA covers per loop pass
    long long groups = (long long)KV * B;
    long long want = (4LL * num_sms + groups - 1) / groups;  // ~4 CTAs per SM
    long long max_chunks = (cap + per_iter - 1) / per_iter;
    long long s = want < max_chunks ? want : max_chunks;
    // the last CTA stages every chunk's partial in shared memory (G <= 8)
    const long long fit = AT_COMBINE_SMEM / (8LL * (hd + 2) * 4);
    if (s > fit) s = fit;
    if (s < 1) s = 1;
    int ch = (int)((cap + s - 1) / s);
    ch = (ch + per_iter - 1) / per_iter * per_iter;
    *CH = ch;
    *S = (cap + ch - 1) / ch;
}

template <int HD, int G>
static cudaError_t at_launch(const AttnArgs &a, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(a.S, a.KV, a.B);
    cfg.blockDim = dim3(AT_WARPS * 32);
    cfg.dynamicSmemBytes = (size_t)a.S * G * (HD + 2) * sizeof(float);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, attn_kernel<HD, G>, a);
}

template <int HD>
static cudaError_t at_launch_g(const AttnArgs &a, cudaStream_t st, bool pdl) {
    switch (a.H / a.KV) {
        case 1: return at_launch<HD, 1>(a, st, pdl);
        case 2: return at_launch<HD, 2>(a, st, pdl);
        case 3: return at_launch<HD, 3>(a, st, pdl);
        case 4: return at_launch<HD, 4>(a, st, pdl);
        case 5: return at_launch<HD, 5>(a, st, pdl);
        case 6: return at_launch<HD, 6>(a, st, pdl);
        case 7: return at_launch<HD, 7>(a, st, pdl);
        case 8: return at_launch<HD, 8>(a, st, pdl);
    }
    return cudaErrorInvalidValue;
}

template <int HD, int G>
static cudaError_t at_attr() {
    return cudaFuncSetAttribute(attn_kernel<HD, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                cudaSharedmemCarveoutMaxShared);
}

cudaError_t attention_prepare() {
    cudaError_t r[16] = {at_attr<64, 1>(),  at_attr<64, 2>(),  at_attr<64, 3>(),  at_attr<64, 4>(),
                         at_attr<64, 5>(),  at_attr<64, 6>(),  at_attr<64, 7>(),  at_attr<64, 8>(),
                         at_attr<128, 1>(), at_attr<128, 2>(), at_attr<128, 3>(), at_attr<128, 4>(),
                         at_attr<128, 5>(), at_attr<128, 6>(), at_attr<128, 7>(), at_attr<128, 8>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

cudaError_t launch_attention(const AttnArgs &a, cudaStream_t st, bool pdl) {
    if ((size_t)a.S * (a.H / a.KV) * (a.hd + 2) * sizeof(float) > AT_COMBINE_SMEM) return cudaErrorInvalidValue;
    if (a.hd == 64) return at_launch_g<64>(a, st, pdl);
    if (a.hd == 128) return at_launch_g<128>(a, st, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace er
