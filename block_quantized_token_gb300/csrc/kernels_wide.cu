// Batched decode GEMV for 5..16 sequences: y[b] = W x[b] for every column b of
// the batch in one pass over the weights ("EdgeRunner Core Architecture"
// section 5.1 projections, decode of several sequences at once).
//
// With 16 columns the activation operand of a whole row (K up to 14336)
// does not fit in shared memory, so the matrix is cut into K-slices of 1024
// columns (16 units).  Slice s is worked by a contiguous group of CTAs, each
// taking a contiguous range of row groups; its warps take whole row groups in
// turn and stream the slice's units of each through their ring of bulk-copy
// slots (as the batch-1 GEMV does).  The unit's weights are turned into exact
// fp16 once and multiplied against NT n8 tiles of operand columns (hi and lo
// fp16 halves of each batch column).  A row group's slice partial (16 rows x
// 16 columns, already scaled) goes to global memory; the last slice to arrive
// at the row group's counter sums the partials in slice order and runs the
// epilogue, so the result does not depend on timing.
//
// Operand: per CTA, once, for its slice: every column's elements of the slice
// times the RMSNorm gain, scaled by one power of two per column (largest
// element in [2^14, 2^15)) and split into hi + lo fp16, in the MMA's B
// fragment order with each column's 16-byte chunks XOR-swizzled by the batch
// column (conflict-free 128-bit stores while it is built).  The slice's sum of
// squares of x per column goes to global memory for the finisher's 1/rms.
#include "gemv_core.cuh"

namespace er {

constexpr int GW_WARPS = 16;
constexpr int GW_SLOTS = 2;                   // ring slots per warp
constexpr int GW_SU = 4;                      // units per ring slot (one slot in flight while one is consumed)
constexpr int GW_SLICE_UNITS = 16;            // 1024 columns
constexpr int GW_NT = 4;                      // n8 tiles: 16 batch columns x (hi, lo)
constexpr int GW_BLOCK_BYTES = GW_NT * 8 * 64;  // operand bytes of one 32-element block
constexpr int GW_OFF_RING = 1024;             // after the mbarriers (room for 8 slots per warp)
static_assert(GW_WARPS * GW_SLOTS * 8 <= GW_OFF_RING, "mbarriers overlap the ring");

__host__ __device__ inline int gw_slices(int UPR) { return (UPR + GW_SLICE_UNITS - 1) / GW_SLICE_UNITS; }

template <int QT>
struct GwCfg {
    static constexpr int UB = GvCfg<QT>::UB;
    static constexpr int SU = GW_SU;
    static constexpr int SLOT = GW_SU * UB;  // 4352 / 2304 bytes
};
template <int QT>
constexpr int gw_off_operand() { return GW_OFF_RING + GW_WARPS * GW_SLOTS * GwCfg<QT>::SLOT; }
template <int QT>
constexpr int gw_smem() {
    // operand of 32 blocks, then per-column factors [16], per-(warp, segment) maxima [16][8], per-item sums of
    // squares [512]
    return gw_off_operand<QT>() + 2 * GW_SLICE_UNITS * GW_BLOCK_BYTES + 16 * 4 + GW_WARPS * 8 * 4 + 512 * 4 + 64;
}

// first CTA of slice s when C CTAs share S slices
__host__ __device__ inline int gw_cta0(int s, int S, int C) { return (int)((long long)s * C / S); }

// One unit (16 rows x 2 blocks): acc[j][0/1] += d(row) * (hi + lo sums) for tile j.
template <int QT>
__device__ inline void gw_unit(uint32_t ub, uint32_t xop, int lane, float (&acc)[GW_NT][2]) {
    const int g = lane >> 2;
    const uint2 sc = lds64(ub + GvCfg<QT>::QB + g * 8);
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    uint4 q0, q1;
    if (QT == Q8_0) {
        q0 = lds128(ub + lane * 16);
        q1 = lds128(ub + 512 + lane * 16);
    } else {
        q0 = lds128(ub + lane * 16);
    }
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        uint32_t a0[4], a1[4];
        if (QT == Q8_0) {
            const uint4 q = blk ? q1 : q0;
            q8_word_to_h2(q.x, a0[0], a0[1]);
            q8_word_to_h2(q.y, a0[2], a0[3]);
            q8_word_to_h2(q.z, a1[0], a1[1]);
            q8_word_to_h2(q.w, a1[2], a1[3]);
        } else {
            q4_word_to_h2(blk ? q0.z : q0.x, a0);
            q4_word_to_h2(blk ? q0.w : q0.y, a1);
        }
        const uint32_t sch = blk ? sc.y : sc.x;
        const float dg = h2f_lo(sch), dg8 = h2f_hi(sch);
        uint4 xb[GW_NT];
#pragma unroll
        for (int j = 0; j < GW_NT; ++j) xb[j] = lds128(xop + blk * GW_BLOCK_BYTES + j * 8 * 64);
#pragma unroll
        for (int j = 0; j < GW_NT; ++j) {
            float c[4];
            mma_16816(c, a0, xb[j].x, xb[j].y, zero4);
            mma_16816(c, a1, xb[j].z, xb[j].w, c);
            acc[j][0] = fmaf(dg, c[0] + c[1], acc[j][0]);
            acc[j][1] = fmaf(dg8, c[2] + c[3], acc[j][1]);
        }
    }
}

// Argmax part of the head epilogue for the whole batch of one row group, then
// one count per row group; the last row group writes the argmax of every column.
__device__ inline void gw_logits(const GemvArgs &a, int rg, const float (&v)[GW_NT][2], const float (&f)[GW_NT],
                                 int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < GW_NT; ++j) {
        const int b = 4 * j + t;
        unsigned long long key = 0;
        if (b < a.B) {
            const int r0 = 16 * rg + g, r1 = r0 + 8;
            const float v0 = v[j][0] * f[j], v1 = v[j][1] * f[j];
            float *y = a.y ? a.y + (size_t)b * a.N : nullptr;
            bool bad = false;
            if (r0 < a.N) {
                if (y) y[r0] = v0;
                bad |= !isfinite(v0);
                key = ((unsigned long long)float_order_key(isnan(v0) ? -INFINITY : v0) << 32) |
                      (0xFFFFFFFFu - (uint32_t)r0);
            }
            if (r1 < a.N) {
                if (y) y[r1] = v1;
                bad |= !isfinite(v1);
                const unsigned long long k1 = ((unsigned long long)float_order_key(isnan(v1) ? -INFINITY : v1) << 32) |
                                              (0xFFFFFFFFu - (uint32_t)r1);
                key = k1 > key ? k1 : key;
            }
            if (bad) atomicOr(a.flags, ER_FLAG_NONFINITE);
        }
        for (int off = 4; off < 32; off <<= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, off);
            key = o > key ? o : key;
        }
        if (b < a.B && g == 0 && key) atomicMax(a.amax + b, key);
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atom_add_acq_rel_gpu(a.done, 1) == a.R - 1;  // releases this warp's maxima
    last = __shfl_sync(0xffffffffu, last, 0);
    __syncwarp();
    if (last) {
        if (lane < a.B) {
            const unsigned long long k = atomicExch(a.amax + lane, 0ull);
            const int idx = k ? (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu)) : 0;
            if (a.argmax_out) a.argmax_out[lane] = idx;
        }
        if (lane == 0) *a.done = 0;
    }
}

template <int QT, int EPI>
__global__ void __launch_bounds__(GW_WARPS * 32, 1) gemv_wide_kernel(const GemvArgs a, float *wpart, float *wssq) {
    using C = GwCfg<QT>;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    uint8_t *op = smem + gw_off_operand<QT>();
    float *fac = reinterpret_cast<float *>(op + 2 * GW_SLICE_UNITS * GW_BLOCK_BYTES);
    float *wmax = fac + 16;  // [warp][i]: largest |x g| of segment warp + 16 i
    float *issq = wmax + GW_WARPS * 8;
    __shared__ int stop_s;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = gw_slices(a.UPR), nC = gridDim.x;
    int s = 0;
    while (s + 1 < S && gw_cta0(s + 1, S, nC) <= (int)blockIdx.x) ++s;
    const int c0 = gw_cta0(s, S, nC), ns = gw_cta0(s + 1, S, nC) - c0, j = blockIdx.x - c0;
    const int rg0 = (int)((long long)j * a.R / ns), rg1 = (int)((long long)(j + 1) * a.R / ns);
    const int ku0 = s * GW_SLICE_UNITS, nu = min(GW_SLICE_UNITS, a.UPR - ku0);
    const int nrg = rg1 - rg0;
    const int my_items = nrg > warp ? (nrg - warp + GW_WARPS - 1) / GW_WARPS : 0;  // rows groups rg0 + warp + 16 i
    const int spi = (nu + C::SU - 1) / C::SU;                                          // ring slots per row group

    uint64_t *wbar = bars + warp * GW_SLOTS;
    uint8_t *ring = smem + GW_OFF_RING + warp * GW_SLOTS * C::SLOT;
    int p_item = 0, p_slot = 0, issued = 0;
    auto issue_next = [&]() {  // lane 0
        if (p_item >= my_items) return;
        const int rg = rg0 + warp + GW_WARPS * p_item;
        const int u0 = p_slot * C::SU, cnt = min(C::SU, nu - u0);
        const uint32_t bytes = (uint32_t)cnt * C::UB;
        const unsigned sidx = (unsigned)issued % GW_SLOTS;
        mbar_arrive_expect_tx(wbar + sidx, bytes);
        bulk_g2s(ring + sidx * C::SLOT, a.W + ((size_t)rg * a.UPR + ku0 + u0) * C::UB, bytes, wbar + sidx);
        ++issued;
        if (++p_slot == spi) {
            p_slot = 0;
            ++p_item;
        }
    };
    if (lane == 0) {
        for (int i = 0; i < GW_SLOTS; ++i) mbar_init(wbar + i, 1);
        fence_mbar_init();
        for (int i = 0; i < GW_SLOTS; ++i) issue_next();
    }
    __syncwarp();

    // ---- everything above touches only constant weights; now wait for inputs
    pdl_wait();
    // an earlier kernel's give-up flag, read now and published after the operand build, so that
    // nothing waits for this load before then
    const int stop_r = tid == 0 ? (*reinterpret_cast<volatile int *>(a.flags) & ER_FLAG_WAIT) : 0;
    // zero the operand columns past the batch (their MMA results are never read, but must be finite)
    const int nbs = (nu * 64) / 32;  // blocks in this slice
    if (2 * a.B < GW_NT * 8)
        for (int i = tid; i < nbs * (GW_NT * 8 - 2 * a.B) * 16; i += blockDim.x) {
            const int per = (GW_NT * 8 - 2 * a.B) * 16, kb = i / per, r = i - kb * per;
            reinterpret_cast<uint32_t *>(op + kb * GW_BLOCK_BYTES + 2 * a.B * 64)[r] = 0u;
        }
    __syncthreads();
    // Warps read x in 512-byte segments of one column (lane l: elements 4l .. 4l + 3 of the segment),
    // so every load instruction touches 4 cache lines; the gain's elements are requested with them.
    // The 8 lanes of one 32-element block reduce its sum of squares by shuffles (lane 8i writes it),
    // and the warp reduces the segment's largest |x g| (lane 0 writes it): no shared-memory atomics.
    const int nel = nu * 64, spc = (nel + 127) / 128, nseg = a.B * spc;  // segments per column, in all
    float v[8][4];
    float4 gv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int seg = warp + GW_WARPS * i;
        const int b = seg / spc, e0 = (seg - b * spc) * 128 + 4 * lane;  // element of the slice
        const bool live = seg < nseg && e0 < nel;
        float4 x4 = make_float4(0.f, 0.f, 0.f, 0.f);
        gv[i] = make_float4(1.f, 1.f, 1.f, 1.f);
        if (live) {
            x4 = __ldcg(reinterpret_cast<const float4 *>(a.x + (size_t)b * a.K + ku0 * 64 + e0));
            if (a.gain) gv[i] = __ldg(reinterpret_cast<const float4 *>(a.gain + ku0 * 64 + e0));
        }
        v[i][0] = x4.x; v[i][1] = x4.y; v[i][2] = x4.z; v[i][3] = x4.w;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int seg = warp + GW_WARPS * i;
        if (seg >= nseg) break;  // warp-uniform
        const int b = seg / spc, e0 = (seg - b * spc) * 128 + 4 * lane;
        const bool live = e0 < nel;
        float ssq = 0.f, m = 0.f;
        if (live) {
#pragma unroll
            for (int c = 0; c < 4; ++c) ssq = fmaf(v[i][c], v[i][c], ssq);
            v[i][0] *= gv[i].x; v[i][1] *= gv[i].y; v[i][2] *= gv[i].z; v[i][3] *= gv[i].w;
#pragma unroll
            for (int c = 0; c < 4; ++c) m = fmaxf(m, fabsf(v[i][c]));
        }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, off);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        if (live && (lane & 7) == 0) issq[(e0 >> 5) * a.B + b] = ssq;
        if (lane == 0) wmax[warp * 8 + i] = isfinite(m) ? m : 0.f;
    }
    __syncthreads();
    if (tid < a.B) {
        float t = 0.f;
        for (int i = tid; i < nbs * a.B; i += a.B) t += issq[i];  // block order: deterministic
        wssq[s * 16 + tid] = t;  // every CTA of the slice writes the same value
        float mx = 0.f;  // the column's segments are tid * spc .. tid * spc + spc - 1
        for (int sg = tid * spc; sg < (tid + 1) * spc; ++sg) mx = fmaxf(mx, wmax[(sg % GW_WARPS) * 8 + sg / GW_WARPS]);
        int e = 0;
        if (mx > 0.f) {
            int E;
            frexpf(mx, &E);
            e = 15 - E;
        }
        fac[tid] = ldexpf(1.f, -e);
    }
    __syncthreads();
    // hi/lo split of each lane's two element pairs; pair p = 8h + 4reg + tt of a block is word 2h + reg of
    // 16-byte chunk tt of the column, stored at chunk tt ^ (b & 3)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int seg = warp + GW_WARPS * i;
        if (seg >= nseg) break;
        const int b = seg / spc, e0 = (seg - b * spc) * 128 + 4 * lane;
        if (e0 >= nel) continue;
        const float sc = 1.f / fac[b];
        uint8_t *area = op + (e0 >> 5) * GW_BLOCK_BYTES + 2 * b * 64;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int p = ((e0 & 31) >> 1) + q;
            const int off = (((p & 3) ^ (b & 3)) << 4) + ((((p >> 3) << 1) | ((p >> 2) & 1)) << 2);
            const float v0 = v[i][2 * q] * sc, v1 = v[i][2 * q + 1] * sc;
            const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
            const __half l0 = __float2half_rn(v0 - __half2float(h0));
            const __half l1 = __float2half_rn(v1 - __half2float(h1));
            *reinterpret_cast<__half2 *>(area + off) = __halves2half2(h0, h1);
            *reinterpret_cast<__half2 *>(area + 64 + off) = __halves2half2(l0, l1);
        }
    }
    if (tid == 0) stop_s = stop_r;
    __syncthreads();
    if (stop_s) {  // an earlier kernel gave up on a wait: drain and stop
        if (lane == 0)
            for (int k = 0; k < issued; ++k) mbar_wait(wbar + k % GW_SLOTS, (k / GW_SLOTS) & 1);
        return;
    }
    pdl_launch_dependents();

    // ---- consume: whole row groups, slice units in order
    const int g = lane >> 2, t = lane & 3;
    // column g of an n8 tile is batch column 4j + g / 2 (hi, lo): its chunk t sits at t ^ ((g / 2) & 3)
    const uint32_t xop = smem_u32(op) + (uint32_t)(g * 64 + ((t ^ ((g >> 1) & 3)) * 16));
    float fj[GW_NT];
#pragma unroll
    for (int jj = 0; jj < GW_NT; ++jj) fj[jj] = (4 * jj + t < a.B) ? fac[4 * jj + t] : 0.f;
    int k = 0;  // ring slot counter
    bool failed = false, fready = false;
    float f[GW_NT];
    for (int it = 0; it < my_items && !failed; ++it) {
        const int rg = rg0 + warp + GW_WARPS * it;
        float acc[GW_NT][2];
#pragma unroll
        for (int jj = 0; jj < GW_NT; ++jj) acc[jj][0] = acc[jj][1] = 0.f;
        for (int sl = 0; sl < spi; ++sl, ++k) {
            const unsigned sidx = (unsigned)k % GW_SLOTS;
            if (!mbar_wait(wbar + sidx, ((unsigned)k / GW_SLOTS) & 1u)) {
                if (lane == 0) atomicOr(a.flags, ER_FLAG_WAIT);
                failed = true;
                break;
            }
            const int u0 = sl * C::SU, cnt = min(C::SU, nu - u0);
            const uint32_t sb = smem_u32(ring + sidx * C::SLOT);
            if (cnt == C::SU) {  // full slot: units unrolled so their loads and MMAs overlap
#pragma unroll
                for (int i = 0; i < C::SU; ++i)
                    gw_unit<QT>(sb + i * C::UB, xop + (uint32_t)(2 * (u0 + i)) * GW_BLOCK_BYTES, lane, acc);
            } else {
                for (int i = 0; i < cnt; ++i)
                    gw_unit<QT>(sb + i * C::UB, xop + (uint32_t)(2 * (u0 + i)) * GW_BLOCK_BYTES, lane, acc);
            }
            // every lane's reads of the slot have returned (their values fed the
            // MMAs above) before lane 0 lets the next bulk copy overwrite it
            __syncwarp();
            if (lane == 0) issue_next();
        }
        if (failed) break;
        float v2[GW_NT][2];
        if (S == 1) {
#pragma unroll
            for (int jj = 0; jj < GW_NT; ++jj) {
                v2[jj][0] = acc[jj][0] * fj[jj];
                v2[jj][1] = acc[jj][1] * fj[jj];
            }
        } else {
            // this slice's partial [lane][tile][2]; the last slice to arrive sums them in slice order
            float4 *pp = reinterpret_cast<float4 *>(wpart + ((size_t)s * a.R + rg) * 256 + lane * 8);
            pp[0] = make_float4(acc[0][0] * fj[0], acc[0][1] * fj[0], acc[1][0] * fj[1], acc[1][1] * fj[1]);
            pp[1] = make_float4(acc[2][0] * fj[2], acc[2][1] * fj[2], acc[3][0] * fj[3], acc[3][1] * fj[3]);
            __syncwarp();
            int old = 0;
            if (lane == 0) old = atom_add_acq_rel_gpu(a.cnt + rg, 1);  // releases the partial
            old = __shfl_sync(0xffffffffu, old, 0);
            __syncwarp();
            if (old != S - 1) continue;
#pragma unroll
            for (int jj = 0; jj < GW_NT; ++jj) v2[jj][0] = v2[jj][1] = 0.f;
            for (int s0 = 0; s0 < S; s0 += 4) {  // 4 slices' loads in flight, added in slice order
                float4 pv[4][2];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (s0 + i < S) {
                        const float4 *qp =
                            reinterpret_cast<const float4 *>(wpart + ((size_t)(s0 + i) * a.R + rg) * 256 + lane * 8);
                        pv[i][0] = __ldcg(qp);
                        pv[i][1] = __ldcg(qp + 1);
                    }
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (s0 + i < S) {
                        const float4 p0 = pv[i][0], p1 = pv[i][1];
                        v2[0][0] += p0.x; v2[0][1] += p0.y; v2[1][0] += p0.z; v2[1][1] += p0.w;
                        v2[2][0] += p1.x; v2[2][1] += p1.y; v2[3][0] += p1.z; v2[3][1] += p1.w;
                    }
            }
            if (lane == 0) a.cnt[rg] = 0;
        }
        // 1/rms of each of this lane's columns, from the slices' sums of squares (slice order), once per
        // warp: every slice's CTA wrote its sums before the partials this warp has acquired
        if (!fready) {
#pragma unroll
            for (int jj = 0; jj < GW_NT; ++jj) {
                f[jj] = 1.f;
                const int bb = 4 * jj + t;
                if (a.gain && bb < a.B) {
                    float t2 = 0.f;
                    for (int ss = 0; ss < S; ++ss) t2 += __ldcg(wssq + ss * 16 + bb);
                    f[jj] = 1.f / sqrtf(t2 / (float)a.K + a.eps);
                }
            }
            fready = true;
        }
        if (EPI == EPI_LOGITS) {
            gw_logits(a, rg, v2, f, lane);
        } else {
#pragma unroll
            for (int jj = 0; jj < GW_NT; ++jj) {
                if (4 * jj >= a.B) break;
                GemvArgs a4 = a;
                a4.b0 = 4 * jj;
                a4.B = min(4, a.B - 4 * jj);
                gv_epilogue<EPI>(a4, rg, v2[jj][0], v2[jj][1], f[jj], lane);
            }
        }
    }
    if (failed && lane == 0)
        for (int kk = k; kk < issued; ++kk) mbar_wait(wbar + kk % GW_SLOTS, (kk / GW_SLOTS) & 1);
}

// ---------------------------------------------------------------------------
template <int QT, int EPI>
static cudaError_t gw_attr() {
    cudaError_t e = cudaFuncSetAttribute(gemv_wide_kernel<QT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         gw_smem<QT>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_wide_kernel<QT, EPI>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t gemv_wide_prepare() {
    if (cudaError_t e = gemv_tc_prepare(); e != cudaSuccess) return e;
    cudaError_t r[10] = {gw_attr<Q8_0, EPI_STORE>(), gw_attr<Q8_0, EPI_RESID>(), gw_attr<Q8_0, EPI_QKV>(),
                         gw_attr<Q8_0, EPI_SWIGLU>(), gw_attr<Q8_0, EPI_LOGITS>(), gw_attr<Q4_0, EPI_STORE>(),
                         gw_attr<Q4_0, EPI_RESID>(), gw_attr<Q4_0, EPI_QKV>(), gw_attr<Q4_0, EPI_SWIGLU>(),
                         gw_attr<Q4_0, EPI_LOGITS>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

bool gemv_wide_fits(int qt, int K, int B, int num_sms) {
    (void)qt;
    const int S = gw_slices(K / 64);
    // one thread per (block, column) of a slice; at least one CTA per slice
    return B >= 1 && B <= 16 && K % 64 == 0 && 32 * B <= GW_WARPS * 32 && S <= num_sms &&
           (K / 64 >= GW_SLICE_UNITS ? 2 * GW_SLICE_UNITS * B : 2 * (K / 64) * B) <= GW_WARPS * 32;
}

// both batched kernels: one 16 x 16 partial per slice and row group (the
// tcgen05 kernel writes one even for a single slice)
size_t gemv_wide_part_floats(int R, int K) { return (size_t)gw_slices(K / 64) * R * 256; }
size_t gemv_wide_ssq_floats(int K) { return (size_t)gw_slices(K / 64) * 16; }

template <int QT, int EPI>
static cudaError_t gw_launch(const GemvArgs &a, float *wpart, float *wssq, int num_sms, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)num_sms);
    cfg.blockDim = dim3(GW_WARPS * 32);
    cfg.dynamicSmemBytes = gw_smem<QT>();
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_wide_kernel<QT, EPI>, a, wpart, wssq);
}

// Which batched kernel: the tcgen05 one from 2^18 units (about 285 MB of Q8_0
// weights) up, where a CTA's warpgroups each stream many full 128-row tiles;
// below that its per-tile fixed costs (prologue, one stage handoff per unit,
// the finisher's tail) outweigh the faster tensor cores, measured on GB300.
bool gemv_wide_uses_tc(int variant, int R, int UPR) {
    if (variant == WIDE_MMA_SYNC) return false;
    if (variant == WIDE_TCGEN05) return true;
    return (long long)R * UPR >= (1ll << 18);
}

cudaError_t launch_gemv_wide(int epi, const GemvArgs &a, float *wpart, float *wssq, int num_sms, cudaStream_t st,
                             bool pdl, int variant) {
    if (gemv_wide_uses_tc(variant, a.R, a.UPR)) return launch_gemv_tc(epi, a, wpart, wssq, num_sms, st, pdl);
    if (!gemv_wide_fits(a.qt, a.K, a.B, num_sms) || a.b0 != 0) return cudaErrorInvalidValue;
    if (a.qt == Q8_0) {
        switch (epi) {
            case EPI_STORE: return gw_launch<Q8_0, EPI_STORE>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_RESID: return gw_launch<Q8_0, EPI_RESID>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_QKV: return gw_launch<Q8_0, EPI_QKV>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_SWIGLU: return gw_launch<Q8_0, EPI_SWIGLU>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_LOGITS: return gw_launch<Q8_0, EPI_LOGITS>(a, wpart, wssq, num_sms, st, pdl);
        }
    } else {
        switch (epi) {
            case EPI_STORE: return gw_launch<Q4_0, EPI_STORE>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_RESID: return gw_launch<Q4_0, EPI_RESID>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_QKV: return gw_launch<Q4_0, EPI_QKV>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_SWIGLU: return gw_launch<Q4_0, EPI_SWIGLU>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_LOGITS: return gw_launch<Q4_0, EPI_LOGITS>(a, wpart, wssq, num_sms, st, pdl);
        }
    }
    return cudaErrorInvalidValue;
}

// this translation unit's copy of the bounded-wait limit
cudaError_t set_wait_limit_wide(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace er
