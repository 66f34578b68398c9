// Batched decode GEMV for 5..16 sequences on the tcgen05 tensor cores:
// y[b] = W x[b] for every column b of the batch in one pass over the weights
// ("EdgeRunner Core Architecture" section 5.1 projections, decode of several
// sequences at once), fp32 accumulators in tensor memory (TMEM).  The same
// operation as the mma.sync kernel of kernels_wide.cu, which launch_gemv_wide
// picks for matrices below 2^18 units (see there).
//
// The matrix is cut into K-slices of 1024 columns (16 units).  Slice s is
// worked by a contiguous group of CTAs, each taking a contiguous range of row
// groups, split in two halves for the CTA's two warpgroups.  A warpgroup works
// tiles of 8 row groups (128 rows, the MMA's M), one unit (2 blocks) per ring
// stage:
//   - its producer warp bulk-copies the tile's 8 row groups of each unit into
//     a ring of stages (one copy per lane, one mbarrier per stage);
//   - its 128 row threads (thread = one weight row = one TMEM lane) turn the
//     unit's 64 elements of their row into exact fp16 and store them to TMEM
//     (the MMA's A operand), then signal the MMA warp;
//   - its MMA warp issues, per block, D = A [Bhi; Blo] over the block's two
//     16-wide K steps (M = 128, N = 32: hi and lo fp16 halves of the 16 batch
//     columns) and commits to the stage's mbarrier;
//   - one stage later the row threads read the two blocks' D back and add
//     d(row, block) * (D hi + D lo) to their accumulators, so the per-block
//     scale never enters the tensor core;
//   - after a tile, the row threads store the slice's partial of their rows
//     and count the tile in; its epilogue warp counts each row group's slice
//     in, and the last slice to arrive sums the partials in slice order and
//     runs the epilogue, so the result does not depend on timing.
// One tcgen05.mma of this kind costs about the same time up to N = 128, so the
// hi and lo halves share one instruction: each 128 x 32 block takes 2 MMAs.
//
// Operand: per CTA, once, for its slice: every column's elements of the slice
// times the RMSNorm gain, scaled by one power of two per column (largest
// element in [2^14, 2^15)) and split into hi + lo fp16, stored K-major with
// the 128-byte swizzle (row n of an 8-row atom keeps its 16-byte chunk c at
// chunk c ^ n), the 16 lo rows right after the 16 hi rows.  The slice's sum
// of squares of x per column goes to global memory for the finisher's 1/rms.
#include "gemv_core.cuh"

namespace er {

constexpr int TW_WG = 2;                          // row warpgroups per CTA
constexpr int TW_EPI = 2;                         // epilogue warps per warpgroup (alternate tiles)
// warps 0-1: producers, 2-3: MMA issuers, 4-11: rows, 12-15: epilogue
constexpr int TW_THREADS = (4 + 4 * TW_WG + TW_EPI * TW_WG) * 32;
constexpr int TW_SLICE_UNITS = 16;                // 1024 columns
constexpr int TW_SU = 1;                          // units per ring stage (2 blocks)
constexpr int TW_NS = 8;                          // ring stages per warpgroup
constexpr int TW_NBUF = 2;                        // TMEM stage buffers (A and D) per warpgroup
constexpr int TW_TMEM_COLS = 512;                 // per warpgroup (256): A 2 x 32 columns, D 2 x 64 columns
constexpr int TW_ATOM_BYTES = 4096;               // 64 K elements: hi tile 16 x 128 B, lo tile 16 x 128 B
constexpr int TW_OPND_BYTES = TW_SLICE_UNITS * TW_ATOM_BYTES;

__host__ __device__ inline int tw_slices(int UPR) { return (UPR + TW_SLICE_UNITS - 1) / TW_SLICE_UNITS; }

// bytes of one row group in a stage: its unit, rounded up to 128 and then
// moved 16 bytes on, so the 8 row groups of a tile start in 8 different
// 16-byte bank groups
template <int QT>
constexpr int tw_rgs() { return (TW_SU * QTraits<QT>::unit_bytes + 127) / 128 * 128 + 16; }
template <int QT>
constexpr int tw_stage() { return 8 * tw_rgs<QT>(); }
template <int QT>
constexpr int tw_off_bars() { return TW_OPND_BYTES + TW_WG * TW_NS * tw_stage<QT>(); }
constexpr int TW_BARS_PER_WG = 2 * TW_NS + 2 * TW_NBUF;  // full, empty, afull, dfull
template <int QT>
constexpr int tw_off_misc() { return tw_off_bars<QT>() + TW_WG * TW_BARS_PER_WG * 8; }
// misc: factors [16], column maxima [16], per-item sums of squares [512], TMEM
// address, stop, abort, tiles done per warpgroup [2]
constexpr int TW_MISC_BYTES = 16 * 4 + 16 * 4 + 512 * 4 + 32;
template <int QT>
constexpr int tw_smem() { return tw_off_misc<QT>() + TW_MISC_BYTES + 1024; }  // + alignment of the base

// first CTA of slice s when C CTAs share S slices
__host__ __device__ inline int tw_cta0(int s, int S, int C) { return (int)((long long)s * C / S); }

// ---------------------------------------------------------------------------
// tcgen05 wrappers
// ---------------------------------------------------------------------------
ER_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
ER_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row atoms of
// 1024 bytes (stride between atoms 1024), descriptor version 1
ER_DEV uint64_t tc_desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor, kind::f16: fp16 A and B (both K-major), fp32 D, N = 32, M = 128
constexpr uint32_t TW_IDESC = (1u << 4) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

// D[tmem] (+)= A[tmem] * B[smem]^T
ER_DEV void tc_mma_ts(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %3, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t}" ::"r"(d),
        "r"(a), "l"(bdesc), "r"(accumulate), "r"(TW_IDESC)
        : "memory");
}
// the mbarrier arrives once every MMA this thread issued before has completed
ER_DEV void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
// 32 consecutive 32-bit columns of this thread's lane (no wait)
ER_DEV void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]) : "memory");
}
ER_DEV void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
ER_DEV void tc_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];" : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]) : "r"(taddr) : "memory");
}
// waits for the loads above; the registers pass through so no use moves ahead of it
ER_DEV void tc_wait_ld(uint32_t (&a)[32], uint32_t (&b)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]), "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]), "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]), "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]), "+r"(b[30]), "+r"(b[31]) : : "memory");
}
ER_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
ER_DEV unsigned ld_acquire_cta(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}
ER_DEV void red_add_release_cta(unsigned *p, unsigned v) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}
ER_DEV uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------
// one row's 32 elements of one block as 16 fp16 pairs, TMEM column order
// (column c holds elements 2c, 2c+1).  In the unit layout the row's elements
// sit in the 16-byte chunks t = 0..3 of fragment row g: word x of chunk t
// holds elements (2t, 2t+1) of half 0, y (8+2t, 9+2t) of half 0, z and w the
// same of half 1, and within each word bytes 0-1 belong to row g, 2-3 to row
// g + 8.
// ---------------------------------------------------------------------------
template <int O>
ER_DEV void tw_q8_block(uint32_t base, uint32_t sel, uint32_t (&col)[32]) {
    const uint32_t k1152 = 0x64806480u;  // half2(1024 + 128): stored bytes are q ^ 0x80
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint4 c = lds128(base + 16 * t);
        col[O + t] = h2_sub(prmt(c.x, 0x64646464u, sel), k1152);
        col[O + 4 + t] = h2_sub(prmt(c.y, 0x64646464u, sel), k1152);
        col[O + 8 + t] = h2_sub(prmt(c.z, 0x64646464u, sel), k1152);
        col[O + 12 + t] = h2_sub(prmt(c.w, 0x64646464u, sel), k1152);
    }
}
// Q4_0: word 2b + h of chunk t holds the 8 nibbles of block b, half h; nibbles
// p = upper, upper + 4 are elements (2t, 2t+1) and p = upper + 2, upper + 6
// elements (8+2t, 9+2t) of the row (upper = row >= 8).  Shifting the word
// right by 4 * upper brings the row's nibbles to bits 0-3 / 16-19 (and, after
// a further 8, the second pair).
ER_DEV uint32_t tw_q4_pair(uint32_t w) {
    return h2_sub(lop3_and_or(w, 0x000F000Fu, 0x64006400u), 0x64086408u);  // (1024 + n) - (1024 + 8)
}
// one unit (both blocks) of the row: columns 0-15 block 0, 16-31 block 1
template <int QT>
ER_DEV void tw_unit_cols(uint32_t base, uint32_t sel, uint32_t sh, uint32_t (&col)[32]) {
    if (QT == Q8_0) {
        tw_q8_block<0>(base, sel, col);
        tw_q8_block<16>(base + 512, sel, col);
    } else {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint4 c = lds128(base + 16 * t);
            const uint32_t w[4] = {c.x >> sh, c.y >> sh, c.z >> sh, c.w >> sh};
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                col[16 * b + t] = tw_q4_pair(w[2 * b]);
                col[16 * b + 4 + t] = tw_q4_pair(w[2 * b] >> 8);
                col[16 * b + 8 + t] = tw_q4_pair(w[2 * b + 1]);
                col[16 * b + 12 + t] = tw_q4_pair(w[2 * b + 1] >> 8);
            }
        }
    }
}

constexpr int TW_NT = 4;  // groups of 4 batch columns in the finisher's lane mapping

// Head epilogue for the whole batch of one row group: the logits are stored
// and each lane keeps, per column, the largest key (value, then lowest row)
// of the rows it has seen; tw_logits_flush merges them once per warp.
__device__ inline void tw_logits(const GemvArgs &a, int rg, const float (&v)[TW_NT][2], const float (&f)[TW_NT],
                                 int lane, unsigned long long (&kbest)[TW_NT]) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < TW_NT; ++j) {
        const int b = 4 * j + t;
        if (b >= a.B) continue;
        const int r0 = 16 * rg + g, r1 = r0 + 8;
        const float v0 = v[j][0] * f[j], v1 = v[j][1] * f[j];
        float *y = a.y ? a.y + (size_t)b * a.N : nullptr;
        bool bad = false;
        unsigned long long key = kbest[j];
        if (r0 < a.N) {
            if (y) y[r0] = v0;
            bad |= !isfinite(v0);
            const unsigned long long k0 = ((unsigned long long)float_order_key(isnan(v0) ? -INFINITY : v0) << 32) |
                                          (0xFFFFFFFFu - (uint32_t)r0);
            key = k0 > key ? k0 : key;
        }
        if (r1 < a.N) {
            if (y) y[r1] = v1;
            bad |= !isfinite(v1);
            const unsigned long long k1 = ((unsigned long long)float_order_key(isnan(v1) ? -INFINITY : v1) << 32) |
                                          (0xFFFFFFFFu - (uint32_t)r1);
            key = k1 > key ? k1 : key;
        }
        kbest[j] = key;
        if (bad) atomicOr(a.flags, ER_FLAG_NONFINITE);
    }
}

// After this warp's `n` row groups: each column's largest key goes to amax,
// then the count; the warp that brings the count to R writes the argmax of
// every column and resets the counters.
__device__ inline void tw_logits_flush(const GemvArgs &a, unsigned long long (&kbest)[TW_NT], int n, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int j = 0; j < TW_NT; ++j) {
        unsigned long long key = kbest[j];
        for (int off = 4; off < 32; off <<= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, off);
            key = o > key ? o : key;
        }
        const int b = 4 * j + t;
        if (b < a.B && g == 0 && key) atomicMax(a.amax + b, key);
    }
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atom_add_acq_rel_gpu(a.done, n) == a.R - n;  // releases this warp's maxima
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

// 1/rms of this lane's columns t, 4 + t, 8 + t, 12 + t from the slices' sums
// of squares (slice order); 1 without a norm.  Valid once every slice's CTA
// has passed its prologue, which a row group's final count implies.
__device__ inline void tw_colscale(const GemvArgs &a, int S, const float *wssq, int lane, float (&f)[TW_NT]) {
    const int t = lane & 3;
#pragma unroll
    for (int jj = 0; jj < TW_NT; ++jj) {
        f[jj] = 1.f;
        const int bb = 4 * jj + t;
        if (a.gain && bb < a.B) {
            float t2 = 0.f;
            for (int ss = 0; ss < S; ++ss) t2 += __ldcg(wssq + ss * 16 + bb);
            f[jj] = 1.f / sqrtf(t2 / (float)a.K + a.eps);
        }
    }
}

// The last slice to arrive at row groups rg[0] and (if rg[1] >= 0) rg[1]: sum
// each one's slice partials in slice order, then the epilogue (for the head:
// logits and per-lane maxima, see tw_logits_flush).  A partial is stored
// finisher-lane-major: lane 4g + t's 8 values (rows g and g + 8 of columns
// t, 4 + t, 8 + t, 12 + t, as [column group][row]) are contiguous, so a lane
// reads two float4 per slice; both row groups' loads for 2 slices at a time
// are in flight together.
template <int EPI>
__device__ inline void tw_finish2(const GemvArgs &a, const int (&rg)[2], int S, const float *wpart,
                                  const float (&f)[TW_NT], int lane, unsigned long long (&kbest)[TW_NT]) {
    float v2[2][TW_NT][2];
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
        for (int jj = 0; jj < TW_NT; ++jj) v2[k][jj][0] = v2[k][jj][1] = 0.f;
    for (int s0 = 0; s0 < S; s0 += 2) {
        float4 pv[2][2][2];
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (rg[k] >= 0 && s0 + i < S) {
                    const float4 *p =
                        reinterpret_cast<const float4 *>(wpart + ((size_t)(s0 + i) * a.R + rg[k]) * 256 + lane * 8);
                    pv[k][i][0] = __ldcg(p);
                    pv[k][i][1] = __ldcg(p + 1);
                }
#pragma unroll
        for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int i = 0; i < 2; ++i)
                if (rg[k] >= 0 && s0 + i < S) {
                    v2[k][0][0] += pv[k][i][0].x; v2[k][0][1] += pv[k][i][0].y;
                    v2[k][1][0] += pv[k][i][0].z; v2[k][1][1] += pv[k][i][0].w;
                    v2[k][2][0] += pv[k][i][1].x; v2[k][2][1] += pv[k][i][1].y;
                    v2[k][3][0] += pv[k][i][1].z; v2[k][3][1] += pv[k][i][1].w;
                }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        if (rg[k] < 0) continue;
        if (EPI == EPI_LOGITS) {
            tw_logits(a, rg[k], v2[k], f, lane, kbest);
        } else {
#pragma unroll
            for (int jj = 0; jj < TW_NT; ++jj) {
                if (4 * jj >= a.B) break;
                GemvArgs a4 = a;
                a4.b0 = 4 * jj;
                a4.B = min(4, a.B - 4 * jj);
                gv_epilogue<EPI>(a4, rg[k], v2[k][jj][0], v2[k][jj][1], f[jj], lane);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// The slice's activation operand, by the CTA's TW_OPT threads past the
// producer warps (which meanwhile start the weight copies): one item per
// (block kb of the slice, column b), 32 elements each.  Columns past the batch
// get zeros (their MMA results are never read, but must be finite).
// ---------------------------------------------------------------------------
constexpr int TW_OPT = TW_THREADS - 32 * TW_WG;
ER_DEV void tw_opbar() { asm volatile("bar.sync 1, %0;" ::"n"(TW_OPT) : "memory"); }

__device__ inline void tw_operand(const GemvArgs &a, int s, int ku0, int nu, uint8_t *opnd, float *fac,
                                  unsigned *cmax, float *issq, float *wssq, int tid) {
    const int nbs = 2 * nu, nitems = nbs * 16;
    if (tid < 16) cmax[tid] = 0u;
    tw_opbar();
    float v[2][32];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {  // both items' loads first: they are independent
        const int it = tid + rr * TW_OPT, kb = it >> 4, b = it & 15;
        if (it < nitems && b < a.B) {
            const float4 *xp = reinterpret_cast<const float4 *>(a.x + (size_t)b * a.K + ku0 * 64 + kb * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 x4 = __ldcg(xp + i);
                v[rr][4 * i] = x4.x; v[rr][4 * i + 1] = x4.y; v[rr][4 * i + 2] = x4.z; v[rr][4 * i + 3] = x4.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[rr][i] = 0.f;
        }
    }
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int it = tid + rr * TW_OPT, kb = it >> 4, b = it & 15;
        float ssq = 0.f, m = 0.f;
        if (it < nitems && b < a.B) {
            const int k = ku0 * 64 + kb * 32;
#pragma unroll
            for (int i = 0; i < 32; ++i) ssq = fmaf(v[rr][i], v[rr][i], ssq);
            if (a.gain) {
                const float4 *gp = reinterpret_cast<const float4 *>(a.gain + k);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 g4 = __ldg(gp + i);
                    v[rr][4 * i] *= g4.x; v[rr][4 * i + 1] *= g4.y; v[rr][4 * i + 2] *= g4.z; v[rr][4 * i + 3] *= g4.w;
                }
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[rr][i]));
            if (!isfinite(m)) m = 0.f;
            atomicMax(cmax + b, __float_as_uint(m));  // non-negative floats order as their bits
        }
        if (it < 512) issq[it] = ssq;
    }
    tw_opbar();
    if (tid < 16) {
        float f = 0.f;
        if (tid < a.B) {
            float t = 0.f;
            for (int kb = 0; kb < nbs; ++kb) t += issq[kb * 16 + tid];  // block order: deterministic
            wssq[s * 16 + tid] = t;  // every CTA of the slice writes the same value
            const float mx = __uint_as_float(cmax[tid]);
            int e = 0;
            if (mx > 0.f) {
                int E;
                frexpf(mx, &E);
                e = 15 - E;
            }
            f = ldexpf(1.f, -e);
        }
        fac[tid] = f;
    }
    tw_opbar();
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int it = tid + rr * TW_OPT, kb = it >> 4, b = it & 15;
        if (it >= nitems) continue;
        const float sc = b < a.B ? 1.f / fac[b] : 0.f;
        uint8_t *row = opnd + (kb >> 1) * TW_ATOM_BYTES + (b >> 3) * 1024 + (b & 7) * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const float v0 = v[rr][8 * cc + 2 * p] * sc, v1 = v[rr][8 * cc + 2 * p + 1] * sc;
                const __half h0 = __float2half_rn(v0), h1 = __float2half_rn(v1);
                const __half l0 = __float2half_rn(v0 - __half2float(h0));
                const __half l1 = __float2half_rn(v1 - __half2float(h1));
                const __half2 hh = __halves2half2(h0, h1), ll = __halves2half2(l0, l1);
                hi[p] = *reinterpret_cast<const uint32_t *>(&hh);
                lo[p] = *reinterpret_cast<const uint32_t *>(&ll);
            }
            const int phys = (((kb & 1) * 4 + cc) ^ (b & 7)) * 16;
            *reinterpret_cast<uint4 *>(row + phys) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4 *>(row + 2048 + phys) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    }
    fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core's reads
}

// ---------------------------------------------------------------------------
template <int QT, int EPI>
__global__ void __launch_bounds__(TW_THREADS, 1) gemv_tc_kernel(const GemvArgs a, float *wpart, float *wssq) {
    static_assert(TW_WG == 2 && TW_EPI == 2, "warp roles are laid out for two warpgroups, two epilogue warps each");
    constexpr int UB = QTraits<QT>::unit_bytes, QB = QTraits<QT>::quant_bytes;
    constexpr int RGS = tw_rgs<QT>(), STAGE = tw_stage<QT>();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // swizzle atoms: 1024-aligned
    uint8_t *opnd = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + tw_off_bars<QT>());
    float *fac = reinterpret_cast<float *>(smem + tw_off_misc<QT>());
    unsigned *cmax = reinterpret_cast<unsigned *>(fac + 16);
    float *issq = reinterpret_cast<float *>(cmax + 16);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(issq + 512);
    volatile int *stop_s = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *abort_s = stop_s + 1;
    unsigned *tiles_done = reinterpret_cast<unsigned *>(tmem_slot + 4);  // [TW_WG], row-warp arrivals

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = tw_slices(a.UPR), nC = gridDim.x;
    int s = 0;
    while (s + 1 < S && tw_cta0(s + 1, S, nC) <= (int)blockIdx.x) ++s;
    const int c0 = tw_cta0(s, S, nC), ns = tw_cta0(s + 1, S, nC) - c0, jc = blockIdx.x - c0;
    const int rg0 = (int)((long long)jc * a.R / ns), rg1 = (int)((long long)(jc + 1) * a.R / ns);
    const int ku0 = s * TW_SLICE_UNITS, nu = min(TW_SLICE_UNITS, a.UPR - ku0);
    const int nst = (nu + TW_SU - 1) / TW_SU;  // ring stages per tile
    // warpgroup w: producer warp w, MMA warp 2 + w, row warps 4 + 4w .. 7 + 4w,
    // epilogue warps 12 + 2w (even tiles) and 13 + 2w (odd tiles)
    const int w = warp < 4 ? (warp & 1) : warp < 12 ? (warp - 4) >> 2 : (warp - 12) >> 1;
    const int wrg0 = rg0 + (int)((long long)w * (rg1 - rg0) / TW_WG);
    const int wrg1 = rg0 + (int)((long long)(w + 1) * (rg1 - rg0) / TW_WG);
    const int ntiles = (wrg1 - wrg0 + 7) / 8;
    uint64_t *full = bars + w * TW_BARS_PER_WG, *empty = full + TW_NS, *afull = empty + TW_NS,
             *dfull = afull + TW_NBUF;
    uint8_t *ring_w = smem + TW_OPND_BYTES + w * TW_NS * STAGE;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(TW_TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 0) {
        for (int i = 0; i < TW_WG; ++i) {
            uint64_t *b = bars + i * TW_BARS_PER_WG;
            for (int k = 0; k < TW_NS; ++k) {
                mbar_init(b + k, 1);              // full: the producer's expect_tx
                mbar_init(b + TW_NS + k, 4);      // empty: one arrival per row warp
            }
            for (int k = 0; k < TW_NBUF; ++k) {
                mbar_init(b + 2 * TW_NS + k, 4);            // afull: one arrival per row warp
                mbar_init(b + 2 * TW_NS + TW_NBUF + k, 1);  // dfull: the MMA warp's commit
            }
            tiles_done[i] = 0u;
        }
        *stop_s = 0;
        *abort_s = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&]() {
        atomicOr(a.flags, ER_FLAG_WAIT);
        *abort_s = 1;
    };

    // ---- producer warp w: stages of (tile, 2 units), in order; lane i copies row group i
    const bool producer = warp < TW_WG;
    int p_tile = 0, p_st = 0;
    unsigned p_cnt = 0;
    auto issue_stage = [&]() {  // whole warp
        const int rgb = wrg0 + 8 * p_tile, nv = min(8, wrg1 - rgb);
        const int u0 = p_st * TW_SU, cnt = min(TW_SU, nu - u0);
        const unsigned slot = p_cnt % TW_NS;
        if (lane == 0) mbar_arrive_expect_tx(full + slot, (uint32_t)(nv * cnt * UB));
        __syncwarp();
        if (lane < nv)
            bulk_g2s(ring_w + slot * STAGE + lane * RGS, a.W + ((size_t)(rgb + lane) * a.UPR + ku0 + u0) * UB,
                     (uint32_t)(cnt * UB), full + slot);
        ++p_cnt;
        if (++p_st == nst) {
            p_st = 0;
            ++p_tile;
        }
    };
    if (producer)  // the weights are constant: start streaming before the inputs are ready
        for (int i = 0; i < TW_NS && p_tile < ntiles; ++i) issue_stage();

    // ---- everything above touches only constant weights; now wait for inputs
    // (the producer warps never read them and go on streaming weights)
    if (!producer) {
        pdl_wait();
        const int ot = tid - 32 * TW_WG;
        // an earlier kernel's give-up flag: published after the operand build, so nothing waits for it before
        const int stop_r = ot == 0 ? (*reinterpret_cast<volatile int *>(a.flags) & ER_FLAG_WAIT) : 0;
        tw_operand(a, s, ku0, nu, opnd, fac, cmax, issq, wssq, ot);
        if (ot == 0) *stop_s = stop_r;
    }
    __syncthreads();
    const bool stop = *stop_s != 0;  // an earlier kernel gave up on a wait: drain and stop
    if (!stop) pdl_launch_dependents();

    if (!stop && warp < TW_WG) {
        // ---- producer: refill each stage once all four row warps have left it
        while (p_tile < ntiles) {
            const unsigned slot = p_cnt % TW_NS;
            int ok = 1;
            if (lane == 0) ok = mbar_wait(empty + slot, ((p_cnt / TW_NS) - 1u) & 1u) ? (*abort_s ? 2 : 1) : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (ok != 1) {
                if (ok == 0 && lane == 0) fail();
                break;
            }
            issue_stage();
        }
    } else if (!stop && warp < 2 * TW_WG) {
        // ---- MMA issuer: per block, D = A Bhi + A Blo over two K steps of 16
        if (lane == 0) {
            const unsigned T = (unsigned)(ntiles * nst);
            const uint32_t tA = tmem + (uint32_t)(w * 256), tD = tA + 64;
            // descriptors are linear in the address: + 64 B per block, + 32 B per K step
            const uint64_t d0 = tc_desc_sw128(smem_u32(opnd));
            unsigned m = 0;
            for (; m < T; ++m) {
                if (!mbar_wait(afull + (m & 1u), (m >> 1) & 1u)) {
                    fail();
                    break;
                }
                if (*abort_s) break;
                tc_fence_after();
                // the stage is unit m % nst of the tile: its two blocks, two K steps each;
                // N = 32 takes the hi rows (0-15) and the lo rows (16-31) of the operand at once
                const uint64_t ds = d0 + (uint64_t)((m % (unsigned)nst) * (TW_ATOM_BYTES >> 4));
                const uint32_t av = tA + (m & 1u) * 32, dv = tD + (m & 1u) * 64;
                tc_mma_ts(dv, av, ds, 0u);
                tc_mma_ts(dv, av + 8, ds + 2, 1u);
                tc_mma_ts(dv + 32, av + 16, ds + 4, 0u);
                tc_mma_ts(dv + 32, av + 24, ds + 6, 1u);
                tc_commit(dfull + (m & 1u));
            }
            if (m > 0 && !mbar_wait(dfull + ((m - 1) & 1u), ((m - 1) >> 1) & 1u)) fail();  // MMAs done
        }
    } else if (!stop && warp >= 12) {
        // ---- epilogue warps: once the four row warps have written a tile's
        // partials, count each row group's slice in; the last slice finishes it
        bool bad = false, fready = false;
        float f[TW_NT];
        unsigned long long kbest[TW_NT] = {0ull, 0ull, 0ull, 0ull};
        int nfin = 0;  // row groups finished by this warp
        for (int tile = (warp - 12) & 1; tile < ntiles; tile += TW_EPI) {
            const unsigned need = 4u * (unsigned)(tile + 1);
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_cta(tiles_done + w) < need) {
                if (*abort_s || globaltimer_ns() - t0 > wait_limit_ns()) {
                    bad = true;
                    break;
                }
                __nanosleep(64);
            }
            if (__any_sync(0xffffffffu, bad)) break;
            const int rgb = wrg0 + 8 * tile, nv = min(8, wrg1 - rgb);
            bool last = false;
            if (lane < nv) last = atom_add_acq_rel_gpu(a.cnt + rgb + lane, 1) == S - 1;  // releases the partials
            unsigned mask = __ballot_sync(0xffffffffu, last);
            nfin += __popc(mask);
            if (mask && !fready) {
                tw_colscale(a, S, wssq, lane, f);
                fready = true;
            }
            while (mask) {
                int rg2[2] = {-1, -1};
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (mask) {
                        const int i = __ffs(mask) - 1;
                        mask &= mask - 1;
                        rg2[k] = rgb + i;
                    }
                tw_finish2<EPI>(a, rg2, S, wpart, f, lane, kbest);
                const int rz = lane == 0 ? rg2[0] : rg2[1];
                if (lane < 2 && rz >= 0) a.cnt[rz] = 0;
                __syncwarp();
            }
        }
        if (EPI == EPI_LOGITS && nfin) tw_logits_flush(a, kbest, nfin, lane);
    } else if (!stop) {
        // ---- row threads: thread = one weight row = one TMEM lane.  Lane l of
        // row warp q takes row group l % 8 of the tile and row q + 4 (l / 8) of
        // it, so the 32 lanes' 16-byte reads of a stage hit 16 distinct
        // addresses spread over all 8 bank groups.
        const int q = warp & 3;
        const int rgi = lane & 7, r = q + 4 * (lane >> 3), g = r & 7, upper = r >> 3;
        const uint32_t tA = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(w * 256), tD = tA + 64;
        const uint32_t qoff = (uint32_t)(rgi * RGS + 64 * g);
        const uint32_t soff = (uint32_t)(rgi * RGS + QB + 8 * g + 2 * upper);
        const uint32_t sel = upper ? 0x4342u : 0x4140u;
        const uint32_t sh = upper ? 4u : 0u;
        const uint32_t rbase = smem_u32(ring_w);
        float fr[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) fr[c] = fac[c];
        unsigned sc = 0;
        bool bad = false;
        float acc[16];
        // adds d(row, block) * (D hi + D lo) for the two blocks of stage m (TMEM buffer m % 2)
        auto readback = [&](unsigned m, float dq0, float dq1) {
            if (!__all_sync(0xffffffffu, mbar_wait(dfull + (m & 1u), (m >> 1) & 1u))) {
                fail();
                bad = true;
                return;
            }
            tc_fence_after();
            uint32_t d0[32], d1[32];
            __syncwarp();
            tc_ld32(tD + (m & 1u) * 64, d0);
            tc_ld32(tD + (m & 1u) * 64 + 32, d1);
            tc_wait_ld(d0, d1);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                acc[c] = fmaf(dq0, __uint_as_float(d0[c]) + __uint_as_float(d0[16 + c]), acc[c]);
                acc[c] = fmaf(dq1, __uint_as_float(d1[c]) + __uint_as_float(d1[16 + c]), acc[c]);
            }
        };
        for (int tile = 0; tile < ntiles && !bad; ++tile) {
            const int rgb = wrg0 + 8 * tile, nv = min(8, wrg1 - rgb);
#pragma unroll
            for (int c = 0; c < 16; ++c) acc[c] = 0.f;
            float dqp0 = 0.f, dqp1 = 0.f;
            bool pend = false;  // the previous stage is still to read back
            for (int st = 0; st < nst; ++st, ++sc) {
                const unsigned slot = sc % TW_NS, buf = sc & 1u;
                const bool ok = __all_sync(0xffffffffu, mbar_wait(full + slot, (sc / TW_NS) & 1u));
                if (!ok || *abort_s) {
                    if (!ok) fail();
                    bad = true;
                    break;
                }
                const uint32_t sb = rbase + slot * STAGE;
                float dq0, dq1;
                {
                    uint32_t col[32];
                    tw_unit_cols<QT>(sb + qoff, sel, sh, col);
                    dq0 = __half2float(__ushort_as_half((unsigned short)lds16(sb + soff)));
                    dq1 = __half2float(__ushort_as_half((unsigned short)lds16(sb + soff + 4)));
                    __syncwarp();
                    tc_st32(tA + buf * 32, col);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + slot);  // the stage's bytes are read
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull + buf);
                if (pend) {
                    readback(sc - 1, dqp0, dqp1);
                    if (bad) break;
                }
                dqp0 = dq0;
                dqp1 = dq1;
                pend = true;
            }
            if (!bad && pend) readback(sc - 1, dqp0, dqp1);
            if (bad) break;
            // this slice's partial of the row: 16 columns, scaled back by the column factors,
            // each to its finisher lane 4g + c % 4, slot 2 (c / 4) + upper
            if (rgi < nv) {
                float *pp = wpart + ((size_t)s * a.R + rgb + rgi) * 256 + 32 * g + upper;
#pragma unroll
                for (int c = 0; c < 16; ++c) pp[8 * (c & 3) + 2 * (c >> 2)] = acc[c] * fr[c];
            }
            __syncwarp();
            if (lane == 0) red_add_release_cta(tiles_done + w, 1u);
        }
    }
    __syncwarp();
    // ---- drain: no copy may still be landing in shared memory at exit
    if (producer && lane == 0) {
        for (unsigned k = p_cnt > TW_NS ? p_cnt - TW_NS : 0u; k < p_cnt; ++k)
            if (!mbar_wait(full + k % TW_NS, (k / TW_NS) & 1u)) {
                atomicOr(a.flags, ER_FLAG_WAIT);
                break;
            }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TW_TMEM_COLS) : "memory");
    }
}

// ---------------------------------------------------------------------------
template <int QT, int EPI>
static cudaError_t tw_attr() {
    cudaError_t e = cudaFuncSetAttribute(gemv_tc_kernel<QT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         tw_smem<QT>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(gemv_tc_kernel<QT, EPI>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

cudaError_t gemv_tc_prepare() {
    cudaError_t r[10] = {tw_attr<Q8_0, EPI_STORE>(), tw_attr<Q8_0, EPI_RESID>(), tw_attr<Q8_0, EPI_QKV>(),
                         tw_attr<Q8_0, EPI_SWIGLU>(), tw_attr<Q8_0, EPI_LOGITS>(), tw_attr<Q4_0, EPI_STORE>(),
                         tw_attr<Q4_0, EPI_RESID>(), tw_attr<Q4_0, EPI_QKV>(), tw_attr<Q4_0, EPI_SWIGLU>(),
                         tw_attr<Q4_0, EPI_LOGITS>()};
    for (cudaError_t x : r)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

bool gemv_tc_fits(int qt, int K, int B, int num_sms) {
    (void)qt;
    // at least one CTA per slice; one operand item per (block, column) for each of at most 2 rounds of threads
    return B >= 1 && B <= 16 && K % 64 == 0 && K > 0 && tw_slices(K / 64) <= num_sms &&
           2 * TW_SLICE_UNITS * 16 <= 2 * TW_OPT;
}

template <int QT, int EPI>
static cudaError_t tw_launch(const GemvArgs &a, float *wpart, float *wssq, int num_sms, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)num_sms);
    cfg.blockDim = dim3(TW_THREADS);
    cfg.dynamicSmemBytes = tw_smem<QT>();
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemv_tc_kernel<QT, EPI>, a, wpart, wssq);
}

cudaError_t launch_gemv_tc(int epi, const GemvArgs &a, float *wpart, float *wssq, int num_sms, cudaStream_t st,
                             bool pdl) {
    if (!gemv_tc_fits(a.qt, a.K, a.B, num_sms) || a.b0 != 0) return cudaErrorInvalidValue;
    if (a.qt == Q8_0) {
        switch (epi) {
            case EPI_STORE: return tw_launch<Q8_0, EPI_STORE>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_RESID: return tw_launch<Q8_0, EPI_RESID>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_QKV: return tw_launch<Q8_0, EPI_QKV>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_SWIGLU: return tw_launch<Q8_0, EPI_SWIGLU>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_LOGITS: return tw_launch<Q8_0, EPI_LOGITS>(a, wpart, wssq, num_sms, st, pdl);
        }
    } else {
        switch (epi) {
            case EPI_STORE: return tw_launch<Q4_0, EPI_STORE>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_RESID: return tw_launch<Q4_0, EPI_RESID>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_QKV: return tw_launch<Q4_0, EPI_QKV>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_SWIGLU: return tw_launch<Q4_0, EPI_SWIGLU>(a, wpart, wssq, num_sms, st, pdl);
            case EPI_LOGITS: return tw_launch<Q4_0, EPI_LOGITS>(a, wpart, wssq, num_sms, st, pdl);
        }
    }
    return cudaErrorInvalidValue;
}

// this translation unit's copy of the bounded-wait limit
cudaError_t set_wait_limit_tc(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace er
