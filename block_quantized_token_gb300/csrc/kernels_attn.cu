// GQA decode attention over the fp16 KV cache on the tensor cores
// ("EdgeRunner Core Architecture" section 5.2: scores q.k / sqrt(hd), causal, a
// query at position p attends rows 0..p, query head h reads KV head h / G;
// softmax over the rows; o = sum p v).
//
// Work split.  The rows of every (sequence b, KV head) pair, rows 0..pos_b
// each, form one list; warp w of the W warps of the grid takes the contiguous
// range [w NR / W, (w+1) NR / W) (at least TA_MIN_ROWS rows per warp), so
// every warp streams the same number of bytes whatever the positions.  A
// warp keeps one online-softmax state (max m, sum l, o = sum e^(s - m) v, in
// log2 units) per query head of the group for each (b, KV head) it touches.
// A pair whose rows one warp covers is finished by that warp; otherwise each
// covering warp leaves its state in global memory and the last one to arrive
// (a counter per pair) merges them in warp order:
//   M = max_w m_w,  o = sum_w e^(m_w - M) o_w / sum_w e^(m_w - M) l_w.
//
// Arithmetic per tile of 16 rows (mma.sync m16n8k16, fp32 accumulate):
//   S^T = Q K^T: A = the group's queries, rows 0..7 the hi fp16 half of head
//         g = row, rows 8..15 the lo half (q = hi + lo, exact to 2^-22 after
//         a power-of-two rescale); B = K rows from shared memory (ldmatrix).
//         Lane (g, t) ends up with head g's scores of rows 2t, 2t+1, 2t+8, 2t+9
//         as hi + lo sums of its accumulator.
//   O += P V: A = the probabilities in exactly that lane layout (hi rows 0..7,
//         lo rows 8..15, p = hi + lo); B = V rows (ldmatrix.trans).
// K and V tiles reach shared memory through cp.async, 16 bytes per lane; the
// 16-byte chunk c of row r is stored at chunk c ^ (r & 7) of the row, so the
// eight rows an ldmatrix reads together sit in eight different bank groups.
// Two tiles per warp are in flight while a third is consumed; a range's first
// two are requested before its queries are read and, in decode with the fp16
// cache, before the warp waits for the kernel that produced the queries and
// the new row (unless those tiles hold the new row).
//
// Q8_0 cache (template flag Q8; layout in kvq.cuh): whole 16-row tiles of the
// code and scale planes are staged (rows outside the warp's range masked), and
// each lane reads its B fragments as 32-bit words of codes, already in fragment
// order, turning them into exact fp16 pairs in registers.  Score sums are kept
// per 32-value block and multiplied by the row's K scale; for P V each block's
// probabilities are multiplied by the row's V scale (and 2^8) before the hi/lo
// split.  The warp whose range ends at a pair's last row first quantises the
// step's new row from the fp32 staging into the planes.
#include "common.cuh"
#include "internal.h"
#include "kvq.cuh"

namespace er {

constexpr int TA_WARPS = 8;     // warps per CTA, fp16 cache
constexpr int TA_WARPS_Q8 = 8;  // warps per CTA, Q8_0 cache
constexpr int ta_warps(bool q8) { return q8 ? TA_WARPS_Q8 : TA_WARPS; }
constexpr int TA_SLOTS = 3;
constexpr int TA_TILE = 16;
constexpr int TA_MIN_ROWS = 64;  // rows per warp at least
constexpr int TA_MAXB = 16;

template <int HD>
struct TaCfg {
    static constexpr int KC = HD / 16;                   // k16 chunks of a head (Q K^T)
    static constexpr int NTD = HD / 8;                   // n8 tiles of a head (P V)
    static constexpr int ROWB = HD * 2;                  // row bytes in shared memory (chunks swizzled)
    static constexpr int TILEB = TA_TILE * ROWB;         // one K or V tile
    static constexpr int SLOT = 2 * TILEB;               // K tile then V tile
    static constexpr int CPL = TA_TILE * HD / 8 / 32;    // 16-byte chunks per lane per tile
    static constexpr int SMEM = TA_WARPS * TA_SLOTS * SLOT;
};

// Q8_0 cache tiles: whole 16-row tiles of the planes (kernels_kvq.cu order), per slot the K codes, the K
// scales [16][HD / 32], the V codes and the V scales.  The codes are already in tensor-core fragment order:
// a lane's B fragments of a tile are 32-bit words of one contiguous run (K: hd / 4 bytes of each of its two
// rows; V: hd / 2 bytes), turned into exact fp16 pairs in registers.  16-byte chunks are XOR-swizzled so
// that the 8 lanes of every 128-bit read phase hit distinct bank groups.
template <int HD>
struct TaQ8Cfg {
    static constexpr int QT = TA_TILE * HD;             // code bytes of one tile
    static constexpr int SROW = HD / 32 * 2;            // scale bytes of one row: 8 or 4
    static constexpr int ST = TA_TILE * SROW;           // scale bytes of one tile
    static constexpr int SLOT = 2 * (QT + ST);          // K codes, K scales, V codes, V scales
    static constexpr int SLOTS = 4;                     // tiles staged per warp
    static constexpr int NQ = HD / 32;                  // 16-byte chunks of a lane's V run
    static constexpr int WARP = SLOTS * SLOT;
    static constexpr int SMEM = TA_WARPS_Q8 * WARP;
    static constexpr float VPRE = 256.f;  // power of two the V-scaled probabilities are multiplied by
};

ER_DEV void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
ER_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
ER_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

ER_DEV void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
ER_DEV void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
ER_DEV uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}
// (a, b) = hi + lo with hi = fp16(a, b) and lo = fp16 of the remainders, as two packed pairs
ER_DEV void split_h2(float a, float b, uint32_t &hi, uint32_t &lo) {
    hi = pack_h2(a, b);
    const float2 h = __half22float2(*reinterpret_cast<const __half2 *>(&hi));
    lo = pack_h2(a - h.x, b - h.y);
}

struct TaGeom {
    int NR, W;  // rows in the list, working warps
    int T[TA_MAXB];
    int base[TA_MAXB + 1];
};

__device__ inline void ta_locate(const TaGeom &g, int B, int u, int &b, int &kvh, int &seg_start, int &seg_end) {
    b = 0;
    while (b + 1 < B && u >= g.base[b + 1]) ++b;
    kvh = (u - g.base[b]) / g.T[b];
    seg_start = g.base[b] + kvh * g.T[b];
    seg_end = seg_start + g.T[b];
}

// State of one warp for its piece of one (b, KV head): lane (g, t) holds head
// g's running max (equal over t), a partial sum over its rows, and the hi/lo
// accumulator tiles of O (dims 8j + 2t, 8j + 2t + 1).
template <int HD>
struct TaState {
    float m, l;
    float o[TaCfg<HD>::NTD][4];
};

// One (sequence, KV head) of the cache: fp16 rows K, V ([cap][HD]), or Q8_0 planes Kq, Vq ([cap][HD] int8)
// with scales Kd, Vd ([cap][HD / 32] fp16).
struct TaSrc {
    const __half *K, *V;
    const int8_t *Kq, *Vq;
    const __half *Kd, *Vd;
};

// Rows [r0, r1) of the cache head `src` for the G query heads at qh (fp32 [G][HD], unscaled).  Q8: the
// cache holds Q8_0 blocks.
template <int HD, int G, bool Q8>
__device__ void ta_attend(const float *qh, const TaSrc &src, int r0, int r1, uint8_t *ring, int lane,
                          TaState<HD> &st, bool dep = false, bool last = false) {
    using C = TaCfg<HD>;
    using Q = TaQ8Cfg<HD>;
    const int g = lane >> 2, t = lane & 3;
    // fp16: tiles from r0; Q8: the whole 16-row tiles of the planes that cover [r0, r1)
    const int tb0 = Q8 ? r0 & ~(TA_TILE - 1) : r0;
    const int ntiles = (r1 - tb0 + TA_TILE - 1) / TA_TILE;
    const uint32_t ring_s = smem_u32(ring);
    constexpr int NS = Q8 ? Q::SLOTS : TA_SLOTS;  // ring slots
    auto issue = [&](int k) {
        if (k < ntiles) {
            const int rb = tb0 + k * TA_TILE;
            if constexpr (!Q8) {
                const uint32_t slot = ring_s + (uint32_t)((k % TA_SLOTS) * C::SLOT);
#pragma unroll
                for (int i = 0; i < C::CPL; ++i) {
                    const int ci = lane + 32 * i;            // chunk of the tile
                    const int row = ci / (HD / 8), col = ci % (HD / 8);
                    const bool ok = rb + row < r1;
                    const size_t off = (size_t)(ok ? rb + row : r0) * HD + col * 8;
                    const uint32_t d = (uint32_t)(row * C::ROWB + (col ^ (row & 7)) * 16);
                    cp_async16(slot + d, src.K + off, ok ? 16u : 0u);
                    cp_async16(slot + C::TILEB + d, src.V + off, ok ? 16u : 0u);
                }
            } else {
                // a whole tile of the planes (rows rb .. rb + 15 lie below the planes' rounded-up rows)
                const uint32_t slot = ring_s + (uint32_t)((k % NS) * Q::SLOT);
#pragma unroll
                for (int i = 0; i < HD / 32; ++i) {
                    const int ci = lane + 32 * i;  // 16-byte chunk of the tile (HD chunks per side)
                    const int row = ci / (HD / 16), j = ci % (HD / 16);
                    cp_async16(slot + row * HD + ((j ^ (row & 1)) << 4), src.Kq + (size_t)(rb + row) * HD + j * 16,
                               16u);
                    const int L = ci / Q::NQ, q = ci % Q::NQ, key = (L * Q::NQ / 8) % Q::NQ;
                    cp_async16(slot + Q::QT + Q::ST + L * (HD / 2) + ((q ^ key) << 4),
                               src.Vq + (size_t)rb * HD + ci * 16, 16u);
                }
                if (lane < Q::SROW) {  // scales: 16 rows x SROW bytes per side, SROW chunks
                    cp_async16(slot + Q::QT + lane * 16, src.Kd + (size_t)rb * (HD / 32) + lane * 8, 16u);
                } else if (lane >= 16 && lane < 16 + Q::SROW) {
                    cp_async16(slot + 2 * Q::QT + Q::ST + (lane - 16) * 16,
                               src.Vd + (size_t)rb * (HD / 32) + (lane - 16) * 8, 16u);
                }
            }
        }
        cp_async_commit();  // an empty group keeps the count uniform
    };
    // dep: the producing kernel (queries, the new row) is still to be waited for.  The first tiles are requested
    // before the wait unless they hold the new row, the pair's last (last: this piece ends the pair).
    const bool pre = !(last && r1 - 1 < tb0 + (NS - 1) * TA_TILE);
    if (dep && !pre) pdl_wait();
    for (int k = 0; k < NS - 1; ++k) issue(k);
    if (dep && pre) pdl_wait();
    // queries: scale to log2 units, rescale by a power of two so that the lo
    // halves stay normal, split hi + lo into A fragments
    const float qscale = 1.4426950408889634f / sqrtf((float)HD);
    float qv[C::KC][4];
    float qmax = 0.f;
#pragma unroll
    for (int c = 0; c < C::KC; ++c) {
        float2 x0 = make_float2(0.f, 0.f), x1 = x0;
        if (g < G) {
            x0 = __ldcg(reinterpret_cast<const float2 *>(qh + g * HD + 16 * c + 2 * t));
            x1 = __ldcg(reinterpret_cast<const float2 *>(qh + g * HD + 16 * c + 2 * t + 8));
        }
        qv[c][0] = x0.x * qscale; qv[c][1] = x0.y * qscale; qv[c][2] = x1.x * qscale; qv[c][3] = x1.y * qscale;
#pragma unroll
        for (int i = 0; i < 4; ++i) qmax = fmaxf(qmax, fabsf(qv[c][i]));
    }
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
    int e = 0;
    if (qmax > 0.f && isfinite(qmax)) {
        int E;
        frexpf(qmax, &E);
        e = 15 - E;
    }
    const float up = ldexpf(1.f, e), down = ldexpf(1.f, -e);
    uint32_t qa[C::KC][4];
#pragma unroll
    for (int c = 0; c < C::KC; ++c) {
        float hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float v = qv[c][i] * up;
            hi[i] = __half2float(__float2half_rn(v));
            lo[i] = v - hi[i];
        }
        qa[c][0] = pack_h2(hi[0], hi[1]);  // row g (hi), k = 2t, 2t+1
        qa[c][1] = pack_h2(lo[0], lo[1]);  // row g + 8 (lo)
        qa[c][2] = pack_h2(hi[2], hi[3]);  // row g, k = 2t + 8, 2t + 9
        qa[c][3] = pack_h2(lo[2], lo[3]);
    }

    st.m = -INFINITY;
    st.l = 0.f;
#pragma unroll
    for (int j = 0; j < C::NTD; ++j) st.o[j][0] = st.o[j][1] = st.o[j][2] = st.o[j][3] = 0.f;

    // ldmatrix row addresses of this lane (see the header): K as the B operand
    // (rows (lane & 7) + 8 (lane >> 4), column half (lane >> 3) & 1), V
    // transposed (rows (lane & 7) + 8 ((lane >> 3) & 1), column half lane >> 4)
    // (the row index mod 8 is lane & 7 in both; chunks are XOR-swizzled by it)
    const int sw = lane & 7;
    const uint32_t k_row = (uint32_t)(((lane & 7) + ((lane >> 4) << 3)) * C::ROWB), k_half = (lane >> 3) & 1;
    const uint32_t v_row = (uint32_t)(C::TILEB + ((lane & 7) + (((lane >> 3) & 1) << 3)) * C::ROWB), v_half = lane >> 4;
    for (int k = 0; k < ntiles; ++k) {
        issue(k + NS - 1);
        cp_async_wait<NS - 1>();
        __syncwarp();
        uint32_t slot;
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        // Q8: the K/V scales of this lane's four rows 2t, 2t + 1, 2t + 8, 2t + 9 (fp16 pairs)
        uint32_t dks[4][HD / 64], dvs[4][HD / 64];
        if constexpr (!Q8) {
            slot = ring_s + (uint32_t)((k % TA_SLOTS) * C::SLOT);
            // scores of 16 rows: two n8 tiles (rows 0..7 and 8..15 of the tile)
#pragma unroll
            for (int c = 0; c < C::KC; ++c) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(slot + k_row + (((2 * c + k_half) ^ sw) << 4), b0, b1, b2, b3);
                mma_16816(s0, qa[c], b0, b1, s0);
                mma_16816(s1, qa[c], b2, b3, s1);
            }
        } else {
            const uint32_t qslot = ring_s + (uint32_t)((k % NS) * Q::SLOT);
            // this lane's K words: rows g and g + 8, dims 16c + {2t, 2t+1, 2t+8, 2t+9} of chunk c
            uint32_t kw[2][HD / 16];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = 8 * h + g;
#pragma unroll
                for (int k2 = 0; k2 < HD / 64; ++k2) {
                    const int ch = (HD / 64) * t + k2;
                    const uint4 w = lds128(qslot + row * HD + ((ch ^ (row & 1)) << 4));
                    kw[h][4 * k2] = w.x; kw[h][4 * k2 + 1] = w.y; kw[h][4 * k2 + 2] = w.z; kw[h][4 * k2 + 3] = w.w;
                }
            }
            // the K / V scales of this lane's four rows 2t, 2t + 1, 2t + 8, 2t + 9 (fp16 pairs): rows 2t and
            // 2t + 1 (and 2t + 8, 2t + 9) are adjacent, one 16- or 8-byte read per pair of rows and side
#pragma unroll
            for (int pr = 0; pr < 2; ++pr) {
                const uint32_t ko = qslot + Q::QT + (2 * t + 8 * pr) * Q::SROW;
                const uint32_t vo = qslot + 2 * Q::QT + Q::ST + (2 * t + 8 * pr) * Q::SROW;
                if constexpr (HD == 128) {
                    const uint4 kx = lds128(ko), vx = lds128(vo);
                    dks[2 * pr][0] = kx.x; dks[2 * pr][1] = kx.y; dks[2 * pr + 1][0] = kx.z; dks[2 * pr + 1][1] = kx.w;
                    dvs[2 * pr][0] = vx.x; dvs[2 * pr][1] = vx.y; dvs[2 * pr + 1][0] = vx.z; dvs[2 * pr + 1][1] = vx.w;
                } else {
                    static_assert(HD == 64, "head dim 64 or 128");
                    const uint2 kx = lds64(ko), vx = lds64(vo);
                    dks[2 * pr][0] = kx.x; dks[2 * pr + 1][0] = kx.y;
                    dvs[2 * pr][0] = vx.x; dvs[2 * pr + 1][0] = vx.y;
                }
            }
            slot = qslot;
            // scores block by block (2 k16 chunks per 32-value block), each block's sums times its row's scale
#pragma unroll
            for (int bb = 0; bb < HD / 32; ++bb) {
                float b0s[4] = {0.f, 0.f, 0.f, 0.f}, b1s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int c = 2 * bb; c < 2 * bb + 2; ++c) {
                    uint32_t b0, b1, b2, b3;
                    q8_word_to_h2(kw[0][c], b0, b1);
                    q8_word_to_h2(kw[1][c], b2, b3);
                    mma_16816(b0s, qa[c], b0, b1, b0s);
                    mma_16816(b1s, qa[c], b2, b3, b1s);
                }
                float dk[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) dk[i] = (bb & 1) ? h2f_hi(dks[i][bb >> 1]) : h2f_lo(dks[i][bb >> 1]);
                s0[0] = fmaf(dk[0], b0s[0], s0[0]); s0[2] = fmaf(dk[0], b0s[2], s0[2]);
                s0[1] = fmaf(dk[1], b0s[1], s0[1]); s0[3] = fmaf(dk[1], b0s[3], s0[3]);
                s1[0] = fmaf(dk[2], b1s[0], s1[0]); s1[2] = fmaf(dk[2], b1s[2], s1[2]);
                s1[1] = fmaf(dk[3], b1s[1], s1[1]); s1[3] = fmaf(dk[3], b1s[3], s1[3]);
            }
        }
        const int rb = tb0 + k * TA_TILE;
        float sc[4] = {(s0[0] + s0[2]) * down, (s0[1] + s0[3]) * down, (s1[0] + s1[2]) * down,
                       (s1[1] + s1[3]) * down};
        const int rr[4] = {rb + 2 * t, rb + 2 * t + 1, rb + 2 * t + 8, rb + 2 * t + 9};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (rr[i] >= r1 || rr[i] < r0) sc[i] = -INFINITY;
        float mt = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
        const float mn = fmaxf(st.m, mt);
        float p[4] = {0.f, 0.f, 0.f, 0.f};
        if (mn != -INFINITY) {
            if (mn != st.m) {
                const float corr = exp2f(st.m - mn);
                st.l *= corr;
#pragma unroll
                for (int j = 0; j < C::NTD; ++j) {
                    st.o[j][0] *= corr; st.o[j][1] *= corr; st.o[j][2] *= corr; st.o[j][3] *= corr;
                }
                st.m = mn;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = exp2f(sc[i] - mn);
            st.l += (p[0] + p[1]) + (p[2] + p[3]);
        }
        if constexpr (!Q8) {
            float ph[4], pl[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                ph[i] = __half2float(__float2half_rn(p[i]));
                pl[i] = p[i] - ph[i];
            }
            const uint32_t pa[4] = {pack_h2(ph[0], ph[1]), pack_h2(pl[0], pl[1]), pack_h2(ph[2], ph[3]),
                                    pack_h2(pl[2], pl[3])};
#pragma unroll
            for (int j2 = 0; j2 < C::NTD / 2; ++j2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(slot + v_row + (((2 * j2 + v_half) ^ sw) << 4), b0, b1, b2, b3);
                mma_16816(st.o[2 * j2], pa, b0, b1, st.o[2 * j2]);
                mma_16816(st.o[2 * j2 + 1], pa, b2, b3, st.o[2 * j2 + 1]);
            }
        } else {
            // this lane's V words: rows {2t, 2t+1, 2t+8, 2t+9} of dim 8j + g for every n8 tile j
            uint32_t vw[HD / 8];
            {
                const int key = (lane * Q::NQ / 8) % Q::NQ;
#pragma unroll
                for (int q = 0; q < Q::NQ; ++q) {
                    const uint4 w = lds128(slot + Q::QT + Q::ST + lane * (HD / 2) + ((q ^ key) << 4));
                    vw[4 * q] = w.x; vw[4 * q + 1] = w.y; vw[4 * q + 2] = w.z; vw[4 * q + 3] = w.w;
                }
            }
            // per 32-value block of V: P times the block's row scales (and 2^8, so that the fp16 halves
            // stay normal), split hi + lo, against the block's four n8 tiles
            float p8[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p8[i] = p[i] * Q::VPRE;
#pragma unroll
            for (int bb = 0; bb < HD / 32; ++bb) {
                float pv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    pv[i] = p8[i] * ((bb & 1) ? h2f_hi(dvs[i][bb >> 1]) : h2f_lo(dvs[i][bb >> 1]));
                uint32_t pa[4];
                split_h2(pv[0], pv[1], pa[0], pa[1]);
                split_h2(pv[2], pv[3], pa[2], pa[3]);
#pragma unroll
                for (int j = 4 * bb; j < 4 * bb + 4; ++j) {
                    uint32_t b0, b1;
                    q8_word_to_h2(vw[j], b0, b1);
                    mma_16816(st.o[j], pa, b0, b1, st.o[j]);
                }
            }
        }
        __syncwarp();  // every lane is done with this slot before it is refilled
    }
    cp_async_wait<0>();
    if constexpr (Q8) {  // undo the probabilities' power-of-two factor
#pragma unroll
        for (int j = 0; j < C::NTD; ++j) {
            st.o[j][0] *= 1.f / Q::VPRE; st.o[j][1] *= 1.f / Q::VPRE;
            st.o[j][2] *= 1.f / Q::VPRE; st.o[j][3] *= 1.f / Q::VPRE;
        }
    }
    // the row sum over the four lanes of the head
    st.l += __shfl_xor_sync(0xffffffffu, st.l, 1);
    st.l += __shfl_xor_sync(0xffffffffu, st.l, 2);
}

template <int HD, int G, bool Q8>
__global__ void __launch_bounds__(ta_warps(Q8) * 32, 1) attn_tc_kernel(const AttnArgs a) {
    using C = TaCfg<HD>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    uint8_t *ring = smem + warp * (Q8 ? TaQ8Cfg<HD>::WARP : TA_SLOTS * C::SLOT);
    const int qd = a.H * HD;

    // fp16 cache in decode: each warp waits for the producing kernel inside its first piece, after requesting
    // tiles that kernel does not write
    const bool defer = !Q8 && a.seqmap == nullptr;
    if (!defer) pdl_wait();
    pdl_launch_dependents();

    // geometry of the row list (positions are inputs of the step)
    TaGeom geo;
    geo.NR = 0;
    for (int b = 0; b < a.B; ++b) {
        const int pos = a.positions[b];
        geo.T[b] = (pos >= 0 && pos < a.cap) ? pos + 1 : 0;
        geo.base[b] = geo.NR;
        geo.NR += a.KV * geo.T[b];
    }
    geo.base[a.B] = geo.NR;
    const int Wmax = gridDim.x * ta_warps(Q8);
    geo.W = (geo.NR + TA_MIN_ROWS - 1) / TA_MIN_ROWS;
    if (geo.W > Wmax) geo.W = Wmax;
    const int w = blockIdx.x * ta_warps(Q8) + warp;
    if (w >= geo.W) return;
    const int wa = (int)((long long)w * geo.NR / geo.W), wb = (int)((long long)(w + 1) * geo.NR / geo.W);

    int u = wa;
    bool dep = defer;
    while (u < wb) {
        int b, kvh, seg_start, seg_end;
        ta_locate(geo, a.B, u, b, kvh, seg_start, seg_end);
        const int r0 = u - seg_start, r1 = (wb < seg_end ? wb : seg_end) - seg_start;
        const bool first_piece = u == wa;
        u = wb < seg_end ? wb : seg_end;
        const size_t head = ((size_t)(a.seqmap ? a.seqmap[b] : b) * a.L + a.layer) * a.KV + kvh;
        TaSrc src;
        if constexpr (Q8) {
            const size_t rows = (size_t)((a.cap + TA_TILE - 1) & ~(TA_TILE - 1));  // whole tiles per head
            src.K = src.V = nullptr;
            src.Kq = a.kq + head * rows * HD;
            src.Vq = a.vq + head * rows * HD;
            src.Kd = a.kd + head * rows * (HD / 32);
            src.Vd = a.vd + head * rows * (HD / 32);
        } else {
            src.K = a.kc + head * a.cap * HD;
            src.V = a.vc + head * a.cap * HD;
            src.Kq = src.Vq = nullptr;
            src.Kd = src.Vd = nullptr;
        }
        if constexpr (Q8) {
            // the step's new row (the pair's last) from the fp32 staging into the planes, by the one warp
            // whose range holds it, before any of its tiles is requested.  Other warps may stage the same
            // 16-row tile meanwhile; the row lies outside their ranges and is masked there.
            if (a.k_stage && r1 == seg_end - seg_start) {
                constexpr int E = HD / 32;
                const int pos = r1 - 1;
#pragma unroll
                for (int kvs = 0; kvs < 2; ++kvs) {
                    const float *xs = (kvs ? a.v_stage : a.k_stage) + ((size_t)b * a.KV + kvh) * HD + E * lane;
                    float x[E];
#pragma unroll
                    for (int e = 0; e < E; ++e) x[e] = __ldcg(xs + e);
                    // the planes are read-only to the tiles' loads, written here once per step
                    kvq_row<E>(x, const_cast<int8_t *>(kvs ? src.Vq : src.Kq), kvs != 0, pos,
                               const_cast<__half *>(kvs ? src.Vd : src.Kd) + (size_t)pos * (HD / 32), lane);
                }
                __threadfence();
                __syncwarp();
            }
        }
        TaState<HD> st;
        ta_attend<HD, G, Q8>(a.q + (size_t)b * qd + (size_t)kvh * G * HD, src, r0, r1, ring, lane, st, dep,
                             r1 == seg_end - seg_start);
        dep = false;
        float *o_grp = a.o + (size_t)b * qd + (size_t)kvh * G * HD;
        if (seg_start >= wa && seg_end <= wb) {  // the whole pair: finish here
            if (g < G) {
                const float inv = st.l > 0.f ? 1.f / st.l : 0.f;
#pragma unroll
                for (int j = 0; j < C::NTD; ++j)
                    *reinterpret_cast<float2 *>(o_grp + g * HD + 8 * j + 2 * t) =
                        make_float2((st.o[j][0] + st.o[j][2]) * inv, (st.o[j][1] + st.o[j][3]) * inv);
            }
            continue;
        }
        // shared with other warps: leave the state [G][m, l, -, -, o[HD]]
        float *ps = a.part + ((size_t)w * 2 + (first_piece ? 0 : 1)) * G * (HD + 4);
        if (g < G) {
            if (t == 0) *reinterpret_cast<float2 *>(ps + g * (HD + 4)) = make_float2(st.m, st.l);
#pragma unroll
            for (int j = 0; j < C::NTD; ++j)
                *reinterpret_cast<float2 *>(ps + g * (HD + 4) + 4 + 8 * j + 2 * t) =
                    make_float2(st.o[j][0] + st.o[j][2], st.o[j][1] + st.o[j][3]);
        }
        __syncwarp();
        const int grp = b * a.KV + kvh;
        int last = 0;
        if (lane == 0) last = atom_add_acq_rel_gpu(a.cnt + grp, 1);  // releases this warp's state
        last = __shfl_sync(0xffffffffu, last, 0);
        const int w_first = (int)(((long long)(seg_start + 1) * geo.W - 1) / geo.NR);
        const int w_last = (int)(((long long)seg_end * geo.W - 1) / geo.NR);
        if (last != w_last - w_first) continue;
        __syncwarp();
        // the last warp of the pair: merge the covering warps' states in warp
        // order; each lane owns float4 chunks of the group's output (one head
        // per chunk) and keeps every contributor's loads in flight together
        const int s0 = ((long long)w_first * geo.NR / geo.W >= seg_start) ? 0 : 1;
        auto state = [&](int ww) {
            return a.part + ((size_t)ww * 2 + (ww == w_first ? s0 : 0)) * G * (HD + 4);
        };
        for (int ch = lane; ch < G * HD / 4; ch += 32) {
            const int gi = (4 * ch) / HD, d = 4 * ch - gi * HD;
            float M = -INFINITY, L = 0.f;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w0 = w_first; w0 <= w_last; w0 += 12) {  // twelve states in flight, online rescale
                float mm[12], ll[12];
                float4 ov[12];
#pragma unroll
                for (int j = 0; j < 12; ++j) {
                    const int ww = w0 + j;
                    mm[j] = -INFINITY;
                    ll[j] = 0.f;
                    ov[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (ww <= w_last) {
                        const float *q = state(ww) + gi * (HD + 4);
                        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(q));
                        mm[j] = ml.x;
                        ll[j] = ml.y;
                        ov[j] = __ldcg(reinterpret_cast<const float4 *>(q + 4 + d));
                    }
                }
                float mc = M;
#pragma unroll
                for (int j = 0; j < 12; ++j) mc = fmaxf(mc, mm[j]);
                if (mc == -INFINITY) continue;
                const float corr = exp2f(M - mc);
                L *= corr;
                O.x *= corr; O.y *= corr; O.z *= corr; O.w *= corr;
                M = mc;
#pragma unroll
                for (int j = 0; j < 12; ++j) {
                    const float ew = exp2f(mm[j] - mc);
                    L = fmaf(ll[j], ew, L);
                    O.x = fmaf(ov[j].x, ew, O.x); O.y = fmaf(ov[j].y, ew, O.y);
                    O.z = fmaf(ov[j].z, ew, O.z); O.w = fmaf(ov[j].w, ew, O.w);
                }
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
            *reinterpret_cast<float4 *>(o_grp + gi * HD + d) = make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv);
        }
        if (lane == 0) a.cnt[grp] = 0;
    }
}

void attention_plan(int hd, int KV, int B, int cap, int num_sms, int *S, int *CH) {
    (void)hd; (void)KV; (void)B; (void)cap;
    *S = num_sms;        // CTAs of the launch (the kernel uses fewer for short lists)
    *CH = TA_MIN_ROWS;   // rows per warp at least
}

size_t attention_part_floats(int hd, int G, int num_sms) {
    return (size_t)num_sms * (TA_WARPS > TA_WARPS_Q8 ? TA_WARPS : TA_WARPS_Q8) * 2 * G * (hd + 4);
}

template <int HD, int G>
static cudaError_t at_launch(const AttnArgs &a, cudaStream_t st, bool pdl) {
    const bool q8 = a.kq != nullptr;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)a.S);
    cfg.blockDim = dim3(ta_warps(q8) * 32);
    cfg.dynamicSmemBytes = q8 ? TaQ8Cfg<HD>::SMEM : TaCfg<HD>::SMEM;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (q8) return cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, G, true>, a);
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, G, false>, a);
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

template <int HD, int G, bool Q8>
static cudaError_t at_attr1() {
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<HD, G, Q8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Q8 ? TaQ8Cfg<HD>::SMEM : TaCfg<HD>::SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(attn_tc_kernel<HD, G, Q8>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    return e;
}

template <int HD, int G>
static cudaError_t at_attr() {
    const cudaError_t e = at_attr1<HD, G, false>();
    return e != cudaSuccess ? e : at_attr1<HD, G, true>();
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
    if (a.B > TA_MAXB || a.S < 1) return cudaErrorInvalidValue;
    if (a.hd == 64) return at_launch_g<64>(a, st, pdl);
    if (a.hd == 128) return at_launch_g<128>(a, st, pdl);
    return cudaErrorInvalidValue;
}

// this translation unit's copy of the bounded-wait limit
cudaError_t set_wait_limit_attn(unsigned long long ns) { return set_wait_limit_here(ns); }

}  // namespace er
