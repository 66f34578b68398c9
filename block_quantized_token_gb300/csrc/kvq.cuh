// The Q8_0 K/V cache's layout and its row quantiser, shared by the quantiser
// kernels (kernels_kvq.cu) and the attention kernel, which quantises a step's
// new rows itself.
// The pages name a packed Q8_0 K/V cache as an option ("llama.cpp Metal (MPS)
// End-to-End Inference Path", P9 quantized-KV flash-attention variants and
// section 5; "EdgeRunner Core Architecture" section 4.1 cache precisions) but
// give no quantiser for it.  Each head's row of hd values is stored as hd/32
// Q8_0 blocks, in two planes per (sequence, layer, KV head), with `rows` =
// capacity rounded up to 16:
//   q  int8 [rows * hd]        the codes, in the order the attention kernel's
//                              tensor-core fragments take them (below)
//   d  fp16 [rows][hd / 32]    one scale per 32-value block
// K codes: row-major, each row's hd bytes permuted so that lane t of an MMA
// quad finds its four values of every 16-value chunk c (dims 16c + 2t, + 1,
// + 8, + 9) as one 32-bit word, and its words of all chunks as one run of
// hd / 4 bytes.  V codes: in tiles of 16 rows, each tile ordered
// [dim % 8][quad lane][dim / 8][4 bytes of rows 2t, 2t + 1, 2t + 8, 2t + 9], so that
// a lane's P.V fragments of the whole tile are one run of hd / 2 bytes.
// Each code byte holds q XOR 0x80 (an untouched byte, 0x80, reads as 0).
// er_kv_read_blocks returns the GGUF blocks in their own order.
// Quantiser (every step in float32, the same on every path that writes the
// cache): amax = largest |x| of the block; d = fp16(amax / 127) (float32
// division, round to nearest even); q = clamp(round(x / d), -127, 127) with
// round half away from zero and the division by the stored scale; q = 0 when
// d = 0.  A value reads back as d * q.
#pragma once
#include "common.cuh"

namespace er {

// byte offset of dim d within a K row, and of (row r of its tile, dim d) within a V tile
__host__ __device__ inline int kvq_kpos(int d, int hd) {
    const int c = d >> 4, w = d & 15;
    return ((w & 7) >> 1) * (hd / 4) + c * 4 + ((w & 1) | ((w >> 3) << 1));
}
__host__ __device__ inline int kvq_vpos(int r, int d, int hd) {
    const int t = (r & 7) >> 1, s = (r & 1) | ((r >> 3) << 1);
    return (((d & 7) * 4 + t) * (hd / 8) + (d >> 3)) * 4 + s;
}
// byte offset of (row r, dim d) in one head's code plane of either side
__host__ __device__ inline size_t kvq_code_off(bool v, int r, int d, int hd) {
    return v ? (size_t)(r >> 4) * 16 * hd + kvq_vpos(r & 15, d, hd) : (size_t)r * hd + kvq_kpos(d, hd);
}

// One head row held by a warp, E = hd / 32 consecutive values per lane (lane l:
// values E l .. E l + E - 1); a 32-value block spans 32 / E lanes.  Writes the
// row's codes (E bytes per lane, at their places in the head's plane `q_head`)
// and its scales.
template <int E>
__device__ inline void kvq_row(const float (&x)[E], int8_t *q_head, bool v, int r, __half *d_row, int lane) {
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
    // the block's lanes: 32 / E consecutive lanes
#pragma unroll
    for (int off = 1; off < 32 / E; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const __half dh = __float2half_rn(amax / 127.f);
    const float d = __half2float(dh);
#pragma unroll
    for (int e = 0; e < E; ++e) {
        float q = d > 0.f ? roundf(x[e] / d) : 0.f;
        q = fminf(fmaxf(q, -127.f), 127.f);
        // stored as q XOR 0x80 (as the repacked weights): one byte permute and one subtraction per pair
        // turn a word of codes into exact fp16
        q_head[kvq_code_off(v, r, E * lane + e, 32 * E)] = (int8_t)((uint8_t)(int8_t)(int)q ^ 0x80u);
    }
    if ((lane & (32 / E - 1)) == 0) d_row[lane / (32 / E)] = dh;
}

}  // namespace er
