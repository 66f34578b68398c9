// The Q8_0 K/V cache: quantising rows into it and reading them back as GGUF
// blocks.
//
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
// er_kv_read_blocks returns the GGUF blocks in their own order.
// Quantiser (every step in float32, the same on every path that writes the
// cache): amax = largest |x| of the block; d = fp16(amax / 127) (float32
// division, round to nearest even); q = clamp(round(x / d), -127, 127) with
// round half away from zero and the division by the stored scale; q = 0 when
// d = 0.  A value reads back as d * q.
#include "common.cuh"
#include "internal.h"

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
        q_head[kvq_code_off(v, r, E * lane + e, 32 * E)] = (int8_t)(int)q;
    }
    if ((lane & (32 / E - 1)) == 0) d_row[lane / (32 / E)] = dh;
}

// base offsets of (sequence b, layer l, KV head h, row r) in the q and d planes
__device__ inline size_t kvq_head(int b, int L, int l, int KV, int h) { return ((size_t)b * L + l) * KV + h; }

// fp16 token-major rows [n][KV * hd] -> cache rows start..start+n-1 of (seq, layer); one warp per (row, head)
template <int E>
__global__ void kvq_write_kernel(const __half *k_rows, const __half *v_rows, int n, KvqCache c, int seq, int layer,
                                 int start) {
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int hd = 32 * E;
    if (item >= 2 * n * c.KV) return;
    const int kv = item / (n * c.KV), rem = item - kv * n * c.KV, row = rem / c.KV, h = rem - row * c.KV;
    const __half *src = (kv ? v_rows : k_rows) + (size_t)row * c.KV * hd + (size_t)h * hd + E * lane;
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = __half2float(src[e]);
    const size_t head = kvq_head(seq, c.L, layer, c.KV, h);
    const int r = start + row;
    kvq_row<E>(x, (kv ? c.vq : c.kq) + head * c.rows * hd, kv != 0, r,
               (kv ? c.vd : c.kd) + (head * c.rows + r) * (hd / 32), lane);
}

// The step's new rows: fp32 staging [B][KV * hd] (written by the Q/K/V epilogue) -> cache row
// positions[b] of sequence seqmap[b] (b without a map) of layer `layer`, for every column whose
// position is in range; one warp per (column, head, K or V).
template <int E>
__global__ void kvq_stage_kernel(const float *k_stage, const float *v_stage, const int32_t *positions,
                                 const int32_t *seqmap, int B, KvqCache c, int layer) {
    pdl_wait();
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    const int hd = 32 * E;
    if (item >= 2 * B * c.KV) return;
    const int kv = item / (B * c.KV), rem = item - kv * B * c.KV, b = rem / c.KV, h = rem - b * c.KV;
    const int pos = positions[b];
    if (pos < 0 || pos >= c.cap) return;  // flagged by the embedding; nothing is written
    const float *src = (kv ? v_stage : k_stage) + ((size_t)b * c.KV + h) * hd + E * lane;
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = __ldcg(src + e);
    const size_t head = kvq_head(seqmap ? seqmap[b] : b, c.L, layer, c.KV, h);
    kvq_row<E>(x, (kv ? c.vq : c.kq) + head * c.rows * hd, kv != 0, pos,
               (kv ? c.vd : c.kd) + (head * c.rows + pos) * (hd / 32), lane);
}

// cache rows start..start+n-1 of (seq, layer) -> token-major GGUF Q8_0 blocks [n][KV * hd / 32][34 bytes]
__global__ void kvq_read_kernel(uint8_t *k_out, uint8_t *v_out, int n, KvqCache c, int hd, int seq, int layer,
                                int start) {
    const int nb = c.KV * hd / 32;  // blocks per row
    const long long total = 2ll * n * nb * 34;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const int kv = (int)(i / ((long long)n * nb * 34));
        const long long rem = i - (long long)kv * n * nb * 34;
        const int row = (int)(rem / (nb * 34)), j = (int)(rem % (nb * 34));
        const int blk = j / 34, byte = j % 34, h = blk / (hd / 32), hb = blk % (hd / 32);
        const size_t head = kvq_head(seq, c.L, layer, c.KV, h);
        const int r = start + row;
        uint8_t out;
        if (byte < 2) {
            const __half d = (kv ? c.vd : c.kd)[(head * c.rows + r) * (hd / 32) + hb];
            out = (uint8_t)(__half_as_ushort(d) >> (8 * byte));
        } else {
            out = (uint8_t)(kv ? c.vq : c.kq)[head * c.rows * hd + kvq_code_off(kv != 0, r, hb * 32 + byte - 2, hd)];
        }
        (kv ? v_out : k_out)[(size_t)rem] = out;
    }
}

cudaError_t launch_kvq_write(const __half *k_rows, const __half *v_rows, int n, const KvqCache &c, int hd, int seq,
                             int layer, int start, cudaStream_t st) {
    const int warps = 2 * n * c.KV, per = 8;
    const unsigned blocks = (unsigned)((warps + per - 1) / per);
    if (hd == 128)
        kvq_write_kernel<4><<<blocks, per * 32, 0, st>>>(k_rows, v_rows, n, c, seq, layer, start);
    else if (hd == 64)
        kvq_write_kernel<2><<<blocks, per * 32, 0, st>>>(k_rows, v_rows, n, c, seq, layer, start);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

cudaError_t launch_kvq_stage(const float *k_stage, const float *v_stage, const int32_t *positions,
                             const int32_t *seqmap, int B, const KvqCache &c, int hd, int layer, cudaStream_t st,
                             bool pdl) {
    const int warps = 2 * B * c.KV, per = 8;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)((warps + per - 1) / per));
    cfg.blockDim = dim3(per * 32);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (hd == 128)
        return cudaLaunchKernelEx(&cfg, kvq_stage_kernel<4>, k_stage, v_stage, positions, seqmap, B, c, layer);
    if (hd == 64)
        return cudaLaunchKernelEx(&cfg, kvq_stage_kernel<2>, k_stage, v_stage, positions, seqmap, B, c, layer);
    return cudaErrorInvalidValue;
}

cudaError_t launch_kvq_read(uint8_t *k_out, uint8_t *v_out, int n, const KvqCache &c, int hd, int seq, int layer,
                            int start, cudaStream_t st) {
    const long long total = 2ll * n * (c.KV * hd / 32) * 34;
    long long blocks = (total + 255) / 256;
    if (blocks > 65535) blocks = 65535;
    if (blocks < 1) return cudaSuccess;
    kvq_read_kernel<<<(unsigned)blocks, 256, 0, st>>>(k_out, v_out, n, c, hd, seq, layer, start);
    return cudaGetLastError();
}

}  // namespace er
