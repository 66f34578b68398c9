// The Q8_0 K/V cache: quantising rows into it and reading them back as GGUF
// blocks.  Layout and quantiser: kvq.cuh.
#include "internal.h"
#include "kvq.cuh"

namespace er {

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

// A prefill chunk's new rows: fp32 staging [B][KV * hd] (written by the Q/K/V epilogue) -> cache row
// positions[b] of sequence seqmap[b] (b without a map) of layer `layer`, for every column whose
// position is in range; one warp per (column, head, K or V).  (In a decode step the attention kernel
// quantises the new rows itself.)
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
            out = (uint8_t)(kv ? c.vq : c.kq)[head * c.rows * hd + kvq_code_off(kv != 0, r, hb * 32 + byte - 2, hd)] ^
                  0x80u;
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
