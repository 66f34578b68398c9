// Create-time repack of GGUF blocks, the dequantisation test kernel, the
// embedding gather and the position increment.
#include "gemv_core.cuh"

namespace er {

// Source row of fragment row r in row group rg, or nullptr for a padding row.
__device__ inline const uint8_t *repack_src_row(const RepackSrc &s, int rowmap, int rg, int r, size_t row_bytes) {
    if (rowmap == MAP_GATEUP) {
        int n = 8 * rg + (r & 7);
        int which = r >> 3;
        return n < s.rows[which] ? s.p[which] + (size_t)n * row_bytes : nullptr;
    }
    int v = rowmap == MAP_PAIR ? 16 * rg + 2 * (r & 7) + (r >> 3) : 16 * rg + r;
    for (int i = 0; i < s.nsrc; ++i) {
        if (v < s.rows[i]) return s.p[i] + (size_t)v * row_bytes;
        v -= s.rows[i];
    }
    return nullptr;
}

// One thread per output byte.  Q8_0 stores q ^ 0x80, Q4_0 the GGUF nibble;
// padding rows and blocks become q = 0 with scale 0.
__global__ void repack_kernel(uint8_t *__restrict__ dst, RepackSrc src, int qt, int rowmap, int K, int UPR,
                              size_t total) {
    const int nb = K / 32;
    const int gbb = gguf_block_bytes_of(qt);
    const size_t row_bytes = (size_t)nb * gbb;
    const int ub = unit_bytes_of(qt);
    const int qb = quant_bytes_of(qt);
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        size_t unit = i / ub;
        int j = (int)(i - unit * ub);
        int rg = (int)(unit / UPR);
        int u = (int)(unit - (size_t)rg * UPR);
        uint8_t out;
        if (j >= qb) {  // scale byte
            int s = j - qb;
            int g = s >> 3, w = (s & 7) >> 1, half = s & 1;
            int blk = w >> 1, upper = w & 1;
            int r = g + 8 * upper;
            int kb = 2 * u + blk;
            const uint8_t *row = repack_src_row(src, rowmap, rg, r, row_bytes);
            out = (row && kb < nb) ? row[(size_t)kb * gbb + half] : 0;
        } else if (qt == Q8_0) {
            int blk = j >> 9, lane = (j & 511) >> 4, jj = j & 15;
            int h = jj >> 3, reg = (jj & 7) >> 1, e = jj & 1;
            int g = lane >> 2, t = lane & 3;
            int r = g + 8 * (reg & 1);
            int c = 16 * h + 8 * (reg >> 1) + 2 * t + e;  // column within the block
            int kb = 2 * u + blk;
            const uint8_t *row = repack_src_row(src, rowmap, rg, r, row_bytes);
            uint8_t q = (row && kb < nb) ? row[(size_t)kb * gbb + 2 + c] : 0;
            out = q ^ 0x80;
        } else {  // Q4_0: two nibbles per byte
            int lane = j >> 4, word = (j & 15) >> 2, bw = j & 3;
            int blk = word >> 1, h = word & 1;
            int g = lane >> 2, t = lane & 3;
            int kb = 2 * u + blk;
            out = 0;
            for (int half = 0; half < 2; ++half) {
                int p = 2 * bw + half;      // nibble index in the word
                int reg = p & 3, e = p >> 2;
                int r = g + 8 * (reg & 1);
                int c = 16 * h + 8 * (reg >> 1) + 2 * t + e;
                const uint8_t *row = repack_src_row(src, rowmap, rg, r, row_bytes);
                uint8_t nib = 8;
                if (row && kb < nb) {
                    uint8_t byte = row[(size_t)kb * gbb + 2 + (c & 15)];
                    nib = c < 16 ? (byte & 15) : (byte >> 4);
                }
                out |= nib << (4 * half);
            }
        }
        dst[i] = out;
    }
}

cudaError_t launch_repack(const Mat &m, const RepackSrc &src, cudaStream_t st) {
    size_t total = m.bytes;
    int threads = 256;
    size_t blocks = (total + threads - 1) / threads;
    if (blocks > 65535u * 16) blocks = 65535u * 16;
    repack_kernel<<<(unsigned)blocks, threads, 0, st>>>(m.d, src, m.qt, m.rowmap, m.K, m.UPR, total);
    return cudaGetLastError();
}

__global__ void dequant_kernel(const uint8_t *__restrict__ W, int qt, int UPR, int N, int K, float *__restrict__ out) {
    size_t total = (size_t)N * K;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        int row = (int)(i / K), col = (int)(i - (size_t)row * K);
        out[i] = repacked_value(W, qt, UPR, row, col);
    }
}

cudaError_t launch_dequant(const Mat &m, float *out, cudaStream_t st) {
    size_t total = (size_t)m.N * m.K;
    size_t blocks = (total + 255) / 256;
    if (blocks > 65535u * 16) blocks = 65535u * 16;
    if (blocks == 0) return cudaSuccess;
    dequant_kernel<<<(unsigned)blocks, 256, 0, st>>>(m.d, m.qt, m.UPR, m.N, m.K, out);
    return cudaGetLastError();
}

// x[b] = embedding row of tokens[b] (fp16 table, or the tied block matrix).
// Checks token and position ranges; a bad value sets a flag and the row is 0.
__global__ void embed_kernel(EmbedArgs a) {
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int tok = a.tokens[b];
    const int pos = a.positions[b];
    const bool tok_ok = tok >= 0 && tok < a.V;
    if (threadIdx.x == 0) {
        if (!tok_ok) atomicOr(a.flags, ER_FLAG_TOKEN);
        if (pos < 0 || pos >= a.cap) atomicOr(a.flags, ER_FLAG_POS);
    }
    float *x = a.x + (size_t)b * a.D;
    for (int k = threadIdx.x; k < a.D; k += blockDim.x) {
        float v = 0.f;
        if (tok_ok) {
            if (a.embd_f16)
                v = __half2float(a.embd_f16[(size_t)tok * a.D + k]);
            else
                v = repacked_value(a.head.d, a.head.qt, a.head.UPR, tok, k);
        }
        x[k] = v;
    }
}

cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t st, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3(a.B);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, embed_kernel, a);
}

__global__ void positions_increment_kernel(int32_t *pos, int n) {
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) pos[i] += 1;
}

cudaError_t launch_positions_increment(int32_t *pos, int n, cudaStream_t st) {
    positions_increment_kernel<<<(n + 127) / 128, 128, 0, st>>>(pos, n);
    return cudaGetLastError();
}

__global__ void prefill_setup_kernel(int32_t *pos, int32_t *seq, int start, int s, int n) {
    const int i = threadIdx.x;
    if (i < n) {
        pos[i] = start + i;
        seq[i] = s;
    }
}

cudaError_t launch_prefill_setup(int32_t *pos, int32_t *seq, int start, int s, int n, cudaStream_t st) {
    prefill_setup_kernel<<<1, 32, 0, st>>>(pos, seq, start, s, n);
    return cudaGetLastError();
}

}  // namespace er
