// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/er.h"

namespace er {

// ---------------------------------------------------------------------------
// a repacked matrix (layout described in layout.cuh)
// ---------------------------------------------------------------------------
struct Mat {
    uint8_t *d = nullptr;
    int qt = 0;      // QType
    int rowmap = 0;  // RowMap
    int N = 0;       // virtual rows carried (GATEUP: rows of each of gate/up)
    int K = 0;       // columns
    int R = 0;       // row groups
    int UPR = 0;     // units per row group
    size_t bytes = 0;
};

struct RepackSrc {
    const uint8_t *p[3];
    int rows[3];
    int nsrc;
};

// queue the repack of `src` (GGUF blocks, concatenated by rows or gate/up
// interleaved per `rowmap`) into m.d (allocated by the caller, m.bytes long)
cudaError_t launch_repack(const Mat &m, const RepackSrc &src, cudaStream_t st);
// dequantise an IDENT-mapped matrix to fp32 [N][K]
cudaError_t launch_dequant(const Mat &m, float *out, cudaStream_t st);

// ---------------------------------------------------------------------------
// GEMV / fused epilogues
// ---------------------------------------------------------------------------
enum Epi : int { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SWIGLU = 3, EPI_LOGITS = 4 };

struct GemvArgs {
    const uint8_t *W;
    int R, UPR, N, K, qt;
    int B, b0;          // columns b0 .. b0+B-1 of the batch (B <= 4)
    const float *x;     // [batch][K]
    const float *gain;  // [K] RMSNorm gain, or nullptr (no norm)
    float eps;
    float *y;  // STORE/RESID/LOGITS: [B][N] (LOGITS: may be nullptr)
    // QKV epilogue
    float *q_out;
    __half *kc, *vc;
    const float2 *rope;
    const int32_t *positions;
    int qd, kvd, hd, KV, L, layer, cap;
    // SWIGLU epilogue
    float *a_out;
    // LOGITS epilogue
    unsigned long long *amax;
    int *done;
    int32_t *argmax_out;
    // scratch + flags
    float *part;
    int *cnt;
    int *flags;
};

// B <= 4 per launch; returns cudaErrorInvalidValue for shapes it cannot take
cudaError_t launch_gemv(int epi, const GemvArgs &a, int num_sms, cudaStream_t st, bool pdl);
cudaError_t gemv_prepare();  // sets kernel attributes once (call before any capture)
size_t gemv_part_floats(int num_sms);
bool gemv_fits(int qt, int K, int B);
int gemv_max_cols(int qt, int K);  // largest B <= 4 that gemv_fits

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------
struct AttnArgs {
    const float *q;  // [B][qd]
    const __half *kc, *vc;
    const int32_t *positions;
    float *o;  // [B][qd]
    float *part;
    int *cnt;
    int *flags;
    int B, H, KV, hd, L, layer, cap, S, CH;
};
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t st, bool pdl);
void attention_plan(int hd, int KV, int B, int cap, int num_sms, int *S, int *CH);
cudaError_t attention_prepare();  // kernel attributes (called by gemv_prepare)

// ---------------------------------------------------------------------------
// small kernels
// ---------------------------------------------------------------------------
struct EmbedArgs {
    const int32_t *tokens, *positions;
    const __half *embd_f16;  // untied fp16 table, or nullptr
    Mat head;                // tied: the repacked token_embd
    float *x;                // [B][D]
    int B, D, V, cap;
    int *flags;
};
cudaError_t launch_embed(const EmbedArgs &a, cudaStream_t st, bool pdl);
cudaError_t launch_positions_increment(int32_t *pos, int n, cudaStream_t st);

}  // namespace er

// ---------------------------------------------------------------------------
// opaque API objects
// ---------------------------------------------------------------------------
struct er_matrix {
    er::Mat m;
    int device;
    int num_sms;
    float *part;
    int *cnt;
    int *flags;
};

struct er_layer_dev {
    er::Mat qkv, wo, gateup, down;
    float *attn_norm, *ffn_norm;
};

struct er_model {
    er_config cfg;
    int device;
    int num_sms;
    std::vector<er_layer_dev> layers;
    er::Mat head;
    __half *embd_f16;
    float *out_norm;
    size_t device_bytes;
    std::vector<void *> allocs;
};

struct er_graph_entry {
    const void *tokens, *positions, *logits, *argmax;
    cudaGraphExec_t exec;
};

struct er_kv {
    er_model *m;
    int B, cap, S, CH;
    __half *kc, *vc;
    float2 *rope;
    float *x, *q, *o, *a;
    float *attn_part;
    int *attn_cnt;
    float *gemv_part;
    int *gemv_cnt;
    unsigned long long *amax;
    int *done;
    int *flags;
    cudaStream_t cap_stream;
    std::vector<er_graph_entry> graphs;
    std::vector<void *> allocs;
};
