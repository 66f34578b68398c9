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
    float *k_stage, *v_stage;  // non-null: K/V rows go to fp32 staging [batch][kvd] instead of kc / vc
    const int32_t *seqmap;     // cache sequence of each column (nullptr: column b is sequence b)
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
    // optional shared-memory copies (persistent step): positions and RoPE rows
    // [b][hd / 2] of the step, and the residual rows [row group - resid_rg0][16][GV_MAXB]
    const int *pos_s;
    const float2 *rope_s;
    const float *resid_s;
    int resid_rg0, resid_nrg;
};

// B <= 4 per launch; returns cudaErrorInvalidValue for shapes it cannot take
cudaError_t launch_gemv(int epi, const GemvArgs &a, int num_sms, cudaStream_t st, bool pdl);
// The whole batch (up to 16 columns, b0 = 0) in one pass over the weights:
// K-slices of 1024 columns, partials wpart (gemv_wide_part_floats), per-slice
// sums of squares wssq (gemv_wide_ssq_floats), counters a.cnt [R] (zero).
// variant: WIDE_AUTO (by matrix size, gemv_wide_uses_tc), WIDE_MMA_SYNC or
// WIDE_TCGEN05 (kernels_wide_tc.cu).
enum WideVariant : int { WIDE_AUTO = 0, WIDE_MMA_SYNC = 1, WIDE_TCGEN05 = 2 };
cudaError_t launch_gemv_wide(int epi, const GemvArgs &a, float *wpart, float *wssq, int num_sms, cudaStream_t st,
                             bool pdl, int variant);
bool gemv_wide_uses_tc(int variant, int R, int UPR);
cudaError_t launch_gemv_tc(int epi, const GemvArgs &a, float *wpart, float *wssq, int num_sms, cudaStream_t st,
                           bool pdl);
cudaError_t gemv_tc_prepare();
bool gemv_tc_fits(int qt, int K, int B, int num_sms);
cudaError_t gemv_wide_prepare();
bool gemv_wide_fits(int qt, int K, int B, int num_sms);
size_t gemv_wide_part_floats(int R, int K);
size_t gemv_wide_ssq_floats(int K);
cudaError_t gemv_prepare();  // sets kernel attributes once (call before any capture)
size_t gemv_part_floats(int num_sms);
bool gemv_fits(int qt, int K, int B);
int gemv_max_cols(int qt, int K);  // largest B <= 4 that gemv_fits

// ---------------------------------------------------------------------------
// attention
// ---------------------------------------------------------------------------
struct AttnArgs {
    const float *q;  // [B][qd]
    const __half *kc, *vc;        // fp16 cache [B][L][KV][cap][hd], or
    const int8_t *kq, *vq;        // Q8_0 cache (kq != nullptr): codes [B][L][KV][rows * hd] (kvq.cuh order)
    const __half *kd, *vd;        //   and block scales [B][L][KV][rows][hd / 32], rows = cap rounded up to 16
    const int32_t *seqmap;        // cache sequence of each column (nullptr: column b is sequence b)
    const float *k_stage, *v_stage;  // Q8_0: the new rows in fp32 [B][KV * hd], quantised by the kernel (or
                                     // nullptr: already in the planes)
    const int32_t *positions;
    float *o;  // [B][qd]
    float *part;  // warp states of pairs shared by warps (attention_part_floats)
    int *cnt;     // [B * KV] arrival counters (zero between launches)
    int *flags;
    // S: CTAs of the launch; CH: rows per warp at least (both from attention_plan)
    int B, H, KV, hd, L, layer, cap, S, CH;
};
cudaError_t launch_attention(const AttnArgs &a, cudaStream_t st, bool pdl);

// ---------------------------------------------------------------------------
// Q8_0 K/V cache (kernels_kvq.cu): values [B][L][KV][cap][hd] int8 and block
// scales [B][L][KV][cap][hd / 32] fp16, one plane pair for K and one for V
// ---------------------------------------------------------------------------
struct KvqCache {
    int8_t *kq, *vq;
    __half *kd, *vd;
    int L, KV, cap;
    int rows;  // rows of each head's planes: cap rounded up to 16 (whole V tiles)
};
// fp16 token-major rows [n][KV * hd] (device) -> cache rows start.. of (seq, layer)
cudaError_t launch_kvq_write(const __half *k_rows, const __half *v_rows, int n, const KvqCache &c, int hd, int seq,
                             int layer, int start, cudaStream_t st);
// a prefill chunk's fp32 staging rows [B][KV * hd] -> cache row positions[b] of sequence seqmap[b], `layer`
cudaError_t launch_kvq_stage(const float *k_stage, const float *v_stage, const int32_t *positions,
                             const int32_t *seqmap, int B, const KvqCache &c, int hd, int layer, cudaStream_t st,
                             bool pdl);
// cache rows start.. of (seq, layer) -> GGUF Q8_0 blocks [n][KV * hd / 32][34] (device)
cudaError_t launch_kvq_read(uint8_t *k_out, uint8_t *v_out, int n, const KvqCache &c, int hd, int seq, int layer,
                            int start, cudaStream_t st);
// launch shape of the attention kernel for a cache of this shape
void attention_plan(int hd, int KV, int B, int cap, int num_sms, int *S, int *CH);
size_t attention_part_floats(int hd, int G, int num_sms);  // AttnArgs::part
cudaError_t attention_prepare();  // kernel attributes (called by gemv_prepare)

// ---------------------------------------------------------------------------
// persistent decode step (kernels_step.cuh)
// ---------------------------------------------------------------------------
#define ER_MK_MAXB 4
#define ER_MK_MAXG 4
struct StepLayer {
    const uint8_t *w[4];  // repacked QKV (PAIR), Wo, gate/up (GATEUP), down
    const float *attn_norm, *ffn_norm;
};
struct StepArgs {
    const StepLayer *layers;  // device array [L]
    const uint8_t *head;      // repacked head (tied: token_embd)
    const float *out_norm;
    const __half *embd_f16;   // untied embedding, or nullptr
    int L, D, H, KV, hd, F, V, qd, kvd, B, cap;
    int R[5], UPR[5];         // row groups / units per row group: QKV, WO, GATEUP, DOWN, HEAD
    float eps;
    const int32_t *tokens, *positions;
    float *x, *q, *o, *a;
    __half *kc, *vc;
    const float2 *rope;
    float *logits;
    int32_t *argmax;
    float *part;    // GEMV cross-CTA partials
    int *cnt;       // GEMV cross-CTA counters
    float *apart;   // attention states of heads split over CTAs [CTA][2][G][hd + 4]
    int *acnt;      // attention counters [B * KV] (unused by the persistent step)
    unsigned long long *amax;
    int *done, *flags;
    unsigned *bar;  // grid barrier counter (zeroed before each launch)
    unsigned bar_extra;  // arrivals the first barrier waits for beyond the grid (0; > 0 only to test give-up)
};
// Whether the persistent step can run this shape (batch, GQA group, head dim,
// shared memory) and the launch itself (cooperative, one CTA per SM).
bool step_supported(int qt, int hd, int G, int B, int KV, int cap, int max_k, const int R[5], const int UPR[5],
                    int num_sms);
cudaError_t launch_step(int qt, const StepArgs &a, int num_sms, cudaStream_t st);
size_t step_apart_floats(int num_sms, int hd);
cudaError_t step_prepare();

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
// prefill chunk columns: pos[i] = start + i, seq[i] = s for i < n
cudaError_t launch_prefill_setup(int32_t *pos, int32_t *seq, int start, int s, int n, cudaStream_t st);

// one device allocation outside any owner list, counted and failure-injectable like the library's own
cudaError_t device_alloc(void **p, size_t bytes);
void device_free(void *p);

// every translation unit's copy of the bounded-wait limit (common.cuh), on the current device
cudaError_t set_wait_limit_gemv(unsigned long long ns);
cudaError_t set_wait_limit_wide(unsigned long long ns);
cudaError_t set_wait_limit_tc(unsigned long long ns);
cudaError_t set_wait_limit_step_q8(unsigned long long ns);
cudaError_t set_wait_limit_step_q4(unsigned long long ns);
cudaError_t set_wait_limit_attn(unsigned long long ns);

}  // namespace er

// error reporting shared by the entry points (sets er_last_error)
er_status er_fail_status(er_status s, const char *msg);
er_status er_fail_cuda(cudaError_t e, const char *what);

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

// recorded step graphs an er_kv keeps (one per pointer set; least recently used dropped first)
#define ER_MAX_GRAPHS 8

struct er_graph_entry {
    const void *tokens, *positions, *logits, *argmax;
    cudaGraphExec_t exec;
    unsigned long long last_use;  // er_decode_step call count at its last launch
};

struct er_kv {
    er_model *m;
    int B, cap, S, CH;
    int schedule;        // ER_SCHEDULE_PERSISTENT or ER_SCHEDULE_KERNELS (resolved)
    bool step_ok;        // the persistent step supports this shape
    er::StepLayer *step_layers;
    float *step_apart;
    int *step_acnt;
    unsigned *step_bar;
    int kv_type;                 // ER_KV_F16 or ER_KV_Q8_0
    __half *kc, *vc;             // fp16 cache (ER_KV_F16)
    er::KvqCache kvq;            // Q8_0 cache (ER_KV_Q8_0)
    float *kstage, *vstage;      // Q8_0: the step's new K/V rows in fp32 [B][kvd]
    const int32_t *seqmap;       // cache sequence of each column (nullptr: column b is sequence b)
    // chunked prefill: a 16-column view sharing this state's cache (created by the first er_prefill)
    er_kv *pf;
    bool view;                   // this state is such a view: cache and flags belong to its owner
    int32_t *pf_pos, *pf_seq;    // view: positions and sequences of the chunk's columns [16]
    float *pf_logits;            // view: logits of the chunk's columns [16][vocab]
    float2 *rope;
    float *x, *q, *o, *a;
    float *attn_part;
    int *attn_cnt;
    float *gemv_part;
    int *gemv_cnt;
    float *wide_part, *wide_ssq;  // batched GEMV scratch (nullptr: column groups instead)
    int wide_variant;             // er::WideVariant of the batched GEMV
    unsigned long long *amax;
    int *done;
    int *flags;
    cudaStream_t cap_stream;
    std::vector<er_graph_entry> graphs;  // at most ER_MAX_GRAPHS, least recently used dropped first
    unsigned long long graph_calls;
    unsigned bar_extra;                  // injected barrier shortfall (tests of the give-up path)
    std::vector<void *> allocs;
};
