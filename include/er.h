/*
 * er.h -- C ABI of liber.so: one decode step of a Llama-style decoder whose 2-D
 * weights are GGUF Q8_0 or Q4_0 blocks, on one NVIDIA GB300 (sm_103a).
 *
 * The step follows "EdgeRunner Core Architecture", Overview and section 5.1:
 *
 *   tokens -> embedding -> [RMSNorm -> Q/K/V -> RoPE + K/V append -> GQA
 *   attention -> Wo + residual -> RMSNorm -> SwiGLU FFN + residual] x N ->
 *   RMSNorm -> LM head -> logits -> greedy argmax
 *
 * Conventions for every call:
 *   - Pointers named *_dev are device memory of the current CUDA device; all
 *     other pointers are host memory.  `stream` is a cudaStream_t passed as
 *     void* (NULL = the legacy default stream).
 *   - Calls return er_status.  Arguments are checked on the host before any
 *     work is queued; a failed check returns ER_EINVAL / ER_EUNSUPPORTED and
 *     queues nothing.  A failed CUDA call returns ER_ECUDA.  er_last_error()
 *     gives a one-line description of the last failure on the calling thread.
 *   - Work is queued asynchronously on `stream`; no call below synchronises
 *     the device unless its comment says so.
 *   - No call throws; no call aborts the process.
 */
#ifndef ER_H
#define ER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ER_API __attribute__((visibility("default")))
#else
#define ER_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ER_OK = 0,
    ER_EINVAL = 1,        /* bad argument (NULL, size out of range, mismatch)   */
    ER_ENOMEM = 2,        /* device allocation failed                           */
    ER_ECUDA = 3,         /* a CUDA runtime call failed                         */
    ER_EUNSUPPORTED = 4,  /* valid but not implemented (e.g. head_dim 96)       */
    ER_EDEVICE = 5        /* a kernel flagged bad data (see er_get_device_error) */
} er_status;

/* Tensor storage types.  The numeric values are GGUF's type codes as listed in
 * "EdgeRunner Core Architecture" section 1.3 (TensorDataType): float32 = 0,
 * float16 = 1, q4_0 = 2 (18-byte blocks), q8_0 = 8 (34-byte blocks). */
typedef enum { ER_F32 = 0, ER_F16 = 1, ER_Q4_0 = 2, ER_Q8_0 = 8 } er_dtype;

/* Model shape ("EdgeRunner Core Architecture" section 1.1, LlamaConfig).
 *   dim        embedding width D
 *   n_layers   decoder layers L
 *   n_heads    query heads H;  n_kv_heads  KV heads (H % n_kv_heads == 0)
 *   head_dim   hd; supported: 64 and 128
 *   ffn_dim    SwiGLU hidden width F
 *   vocab      V
 *   rope_base  RoPE frequency base (angle of pair i at position p: p * base^(-2i/hd))
 *   rms_eps    RMSNorm epsilon (inside the square root)
 *   w_type     ER_Q8_0 or ER_Q4_0: the format of every 2-D weight
 *   tied       0: token_embd is fp16 [V x D] and `output` is a w_type [V x D]
 *                 head;  1: token_embd is a w_type [V x D] matrix used both
 *                 as the embedding table and as the head (output must be NULL)
 *   max_batch  largest batch an er_kv of this model may hold (1..16)
 * D, H*hd, n_kv_heads*hd and F must be multiples of 32 (whole blocks). */
typedef struct {
    int32_t dim, n_layers, n_heads, n_kv_heads, head_dim, ffn_dim, vocab;
    double rope_base;
    double rms_eps;
    int32_t w_type;
    int32_t tied;
    int32_t max_batch;
} er_config;

/* Device pointers to one layer's tensors in GGUF layout.  Norm gains are fp32
 * [D].  Matrices are [rows = outputs] x [cols = inputs], row-major, each row
 * cols/32 consecutive blocks ("EdgeRunner Core Architecture" section 3.2):
 *   wq [H*hd x D], wk/wv [KV*hd x D], wo [D x H*hd],
 *   w_gate/w_up [F x D], w_down [D x F]. */
typedef struct {
    const void *attn_norm, *wq, *wk, *wv, *wo, *ffn_norm, *w_gate, *w_up, *w_down;
} er_layer_weights;

/* tok_embd: see er_config.tied; output_norm: fp32 [D]; output: w_type [V x D]
 * head or NULL when tied; layers: HOST array of n_layers entries. */
typedef struct {
    const void *tok_embd, *output_norm, *output;
    const er_layer_weights *layers;
} er_weights;

typedef struct er_model er_model;
typedef struct er_kv er_kv;
typedef struct er_matrix er_matrix;

/* Builds a model on the current device.  Every weight is repacked from GGUF
 * blocks into the library's own 16-byte-aligned tiled layout (the same bytes,
 * rearranged) in model-owned memory; norm gains and the fp16 embedding are
 * copied.  Synchronises `stream` before returning, so the caller may free its
 * copies afterwards.  *out is set only on ER_OK. */
ER_API er_status er_model_create(const er_config *cfg, const er_weights *w, void *stream, er_model **out);
ER_API void er_model_destroy(er_model *m);
/* Bytes of device memory the model owns (repacked weights, gains, embedding). */
ER_API size_t er_model_device_bytes(const er_model *m);

/* Creates the decode state of `batch` independent sequences with room for
 * `capacity` positions each: the fp16 K/V cache (zeroed), a RoPE cos/sin table
 * for positions 0..capacity-1 (computed in double on the host, stored fp32),
 * activations and kernel scratch.  Synchronises the device.  An er_kv must
 * not outlive its model. */
ER_API er_status er_kv_create(er_model *m, int32_t batch, int32_t capacity, er_kv **out);
ER_API void er_kv_destroy(er_kv *kv);

/* er_kv_create with a choice of cache storage, kv_type:
 *   ER_F16   the fp16 cache of er_kv_create
 *   ER_Q8_0  a packed Q8_0 cache: each head's row of head_dim values is kept as
 *            head_dim / 32 blocks of one fp16 scale d and 32 int8 codes q, and
 *            attention reads d * q.  The pages list a packed Q8_0 K/V cache as
 *            an option ("llama.cpp Metal (MPS) End-to-End Inference Path",
 *            table P9, the quantised-KV flash-attention variant, and the KV
 *            format note of its section 5) without giving its quantiser; the one
 *            used here, for every row written (er_kv_write and the step's new
 *            rows), in float32: amax = max |x| over the block,
 *            d = fp16(amax / 127) (round to nearest even),
 *            q = round(x / d) half away from zero, clamped to [-127, 127],
 *            q = 0 where d = 0.  A step's new K/V rows are quantised from the
 *            fp32 projection (after RoPE for K); er_kv_write quantises fp16 rows.
 *            Runs the per-phase schedule only (ER_SCHEDULE_PERSISTENT is
 *            ER_EUNSUPPORTED); head_dim 64 or 128.  Cache bytes per row and KV
 *            head: 2 * 34 * head_dim / 32 (K and V), against 4 * head_dim.
 * Any other kv_type is ER_EINVAL. */
ER_API er_status er_kv_create_typed(er_model *m, int32_t batch, int32_t capacity, int32_t kv_type, er_kv **out);
/* The cache storage of kv (ER_F16 or ER_Q8_0), or -1 for NULL. */
ER_API int32_t er_kv_type(const er_kv *kv);

/* Chunked prefill ("EdgeRunner Core Architecture" section 9.1, the fused
 * prefill pass; "alpaca.swift" Results, prefill): runs the decoder over the n
 * tokens tokens_dev[0..n-1] (device int32) of sequence `seq` at positions
 * start..start+n-1, writing their K/V rows of every layer into the cache, in
 * chunks of 16 tokens.  A chunk is one pass of the step's kernels over 16
 * columns that all belong to sequence `seq`: each GEMV reads its weights once
 * for the chunk, and the token at position p attends rows 0..p (the chunk's
 * earlier rows included), so the result equals n decode steps.  Rows below
 * `start` must already hold that sequence's keys and values; other sequences
 * are untouched.  logits_dev (fp32 [vocab], may be NULL) receives the logits of
 * the last token.  Queued on `stream`, no synchronisation.  The first call
 * allocates a 16-column scratch (activations and partials, about as much as a
 * 16-sequence decode state without its cache) and synchronises the device; it is
 * freed with kv.  Bad tokens and positions set the flags er_get_device_error
 * reports.  It writes the rows it is given and reads the sequence's rows
 * below them: do not run it concurrently (on another stream) with a decode
 * step or another prefill of the same kv.  ER_EINVAL: kv NULL, seq out of
 * range, start < 0, n < 0, start + n > capacity, or tokens_dev NULL with
 * n > 0. */
ER_API er_status er_prefill(er_kv *kv, int32_t seq, const int32_t *tokens_dev, int32_t n, int32_t start,
                            float *logits_dev, void *stream);

/* Reads cache rows start..start+n-1 of sequence `seq`, layer `layer` of an
 * ER_Q8_0 cache as GGUF Q8_0 blocks: k_blocks_dev / v_blocks_dev receive
 * [n][n_kv_heads * head_dim / 32] blocks of 34 bytes (little-endian fp16 d,
 * then 32 int8 q), token-major with heads contiguous, n * n_kv_heads *
 * head_dim / 32 * 34 bytes each (device memory the caller owns).  Queued on
 * `stream`.  ER_EUNSUPPORTED on an fp16 cache; ER_EINVAL for rows out of
 * range. */
ER_API er_status er_kv_read_blocks(er_kv *kv, int32_t seq, int32_t layer, int32_t start, int32_t n,
                                   void *k_blocks_dev, void *v_blocks_dev, void *stream);

/* Device addresses of the K and V cache of sequence `seq`, layer `layer`.
 * Layout of each: fp16 [n_kv_heads][capacity][head_dim] (head-major, then
 * position, then dimension).  K rows hold keys after RoPE; V rows are not
 * rotated.  Callers prefill rows below a sequence's first position here.
 * ER_EUNSUPPORTED on an ER_Q8_0 cache. */
ER_API er_status er_kv_layer_ptrs(er_kv *kv, int32_t seq, int32_t layer, void **k_dev, void **v_dev);

/* Copy n token-major rows k_rows_dev / v_rows_dev (fp16 [n][n_kv_heads*head_dim],
 * heads contiguous within a row, the layout GGUF runtimes use) into cache rows
 * start..start+n-1 of sequence `seq`, layer `layer` (er_kv_write), or the
 * reverse (er_kv_read).  Queued on `stream`; no synchronisation.  On an
 * ER_Q8_0 cache er_kv_write quantises the rows (er_kv_create_typed) and
 * er_kv_read is ER_EUNSUPPORTED (er_kv_read_blocks reads the blocks). */
ER_API er_status er_kv_write(er_kv *kv, int32_t seq, int32_t layer, int32_t start, int32_t n, const void *k_rows_dev,
                             const void *v_rows_dev, void *stream);
ER_API er_status er_kv_read(er_kv *kv, int32_t seq, int32_t layer, int32_t start, int32_t n, void *k_rows_dev,
                            void *v_rows_dev, void *stream);

/* One decode step for every sequence b of kv:
 *   tokens_dev[b]     int32 token id of sequence b (0 <= id < vocab)
 *   positions_dev[b]  int32 position p of that token (0 <= p < capacity)
 * Writes K/V of each sequence at row p, attends rows 0..p (rows below p must
 * hold earlier keys/values), and writes
 *   logits_dev  fp32 [batch][vocab] (may be NULL)
 *   argmax_dev  int32 [batch]: greedy token = index of the largest logit,
 *               lowest index on ties, NaN never chosen (may be NULL; may
 *               alias tokens_dev to chain steps on the device).
 * The step runs as one CUDA graph: the first call with a given set of pointers
 * records it (on a stream the library owns) and later calls replay it.  It
 * allocates no device memory after the first call for a pointer set and never
 * synchronises.  A token or position out of range sets a device error flag
 * (er_get_device_error) and leaves that sequence's outputs unspecified; no
 * out-of-range memory is touched.  Any non-finite logit sets the non-finite
 * flag (mirrors greedyToken's hasNonFinite, "EdgeRunner Core Architecture"
 * section 2.3). */
ER_API er_status er_decode_step(const int32_t *tokens_dev, const int32_t *positions_dev, er_kv *kv,
                         float *logits_dev, int32_t *argmax_dev, void *stream);
/* The same kernels queued directly (no graph); for debugging and tests. */
ER_API er_status er_decode_step_eager(const int32_t *tokens_dev, const int32_t *positions_dev, er_kv *kv,
                               float *logits_dev, int32_t *argmax_dev, void *stream);

/* How er_decode_step runs the step:
 *   ER_SCHEDULE_AUTO        persistent when the shape allows it (default)
 *   ER_SCHEDULE_PERSISTENT  one cooperative kernel, one CTA per SM, that runs
 *                           every phase with grid barriers in between and
 *                           streams weights continuously (batch <= 4,
 *                           n_heads / n_kv_heads <= 4, shared memory permitting)
 *   ER_SCHEDULE_KERNELS     one kernel per phase (any supported shape)
 * Both compute the same step; the choice drops kv's recorded graphs.
 * ER_EUNSUPPORTED if PERSISTENT is asked for a shape it cannot run. */
typedef enum { ER_SCHEDULE_AUTO = 0, ER_SCHEDULE_PERSISTENT = 1, ER_SCHEDULE_KERNELS = 2 } er_schedule;
ER_API er_status er_kv_set_schedule(er_kv *kv, int32_t schedule);
/* The schedule in effect (ER_SCHEDULE_PERSISTENT or ER_SCHEDULE_KERNELS), or -1 for NULL. */
ER_API int32_t er_kv_get_schedule(const er_kv *kv);
/* Which kernel runs the one-pass batched GEMV (batches of 5..16, per-phase
 * schedule).  Both compute the same products and epilogues:
 *   ER_WIDE_AUTO       by matrix size: the tcgen05 kernel for matrices of at
 *                      least 2^18 units of 16 rows x 64 columns (such as an
 *                      8B-class LM head), the mma.sync kernel below (default)
 *   ER_WIDE_MMA_SYNC   warp-level mma.sync, weights dequantised in registers
 *   ER_WIDE_TCGEN05    tcgen05.mma, weights dequantised into tensor memory,
 *                      fp32 accumulators in tensor memory
 * The choice drops kv's recorded graphs.  ER_EINVAL for another value; no
 * effect on batches the batched GEMV does not take. */
typedef enum { ER_WIDE_AUTO = 0, ER_WIDE_MMA_SYNC = 1, ER_WIDE_TCGEN05 = 2 } er_wide_gemv;
ER_API er_status er_kv_set_wide_gemv(er_kv *kv, int32_t variant);
/* Kernel launches one er_decode_step enqueues under the schedule in effect
 * (memsets not counted), or -1 for NULL: 1 for the persistent schedule; for
 * the per-phase one, the embedding, per layer the QKV, attention, Wo, gate/up
 * and down launches, and the head.  A GEMV is one launch for batches up to 4
 * and for batches of 5..16 whose matrices take the one-pass batched kernel
 * (K a multiple of 64); otherwise one launch per group of at most 4 batch
 * columns that fit its shared memory. */
ER_API int32_t er_kv_launches_per_step(const er_kv *kv);

/* positions_dev[b] += 1 for b < batch (chains steps without a host round trip). */
ER_API er_status er_positions_increment(int32_t *positions_dev, int32_t batch, void *stream);

/* Synchronises the device, then reports and clears kv's device flags:
 *   *code        bit 0: a token was out of range; bit 1: a position was out of
 *                range; bit 2: a pipeline wait in a kernel gave up (internal
 *                error); 0 if none
 *   *non_finite  1 if any logit since the last call was NaN or infinite
 * Returns ER_EDEVICE if *code != 0, else ER_OK. */
ER_API er_status er_get_device_error(er_kv *kv, int32_t *code, int32_t *non_finite);

/* Recorded step graphs kv holds (one per set of pointers passed to
 * er_decode_step), or -1 for NULL.  At most 8 are kept: a call with a new
 * pointer set beyond that drops the least recently launched graph (a dropped
 * graph still running finishes normally), so a caller that rotates buffers
 * holds a bounded number of graphs. */
ER_API int32_t er_kv_cached_graphs(const er_kv *kv);

/* Failure injection for tests of the bounded waits, on the host side; it
 * mirrors the pages' check of a command buffer's status and timeout ("llama.cpp
 * Metal (MPS) End-to-End Inference Path", step table).  With extra > 0 the
 * first grid barrier of the persistent step waits for `extra` more arrivals
 * than its grid can supply, so every CTA's wait runs out: the kernel returns,
 * er_get_device_error reports bit 2, and that step's outputs are unspecified.
 * extra = 0 (the default) restores normal steps.  Drops kv's recorded graphs;
 * has no effect under ER_SCHEDULE_KERNELS.  ER_EINVAL outside 0..2^20. */
ER_API er_status er_kv_inject_wait_shortfall(er_kv *kv, int32_t extra);
/* Limit of every bounded wait in the library's kernels (grid barriers, ring
 * and pipeline waits), in nanoseconds of %globaltimer, on the current device;
 * 0 restores the default of one second.  Synchronous.  For tests that make a
 * wait run out in milliseconds. */
ER_API er_status er_set_wait_limit_ns(uint64_t ns);
/* Test hooks of the allocation-failure paths.  After er_debug_fail_allocation(n)
 * the library's device allocation number n from now on (0 = the next one)
 * fails as if the device were out of memory, so the call making it returns
 * ER_ENOMEM and frees what it had taken; n = -1 (the default) turns the hook
 * off.  er_debug_live_allocations gives the number of device allocations the
 * library currently holds (models, decode states, matrices). */
ER_API er_status er_debug_fail_allocation(int64_t n);
ER_API int64_t er_debug_live_allocations(void);

/* Stage kernels of the per-phase schedule (ER_SCHEDULE_KERNELS), queued alone
 * with the step's own arguments for layer `layer` (ignored by EMBED and HEAD).
 * For per-kernel timing. */
typedef enum {
    ER_STAGE_EMBED = 0,   /* token row -> residual x                          */
    ER_STAGE_QKV = 1,     /* RMSNorm + [Wq;Wk;Wv] + RoPE + K/V append          */
    ER_STAGE_ATTN = 2,    /* GQA attention (rows split over warps) + merges    */
    ER_STAGE_WO = 3,      /* Wo + residual                                     */
    ER_STAGE_GATEUP = 4,  /* RMSNorm + [Wgate;Wup] + SwiGLU                    */
    ER_STAGE_DOWN = 5,    /* Wdown + residual                                  */
    ER_STAGE_HEAD = 6     /* final RMSNorm + LM head + argmax                  */
} er_stage;
ER_API er_status er_launch_stage(er_kv *kv, int32_t stage, int32_t layer, const int32_t *tokens_dev,
                          const int32_t *positions_dev, float *logits_dev, int32_t *argmax_dev, void *stream);

/* Stand-alone block-quantized matrix ("EdgeRunner Core Architecture" section
 * 3.4, tier 1: the raw blocks feed the product directly).  `blocks_dev` is a
 * GGUF [rows x cols] matrix of type w_type (ER_Q8_0 / ER_Q4_0); it is repacked
 * into memory the er_matrix owns (synchronises `stream`). */
ER_API er_status er_matrix_create(int32_t w_type, int32_t rows, int32_t cols, const void *blocks_dev, void *stream,
                           er_matrix **out);
ER_API void er_matrix_destroy(er_matrix *mat);
/* out_dev fp32 [rows][cols] = d * q of every element, from the repacked bytes
 * (exact: each value has at most 19 significant bits). */
ER_API er_status er_matrix_dequant(const er_matrix *mat, float *out_dev, void *stream);
/* y_dev fp32 [batch][rows] = W x_b for x_dev fp32 [batch][cols], 1 <= batch <= 16.
 * One pass over the weights serves up to 4 batch columns (fewer for very wide
 * rows).  fp32 activations, fp32 accumulation; deterministic. */
ER_API er_status er_matrix_gemv(const er_matrix *mat, const float *x_dev, int32_t batch, float *y_dev, void *stream);

/* The product of er_matrix_gemv for callers that cannot allocate device
 * memory when they run it (a process whose device memory is all handed out by
 * its own pool, code that must not call cudaMalloc while other threads capture
 * CUDA graphs, ...).  The weights are read from `mat`; x_dev and y_dev are the
 * caller's, as for er_matrix_gemv.  The partial sums and counters that
 * er_matrix_gemv keeps in buffers er_matrix_create allocated live here in one
 * array compiled into the library instead: 192.25 KiB per GPU, held by every
 * GPU that loads the library until the process exits.  No cudaMalloc, cudaFree
 * or allocating library call is made.
 *   - The first call on a device looks up the array's device address (with
 *     that device current); make that first call before any stream capture.
 *   - Every call shares the array and it keeps the last call's contents; the
 *     call clears the part that must start at zero.  Calls that overlap on the
 *     GPU (other streams, other threads) race on it: serialise them.
 *   - Limits: at most 262144 rows (16384 row groups) and 256 SMs; larger
 *     matrices give ER_EINVAL, more SMs ER_EUNSUPPORTED.  `mat` must belong to
 *     the current device (else ER_EINVAL).
 *   - A bounded wait that gives up inside a call is not returned by the call
 *     (it is queued asynchronously): er_matrix_gemv_noalloc_error reports it.
 * There is no counterpart on the pages; it exists for this library's callers. */
ER_API er_status er_matrix_gemv_noalloc(const er_matrix *mat, const float *x_dev, int32_t batch, float *y_dev,
                                        void *stream);
/* Synchronises the current device, then reports and clears the flag word of
 * er_matrix_gemv_noalloc's array there: *code = 4 if a bounded wait inside the
 * most recent call on this device gave up (its y_dev is then unspecified),
 * else 0.  Every call clears the flag when it starts, so query after each call
 * whose result matters.  Returns ER_EDEVICE if *code != 0.  Allocates nothing.
 * No counterpart on the pages. */
ER_API er_status er_matrix_gemv_noalloc_error(int32_t *code);

/* GGUF container ("EdgeRunner Core Architecture" section 2.2, Model Loading:
 * the loader maps the file and parses the model configuration from its
 * metadata; "alpaca.swift" Capabilities: GGUF v2/v3, F16/Q8_0/Q4_0 tensors).
 * The file is treated as untrusted: every count, length, dimension and offset
 * is checked against the bytes present (overflow-checked) before use, and a
 * malformed file gives ER_EINVAL with the reason in er_last_error().
 *
 * er_gguf_open maps `path` read-only (host memory, owned by the handle until
 * er_gguf_close) and parses the header, metadata and tensor table.  Data
 * pointers returned below point into that mapping. */
typedef struct er_gguf er_gguf;
ER_API er_status er_gguf_open(const char *path, er_gguf **out);
ER_API void er_gguf_close(er_gguf *g);
/* Tensors in the file (-1 for NULL). */
ER_API int64_t er_gguf_tensor_count(const er_gguf *g);
/* Tensor i: its NUL-terminated name, GGUF type code (er_dtype values for the
 * types this library computes with), dimension count, dims[4] (innermost
 * first: a matrix of `rows` x `cols` has dims {cols, rows, 1, 1}), its bytes in
 * the mapping and their count.  Any output pointer may be NULL. */
ER_API er_status er_gguf_tensor_info(const er_gguf *g, int64_t i, const char **name, int32_t *type, int32_t *n_dims,
                                     int64_t *dims, const void **data, uint64_t *bytes);
/* Index of the tensor named `name` (ER_EINVAL if absent). */
ER_API er_status er_gguf_find(const er_gguf *g, const char *name, int64_t *index);
/* The model shape from the llama.* metadata ("EdgeRunner Core Architecture"
 * section 1.1: embedding_length, block_count, feed_forward_length,
 * attention.head_count, attention.head_count_kv (default: head_count),
 * attention.key_length (default: embedding_length / head_count),
 * rope.freq_base (default 10000), attention.layer_norm_rms_epsilon (default
 * 1e-5)); vocab from token_embd.weight; w_type from blk.0.attn_q.weight; tied
 * when output.weight is absent; max_batch as given.  Every tensor the decode
 * step reads is checked to exist with the type and shape this implies:
 * ER_EINVAL (reason in er_last_error) otherwise. */
ER_API er_status er_gguf_config(const er_gguf *g, int32_t max_batch, er_config *cfg);
/* er_model_create from the file: the data section is copied to the device
 * once, handed to er_model_create (which repacks it into model-owned memory)
 * and freed.  Synchronises `stream`.  The er_gguf may be closed afterwards. */
ER_API er_status er_model_create_from_gguf(const er_gguf *g, int32_t max_batch, void *stream, er_model **out);

ER_API const char *er_status_str(er_status s);
ER_API const char *er_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* ER_H */
