// The C ABI (include/er.h): argument checks, memory ownership, the decode
// step's kernel schedule and its CUDA-graph cache.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <string>

#include "common.cuh"
#include "internal.h"
#include "layout.cuh"

using namespace er;

namespace {

thread_local std::string g_last_error;

er_status fail(er_status s, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
er_status fail(er_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

er_status cuda_fail(cudaError_t e, const char *what) {
    return fail(e == cudaErrorMemoryAllocation ? ER_ENOMEM : ER_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define ER_CUDA(call)                                        \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);  \
    } while (0)

// Test hooks of the allocation-failure paths: the allocation numbered
// g_alloc_fail_at from the hook's setting on fails as if the device were out
// of memory (-1: never), and g_live_allocs counts the device allocations the
// library holds.
std::atomic<long long> g_alloc_fail_at{-1};
std::atomic<long long> g_live_allocs{0};

template <class T>
cudaError_t dalloc(std::vector<void *> &owner, T **p, size_t bytes) {
    if (g_alloc_fail_at.load() >= 0 && g_alloc_fail_at.fetch_sub(1) == 0) return cudaErrorMemoryAllocation;
    void *q = nullptr;
    cudaError_t e = cudaMalloc(&q, bytes ? bytes : 16);
    if (e != cudaSuccess) return e;
    owner.push_back(q);
    ++g_live_allocs;
    *p = reinterpret_cast<T *>(q);
    return cudaSuccess;
}

void free_all(std::vector<void *> &owner) {
    for (void *p : owner) cudaFree(p);
    g_live_allocs -= (long long)owner.size();
    owner.clear();
}

int rows_per_group(int rowmap) { return rowmap == MAP_GATEUP ? 8 : 16; }

Mat mat_shape(int qt, int rowmap, int N, int K) {
    Mat m;
    m.qt = qt;
    m.rowmap = rowmap;
    m.N = N;
    m.K = K;
    int rpg = rows_per_group(rowmap);
    m.R = (N + rpg - 1) / rpg;
    m.UPR = ((K / 32) + 1) / 2;
    m.bytes = (size_t)m.R * m.UPR * unit_bytes_of(qt);
    return m;
}

bool valid_qt(int t) { return t == ER_Q8_0 || t == ER_Q4_0; }

int device_sms(int *dev) {
    int n = 0;
    if (cudaGetDevice(dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

cudaError_t er::device_alloc(void **p, size_t bytes) {
    std::vector<void *> own;
    return dalloc(own, p, bytes);
}

void er::device_free(void *p) {
    if (!p) return;
    cudaFree(p);
    --g_live_allocs;
}

// error reporting for entry points defined in other files
er_status er_fail_status(er_status s, const char *msg) { return fail(s, "%s", msg); }
er_status er_fail_cuda(cudaError_t e, const char *what) { return cuda_fail(e, what); }

extern "C" {

const char *er_status_str(er_status s) {
    switch (s) {
        case ER_OK: return "ok";
        case ER_EINVAL: return "invalid argument";
        case ER_ENOMEM: return "out of device memory";
        case ER_ECUDA: return "CUDA error";
        case ER_EUNSUPPORTED: return "unsupported";
        case ER_EDEVICE: return "device-side error flag set";
    }
    return "unknown status";
}

const char *er_last_error(void) { return g_last_error.c_str(); }

// ---------------------------------------------------------------------------
// model
// ---------------------------------------------------------------------------
static er_status check_config(const er_config *c) {
    if (!c) return fail(ER_EINVAL, "config is NULL");
    if (c->dim <= 0 || c->n_layers <= 0 || c->n_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
        c->ffn_dim <= 0 || c->vocab <= 0)
        return fail(ER_EINVAL, "config sizes must be positive");
    if (c->n_heads % c->n_kv_heads) return fail(ER_EINVAL, "n_heads must be a multiple of n_kv_heads");
    if (c->n_heads / c->n_kv_heads > 8) return fail(ER_EUNSUPPORTED, "more than 8 query heads per KV head");
    if (c->head_dim != 64 && c->head_dim != 128) return fail(ER_EUNSUPPORTED, "head_dim must be 64 or 128");
    if (c->dim % 32 || c->ffn_dim % 32) return fail(ER_EINVAL, "dim and ffn_dim must be multiples of 32");
    if (!valid_qt(c->w_type)) return fail(ER_EINVAL, "w_type must be ER_Q8_0 or ER_Q4_0");
    if (c->tied != 0 && c->tied != 1) return fail(ER_EINVAL, "tied must be 0 or 1");
    if (c->max_batch < 1 || c->max_batch > 16) return fail(ER_EINVAL, "max_batch must be in 1..16");
    if (!(c->rope_base > 0) || !(c->rms_eps >= 0)) return fail(ER_EINVAL, "rope_base must be > 0, rms_eps >= 0");
    if ((long long)c->n_heads * c->head_dim > (1 << 20) || (long long)c->dim > (1 << 20) ||
        (long long)c->ffn_dim > (1 << 20))
        return fail(ER_EINVAL, "dimension too large");
    // every GEMV input width must fit the kernel's shared-memory operand for one column
    int K[3] = {c->dim, c->n_heads * c->head_dim, c->ffn_dim};
    for (int k : K)
        if (gemv_max_cols(c->w_type, k) < 1) return fail(ER_EUNSUPPORTED, "input width %d too large", k);
    return ER_OK;
}

static cudaError_t make_mat(er_model *m, Mat *out, int qt, int rowmap, int N, int K, const RepackSrc &src,
                            cudaStream_t st) {
    *out = mat_shape(qt, rowmap, N, K);
    cudaError_t e = dalloc(m->allocs, &out->d, out->bytes);
    if (e != cudaSuccess) return e;
    m->device_bytes += out->bytes;
    return launch_repack(*out, src, st);
}

static RepackSrc src1(const void *p, int rows) {
    RepackSrc s = {};
    s.p[0] = (const uint8_t *)p;
    s.rows[0] = rows;
    s.nsrc = 1;
    return s;
}

er_status er_model_create(const er_config *cfg, const er_weights *w, void *stream, er_model **out) {
    if (!out) return fail(ER_EINVAL, "out is NULL");
    er_status s = check_config(cfg);
    if (s != ER_OK) return s;
    if (!w || !w->layers || !w->tok_embd || !w->output_norm) return fail(ER_EINVAL, "weights incomplete");
    if (cfg->tied ? (w->output != nullptr) : (w->output == nullptr))
        return fail(ER_EINVAL, "output must be NULL iff tied");
    for (int l = 0; l < cfg->n_layers; ++l) {
        const er_layer_weights &L = w->layers[l];
        if (!L.attn_norm || !L.wq || !L.wk || !L.wv || !L.wo || !L.ffn_norm || !L.w_gate || !L.w_up || !L.w_down)
            return fail(ER_EINVAL, "layer %d has a NULL weight", l);
    }
    cudaStream_t st = (cudaStream_t)stream;
    er_model *m = new er_model();
    m->cfg = *cfg;
    m->num_sms = device_sms(&m->device);
    m->device_bytes = 0;
    m->embd_f16 = nullptr;
    if (m->num_sms <= 0) {
        delete m;
        return fail(ER_ECUDA, "no CUDA device");
    }
    cudaError_t e = gemv_prepare();
    const int D = cfg->dim, qd = cfg->n_heads * cfg->head_dim, kvd = cfg->n_kv_heads * cfg->head_dim;
    const int F = cfg->ffn_dim, V = cfg->vocab, qt = cfg->w_type;
    m->layers.resize(cfg->n_layers);
    for (int l = 0; l < cfg->n_layers && e == cudaSuccess; ++l) {
        const er_layer_weights &L = w->layers[l];
        er_layer_dev &d = m->layers[l];
        RepackSrc qkv = {};
        qkv.p[0] = (const uint8_t *)L.wq;
        qkv.p[1] = (const uint8_t *)L.wk;
        qkv.p[2] = (const uint8_t *)L.wv;
        qkv.rows[0] = qd;
        qkv.rows[1] = kvd;
        qkv.rows[2] = kvd;
        qkv.nsrc = 3;
        e = make_mat(m, &d.qkv, qt, MAP_PAIR, qd + 2 * kvd, D, qkv, st);
        if (e == cudaSuccess) e = make_mat(m, &d.wo, qt, MAP_IDENT, D, qd, src1(L.wo, D), st);
        RepackSrc gu = {};
        gu.p[0] = (const uint8_t *)L.w_gate;
        gu.p[1] = (const uint8_t *)L.w_up;
        gu.rows[0] = F;
        gu.rows[1] = F;
        gu.nsrc = 2;
        if (e == cudaSuccess) e = make_mat(m, &d.gateup, qt, MAP_GATEUP, F, D, gu, st);
        if (e == cudaSuccess) e = make_mat(m, &d.down, qt, MAP_IDENT, D, F, src1(L.w_down, D), st);
        if (e == cudaSuccess) e = dalloc(m->allocs, &d.attn_norm, D * sizeof(float));
        if (e == cudaSuccess) e = dalloc(m->allocs, &d.ffn_norm, D * sizeof(float));
        if (e == cudaSuccess) e = cudaMemcpyAsync(d.attn_norm, L.attn_norm, D * sizeof(float), cudaMemcpyDefault, st);
        if (e == cudaSuccess) e = cudaMemcpyAsync(d.ffn_norm, L.ffn_norm, D * sizeof(float), cudaMemcpyDefault, st);
        m->device_bytes += 2 * D * sizeof(float);
    }
    if (e == cudaSuccess)
        e = make_mat(m, &m->head, qt, MAP_IDENT, V, D, src1(cfg->tied ? w->tok_embd : w->output, V), st);
    if (e == cudaSuccess && !cfg->tied) {
        e = dalloc(m->allocs, &m->embd_f16, (size_t)V * D * sizeof(__half));
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(m->embd_f16, w->tok_embd, (size_t)V * D * sizeof(__half), cudaMemcpyDefault, st);
        m->device_bytes += (size_t)V * D * sizeof(__half);
    }
    if (e == cudaSuccess) e = dalloc(m->allocs, &m->out_norm, D * sizeof(float));
    if (e == cudaSuccess) e = cudaMemcpyAsync(m->out_norm, w->output_norm, D * sizeof(float), cudaMemcpyDefault, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        cudaStreamSynchronize(st);
        free_all(m->allocs);
        delete m;
        return cuda_fail(e, "er_model_create");
    }
    *out = m;
    return ER_OK;
}

void er_model_destroy(er_model *m) {
    if (!m) return;
    free_all(m->allocs);
    delete m;
}

size_t er_model_device_bytes(const er_model *m) { return m ? m->device_bytes : 0; }

// ---------------------------------------------------------------------------
// decode state
// ---------------------------------------------------------------------------
er_status er_kv_create(er_model *m, int32_t batch, int32_t capacity, er_kv **out) {
    return er_kv_create_typed(m, batch, capacity, ER_F16, out);
}

// A decode state; with `owner`, a 16-column prefill view of the owner's cache: it allocates its own
// activations and scratch but takes the owner's cache and flag word.
static er_status kv_create(er_model *m, int32_t batch, int32_t capacity, int32_t kv_type, er_kv *owner,
                           er_kv **out) {
    const er_config &c = m->cfg;
    er_kv *kv = new er_kv();
    kv->m = m;
    kv->B = batch;
    kv->cap = capacity;
    kv->kv_type = kv_type;
    kv->kc = kv->vc = nullptr;
    kv->kvq = {};
    kv->kstage = kv->vstage = nullptr;
    kv->seqmap = nullptr;
    kv->pf = nullptr;
    kv->view = owner != nullptr;
    kv->pf_pos = kv->pf_seq = nullptr;
    kv->pf_logits = nullptr;
    kv->cap_stream = nullptr;
    kv->graph_calls = 0;
    kv->bar_extra = 0;
    const int D = c.dim, qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim, F = c.ffn_dim, hd = c.head_dim;
    const int G = c.n_heads / c.n_kv_heads;
    attention_plan(hd, c.n_kv_heads, batch, capacity, m->num_sms, &kv->S, &kv->CH);
    int max_r = m->head.R;
    for (auto &L : m->layers) {
        max_r = max_r > L.qkv.R ? max_r : L.qkv.R;
        max_r = max_r > L.wo.R ? max_r : L.wo.R;
        max_r = max_r > L.gateup.R ? max_r : L.gateup.R;
        max_r = max_r > L.down.R ? max_r : L.down.R;
    }
    size_t cache_elems = (size_t)batch * c.n_layers * kvd * (size_t)capacity;
    cudaError_t e = cudaSuccess;
    auto A = [&](auto **p, size_t bytes, bool zero = true) {
        if (e != cudaSuccess) return;
        e = dalloc(kv->allocs, p, bytes);
        if (e == cudaSuccess && zero) e = cudaMemset(*p, 0, bytes);
    };
    if (owner) {
        kv->kc = owner->kc;
        kv->vc = owner->vc;
        kv->kvq = owner->kvq;
        A(&kv->pf_pos, 16 * sizeof(int32_t));
        A(&kv->pf_seq, 16 * sizeof(int32_t));
        A(&kv->pf_logits, (size_t)16 * c.vocab * sizeof(float), false);
        kv->seqmap = kv->pf_seq;
    } else if (kv_type == ER_F16) {
        A(&kv->kc, cache_elems * sizeof(__half));
        A(&kv->vc, cache_elems * sizeof(__half));
    } else {
        const int rows = (capacity + 15) & ~15;  // whole tiles of 16 rows per head
        const size_t q_elems = cache_elems / capacity * rows;
        A(&kv->kvq.kq, q_elems, false);  // codes are stored as q XOR 0x80: 0x80 is a zero code
        A(&kv->kvq.vq, q_elems, false);
        if (e == cudaSuccess) e = cudaMemset(kv->kvq.kq, 0x80, q_elems);
        if (e == cudaSuccess) e = cudaMemset(kv->kvq.vq, 0x80, q_elems);
        A(&kv->kvq.kd, q_elems / 32 * sizeof(__half));
        A(&kv->kvq.vd, q_elems / 32 * sizeof(__half));
        kv->kvq.L = c.n_layers;
        kv->kvq.KV = c.n_kv_heads;
        kv->kvq.cap = capacity;
        kv->kvq.rows = rows;
    }
    if (kv_type == ER_Q8_0) {
        A(&kv->kstage, (size_t)batch * kvd * sizeof(float));
        A(&kv->vstage, (size_t)batch * kvd * sizeof(float));
    }
    A(&kv->rope, (size_t)capacity * (hd / 2) * sizeof(float2), false);
    A(&kv->x, (size_t)batch * D * sizeof(float));
    A(&kv->q, (size_t)batch * qd * sizeof(float));
    A(&kv->o, (size_t)batch * qd * sizeof(float));
    A(&kv->a, (size_t)batch * F * sizeof(float));
    A(&kv->attn_part, attention_part_floats(hd, G, m->num_sms) * sizeof(float));
    A(&kv->attn_cnt, (size_t)batch * c.n_kv_heads * sizeof(int));
    A(&kv->gemv_part, gemv_part_floats(m->num_sms) * sizeof(float));
    A(&kv->gemv_cnt, (size_t)max_r * sizeof(int));
    // batched GEMV (one pass over the weights for the whole batch) where every matrix takes it
    kv->wide_part = kv->wide_ssq = nullptr;
    if (batch > 4) {  // more columns than one pass of the batch-1 GEMV takes
        bool ok = true;
        size_t part = 0, ssq = 0;
        auto need = [&](const er::Mat &w) {
            ok = ok && gemv_wide_fits(w.qt, w.K, batch, m->num_sms) && gemv_tc_fits(w.qt, w.K, batch, m->num_sms);
            part = std::max(part, gemv_wide_part_floats(w.R, w.K));
            ssq = std::max(ssq, gemv_wide_ssq_floats(w.K));
        };
        for (int l = 0; l < c.n_layers; ++l) {
            need(m->layers[l].qkv);
            need(m->layers[l].wo);
            need(m->layers[l].gateup);
            need(m->layers[l].down);
        }
        need(m->head);
        if (ok) {
            A(&kv->wide_part, std::max<size_t>(part, 1) * sizeof(float), false);
            A(&kv->wide_ssq, ssq * sizeof(float), false);
        }
    }
    A(&kv->amax, 16 * sizeof(unsigned long long));
    A(&kv->done, sizeof(int));
    if (owner)
        kv->flags = owner->flags;  // prefill errors show in the owner's er_get_device_error
    else
        A(&kv->flags, sizeof(int));
    if (e == cudaSuccess) {
        // RoPE table: angle p * base^(-2i/hd) in double, cos/sin rounded to fp32
        std::vector<float2> cs((size_t)capacity * (hd / 2));
        for (int p = 0; p < capacity; ++p)
            for (int i = 0; i < hd / 2; ++i) {
                double th = (double)p * pow(c.rope_base, -2.0 * i / hd);
                cs[(size_t)p * (hd / 2) + i] = make_float2((float)cos(th), (float)sin(th));
            }
        e = cudaMemcpy(kv->rope, cs.data(), cs.size() * sizeof(float2), cudaMemcpyHostToDevice);
    }
    // persistent step: layer table, attention partial states, grid barrier
    {
        const int max_k = D > qd ? (D > F ? D : F) : (qd > F ? qd : F);
        const er::Mat *mats[5] = {&m->layers[0].qkv, &m->layers[0].wo, &m->layers[0].gateup, &m->layers[0].down,
                                  &m->head};
        int R[5], UPR[5];
        for (int i = 0; i < 5; ++i) {
            R[i] = mats[i]->R;
            UPR[i] = mats[i]->UPR;
        }
        kv->step_ok = e == cudaSuccess && kv_type == ER_F16 && !owner &&
                      step_supported(c.w_type, hd, G, batch, c.n_kv_heads, capacity, max_k, R, UPR, m->num_sms);
        kv->schedule = kv->step_ok ? ER_SCHEDULE_PERSISTENT : ER_SCHEDULE_KERNELS;
        A(&kv->step_layers, (size_t)c.n_layers * sizeof(StepLayer), false);
        A(&kv->step_apart, step_apart_floats(m->num_sms, hd) * sizeof(float), false);
        A(&kv->step_acnt, (size_t)batch * c.n_kv_heads * sizeof(int));
        A(&kv->step_bar, sizeof(unsigned));
        if (e == cudaSuccess) {
            std::vector<StepLayer> ls(c.n_layers);
            for (int l = 0; l < c.n_layers; ++l) {
                const er_layer_dev &L = m->layers[l];
                ls[l].w[0] = L.qkv.d;
                ls[l].w[1] = L.wo.d;
                ls[l].w[2] = L.gateup.d;
                ls[l].w[3] = L.down.d;
                ls[l].attn_norm = L.attn_norm;
                ls[l].ffn_norm = L.ffn_norm;
            }
            e = cudaMemcpy(kv->step_layers, ls.data(), ls.size() * sizeof(StepLayer), cudaMemcpyHostToDevice);
        }
    }
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&kv->cap_stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        free_all(kv->allocs);
        if (kv->cap_stream) cudaStreamDestroy(kv->cap_stream);
        delete kv;
        return cuda_fail(e, "er_kv_create");
    }
    *out = kv;
    return ER_OK;
}

er_status er_kv_create_typed(er_model *m, int32_t batch, int32_t capacity, int32_t kv_type, er_kv **out) {
    if (!m || !out) return fail(ER_EINVAL, "NULL argument");
    const er_config &c = m->cfg;
    if (batch < 1 || batch > c.max_batch) return fail(ER_EINVAL, "batch must be in 1..max_batch");
    if (capacity < 1 || capacity > (1 << 24)) return fail(ER_EINVAL, "capacity out of range");
    if (kv_type != ER_F16 && kv_type != ER_Q8_0) return fail(ER_EINVAL, "kv_type must be ER_F16 or ER_Q8_0");
    return kv_create(m, batch, capacity, kv_type, nullptr, out);
}

void er_kv_destroy(er_kv *kv) {
    if (!kv) return;
    er_kv_destroy(kv->pf);
    for (auto &g : kv->graphs) cudaGraphExecDestroy(g.exec);
    if (kv->cap_stream) cudaStreamDestroy(kv->cap_stream);
    free_all(kv->allocs);
    delete kv;
}

int32_t er_kv_type(const er_kv *kv) { return kv ? kv->kv_type : -1; }

er_status er_kv_layer_ptrs(er_kv *kv, int32_t seq, int32_t layer, void **k_dev, void **v_dev) {
    if (!kv || !k_dev || !v_dev) return fail(ER_EINVAL, "NULL argument");
    if (kv->kv_type != ER_F16) return fail(ER_EUNSUPPORTED, "the cache holds Q8_0 blocks, not fp16 rows");
    const er_config &c = kv->m->cfg;
    if (seq < 0 || seq >= kv->B || layer < 0 || layer >= c.n_layers) return fail(ER_EINVAL, "seq or layer out of range");
    size_t off = ((size_t)seq * c.n_layers + layer) * (size_t)c.n_kv_heads * kv->cap * c.head_dim;
    *k_dev = kv->kc + off;
    *v_dev = kv->vc + off;
    return ER_OK;
}

static er_status kv_copy(er_kv *kv, int seq, int layer, int start, int n, bool write, void *k, void *v,
                         cudaStream_t st) {
    if (!kv || !k || !v) return fail(ER_EINVAL, "NULL argument");
    const er_config &c = kv->m->cfg;
    if (seq < 0 || seq >= kv->B || layer < 0 || layer >= c.n_layers) return fail(ER_EINVAL, "seq or layer out of range");
    if (n < 0 || start < 0 || (long long)start + n > kv->cap) return fail(ER_EINVAL, "rows out of range");
    if (n == 0) return ER_OK;
    const int hd = c.head_dim, kvd = c.n_kv_heads * hd;
    if (kv->kv_type == ER_Q8_0) {
        if (!write) return fail(ER_EUNSUPPORTED, "the cache holds Q8_0 blocks: read them with er_kv_read_blocks");
        ER_CUDA(launch_kvq_write((const __half *)k, (const __half *)v, n, kv->kvq, hd, seq, layer, start, st));
        return ER_OK;
    }
    size_t base = ((size_t)seq * c.n_layers + layer) * (size_t)c.n_kv_heads * kv->cap * hd;
    for (int h = 0; h < c.n_kv_heads; ++h) {
        __half *ck = kv->kc + base + ((size_t)h * kv->cap + start) * hd;
        __half *cv = kv->vc + base + ((size_t)h * kv->cap + start) * hd;
        __half *rk = (__half *)k + (size_t)h * hd;
        __half *rv = (__half *)v + (size_t)h * hd;
        const size_t w = hd * sizeof(__half), rp = kvd * sizeof(__half);
        if (write) {
            ER_CUDA(cudaMemcpy2DAsync(ck, w, rk, rp, w, n, cudaMemcpyDeviceToDevice, st));
            ER_CUDA(cudaMemcpy2DAsync(cv, w, rv, rp, w, n, cudaMemcpyDeviceToDevice, st));
        } else {
            ER_CUDA(cudaMemcpy2DAsync(rk, rp, ck, w, w, n, cudaMemcpyDeviceToDevice, st));
            ER_CUDA(cudaMemcpy2DAsync(rv, rp, cv, w, w, n, cudaMemcpyDeviceToDevice, st));
        }
    }
    return ER_OK;
}

er_status er_kv_write(er_kv *kv, int32_t seq, int32_t layer, int32_t start, int32_t n, const void *k, const void *v,
                      void *stream) {
    return kv_copy(kv, seq, layer, start, n, true, (void *)k, (void *)v, (cudaStream_t)stream);
}

er_status er_kv_read(er_kv *kv, int32_t seq, int32_t layer, int32_t start, int32_t n, void *k, void *v,
                     void *stream) {
    return kv_copy(kv, seq, layer, start, n, false, k, v, (cudaStream_t)stream);
}

er_status er_kv_read_blocks(er_kv *kv, int32_t seq, int32_t layer, int32_t start, int32_t n, void *k_blocks,
                            void *v_blocks, void *stream) {
    if (!kv || !k_blocks || !v_blocks) return fail(ER_EINVAL, "NULL argument");
    if (kv->kv_type != ER_Q8_0) return fail(ER_EUNSUPPORTED, "the cache holds fp16 rows: read them with er_kv_read");
    const er_config &c = kv->m->cfg;
    if (seq < 0 || seq >= kv->B || layer < 0 || layer >= c.n_layers) return fail(ER_EINVAL, "seq or layer out of range");
    if (n < 0 || start < 0 || (long long)start + n > kv->cap) return fail(ER_EINVAL, "rows out of range");
    if (n == 0) return ER_OK;
    ER_CUDA(launch_kvq_read((uint8_t *)k_blocks, (uint8_t *)v_blocks, n, kv->kvq, c.head_dim, seq, layer, start,
                            (cudaStream_t)stream));
    return ER_OK;
}

// ---------------------------------------------------------------------------
// the step schedule
// ---------------------------------------------------------------------------
static GemvArgs gemv_base(er_kv *kv, const Mat &w) {
    GemvArgs a = {};
    a.W = w.d;
    a.R = w.R;
    a.UPR = w.UPR;
    a.N = w.N;
    a.K = w.K;
    a.qt = w.qt;
    a.eps = (float)kv->m->cfg.rms_eps;
    a.part = kv->gemv_part;
    a.cnt = kv->gemv_cnt;
    a.flags = kv->flags;
    a.amax = kv->amax;
    a.done = kv->done;
    return a;
}

// one GEMV over the whole batch: one pass for a batch of more than 4 columns
// where the batched kernel takes it, else as few column groups as the kernel takes
static cudaError_t gemv_all(er_kv *kv, int epi, GemvArgs a, cudaStream_t st, bool pdl) {
    if (kv->wide_part) {
        a.b0 = 0;
        a.B = kv->B;
        return launch_gemv_wide(epi, a, kv->wide_part, kv->wide_ssq, kv->m->num_sms, st, pdl, kv->wide_variant);
    }
    int per = gemv_max_cols(a.qt, a.K);
    for (int b0 = 0; b0 < kv->B; b0 += per) {
        a.b0 = b0;
        a.B = kv->B - b0 < per ? kv->B - b0 : per;
        cudaError_t e = launch_gemv(epi, a, kv->m->num_sms, st, pdl);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

static cudaError_t enqueue_stage(er_kv *kv, int stage, int l, const int32_t *tokens, const int32_t *positions,
                                 float *logits, int32_t *argmax, cudaStream_t st, bool pdl) {
    er_model *m = kv->m;
    const er_config &c = m->cfg;
    const int qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
    switch (stage) {
        case ER_STAGE_EMBED: {
            EmbedArgs e = {};
            e.tokens = tokens;
            e.positions = positions;
            e.embd_f16 = c.tied ? nullptr : m->embd_f16;
            e.head = m->head;
            e.x = kv->x;
            e.B = kv->B;
            e.D = c.dim;
            e.V = c.vocab;
            e.cap = kv->cap;
            e.flags = kv->flags;
            return launch_embed(e, st, pdl);
        }
        case ER_STAGE_QKV: {
            const er_layer_dev &L = m->layers[l];
            GemvArgs a = gemv_base(kv, L.qkv);
            a.x = kv->x;
            a.gain = L.attn_norm;
            a.q_out = kv->q;
            a.kc = kv->kc;
            a.vc = kv->vc;
            a.rope = kv->rope;
            a.positions = positions;
            a.qd = qd;
            a.kvd = kvd;
            a.hd = c.head_dim;
            a.KV = c.n_kv_heads;
            a.L = c.n_layers;
            a.layer = l;
            a.cap = kv->cap;
            a.k_stage = kv->kstage;  // Q8_0 cache: fp32 rows, quantised by the next launch
            a.v_stage = kv->vstage;
            a.seqmap = kv->seqmap;
            cudaError_t e = gemv_all(kv, EPI_QKV, a, st, pdl);
            // Q8_0 cache: the attention kernel quantises each sequence's new rows itself, except in a prefill
            // chunk, whose columns read each other's new rows: those are quantised first, by their own launch
            if (e == cudaSuccess && kv->kv_type == ER_Q8_0 && kv->seqmap)
                e = launch_kvq_stage(kv->kstage, kv->vstage, positions, kv->seqmap, kv->B, kv->kvq, c.head_dim, l,
                                     st, pdl);
            return e;
        }
        case ER_STAGE_ATTN: {
            AttnArgs a = {};
            a.q = kv->q;
            a.kc = kv->kc;
            a.vc = kv->vc;
            a.kq = kv->kvq.kq;  // nullptr on an fp16 cache
            a.vq = kv->kvq.vq;
            a.kd = kv->kvq.kd;
            a.vd = kv->kvq.vd;
            a.seqmap = kv->seqmap;
            if (kv->kv_type == ER_Q8_0 && !kv->seqmap) {
                a.k_stage = kv->kstage;
                a.v_stage = kv->vstage;
            }
            a.positions = positions;
            a.o = kv->o;
            a.part = kv->attn_part;
            a.cnt = kv->attn_cnt;
            a.flags = kv->flags;
            a.B = kv->B;
            a.H = c.n_heads;
            a.KV = c.n_kv_heads;
            a.hd = c.head_dim;
            a.L = c.n_layers;
            a.layer = l;
            a.cap = kv->cap;
            a.S = kv->S;
            a.CH = kv->CH;
            return launch_attention(a, st, pdl);
        }
        case ER_STAGE_WO: {
            GemvArgs a = gemv_base(kv, m->layers[l].wo);
            a.x = kv->o;
            a.y = kv->x;
            return gemv_all(kv, EPI_RESID, a, st, pdl);
        }
        case ER_STAGE_GATEUP: {
            const er_layer_dev &L = m->layers[l];
            GemvArgs a = gemv_base(kv, L.gateup);
            a.x = kv->x;
            a.gain = L.ffn_norm;
            a.a_out = kv->a;
            return gemv_all(kv, EPI_SWIGLU, a, st, pdl);
        }
        case ER_STAGE_DOWN: {
            GemvArgs a = gemv_base(kv, m->layers[l].down);
            a.x = kv->a;
            a.y = kv->x;
            return gemv_all(kv, EPI_RESID, a, st, pdl);
        }
        case ER_STAGE_HEAD: {
            GemvArgs a = gemv_base(kv, m->head);
            a.x = kv->x;
            a.gain = m->out_norm;
            a.y = logits;
            a.argmax_out = argmax;
            return gemv_all(kv, EPI_LOGITS, a, st, pdl);
        }
    }
    return cudaErrorInvalidValue;
}

static cudaError_t enqueue_persistent(er_kv *kv, const int32_t *tokens, const int32_t *positions, float *logits,
                                      int32_t *argmax, cudaStream_t st) {
    er_model *m = kv->m;
    const er_config &c = m->cfg;
    StepArgs a = {};
    a.layers = kv->step_layers;
    a.head = m->head.d;
    a.out_norm = m->out_norm;
    a.embd_f16 = c.tied ? nullptr : m->embd_f16;
    a.L = c.n_layers;
    a.D = c.dim;
    a.H = c.n_heads;
    a.KV = c.n_kv_heads;
    a.hd = c.head_dim;
    a.F = c.ffn_dim;
    a.V = c.vocab;
    a.qd = c.n_heads * c.head_dim;
    a.kvd = c.n_kv_heads * c.head_dim;
    a.B = kv->B;
    a.cap = kv->cap;
    const er::Mat *mats[5] = {&m->layers[0].qkv, &m->layers[0].wo, &m->layers[0].gateup, &m->layers[0].down, &m->head};
    for (int i = 0; i < 5; ++i) {
        a.R[i] = mats[i]->R;
        a.UPR[i] = mats[i]->UPR;
    }
    a.eps = (float)c.rms_eps;
    a.tokens = tokens;
    a.positions = positions;
    a.x = kv->x;
    a.q = kv->q;
    a.o = kv->o;
    a.a = kv->a;
    a.kc = kv->kc;
    a.vc = kv->vc;
    a.rope = kv->rope;
    a.logits = logits;
    a.argmax = argmax;
    a.part = kv->gemv_part;
    a.cnt = kv->gemv_cnt;
    a.apart = kv->step_apart;
    a.acnt = kv->step_acnt;
    a.amax = kv->amax;
    a.done = kv->done;
    a.flags = kv->flags;
    a.bar = kv->step_bar;
    a.bar_extra = kv->bar_extra;
    cudaError_t e = cudaMemsetAsync(kv->step_bar, 0, sizeof(unsigned), st);
    if (e == cudaSuccess) e = launch_step(c.w_type, a, m->num_sms, st);
    return e;
}

static cudaError_t enqueue_step(er_kv *kv, const int32_t *tokens, const int32_t *positions, float *logits,
                                int32_t *argmax, cudaStream_t st, bool pdl) {
    if (kv->schedule == ER_SCHEDULE_PERSISTENT) return enqueue_persistent(kv, tokens, positions, logits, argmax, st);
    cudaError_t e = enqueue_stage(kv, ER_STAGE_EMBED, 0, tokens, positions, logits, argmax, st, pdl);
    for (int l = 0; l < kv->m->cfg.n_layers && e == cudaSuccess; ++l)
        for (int s = ER_STAGE_QKV; s <= ER_STAGE_DOWN && e == cudaSuccess; ++s)
            e = enqueue_stage(kv, s, l, tokens, positions, logits, argmax, st, pdl);
    if (e == cudaSuccess) e = enqueue_stage(kv, ER_STAGE_HEAD, 0, tokens, positions, logits, argmax, st, pdl);
    return e;
}

static er_status check_step(const int32_t *tokens, const int32_t *positions, er_kv *kv) {
    if (!kv) return fail(ER_EINVAL, "kv is NULL");
    if (!tokens || !positions) return fail(ER_EINVAL, "tokens and positions are required");
    return ER_OK;
}

er_status er_decode_step_eager(const int32_t *tokens, const int32_t *positions, er_kv *kv, float *logits,
                               int32_t *argmax, void *stream) {
    er_status s = check_step(tokens, positions, kv);
    if (s != ER_OK) return s;
    ER_CUDA(enqueue_step(kv, tokens, positions, logits, argmax, (cudaStream_t)stream, false));
    return ER_OK;
}

er_status er_decode_step(const int32_t *tokens, const int32_t *positions, er_kv *kv, float *logits, int32_t *argmax,
                         void *stream) {
    er_status s = check_step(tokens, positions, kv);
    if (s != ER_OK) return s;
    cudaGraphExec_t exec = nullptr;
    const unsigned long long now = ++kv->graph_calls;
    for (auto &g : kv->graphs)
        if (g.tokens == tokens && g.positions == positions && g.logits == logits && g.argmax == argmax) {
            exec = g.exec;
            g.last_use = now;
            break;
        }
    if (!exec) {
        if (kv->graphs.size() >= ER_MAX_GRAPHS) {  // drop the least recently launched graph
            auto lru = std::min_element(kv->graphs.begin(), kv->graphs.end(),
                                        [](const er_graph_entry &x, const er_graph_entry &y) {
                                            return x.last_use < y.last_use;
                                        });
            // an executable graph still in flight is freed when it completes
            cudaGraphExecDestroy(lru->exec);
            kv->graphs.erase(lru);
        }
        cudaGraph_t graph = nullptr;
        ER_CUDA(cudaStreamBeginCapture(kv->cap_stream, cudaStreamCaptureModeThreadLocal));
        cudaError_t e = enqueue_step(kv, tokens, positions, logits, argmax, kv->cap_stream, true);
        cudaError_t e2 = cudaStreamEndCapture(kv->cap_stream, &graph);
        if (e != cudaSuccess) {
            if (graph) cudaGraphDestroy(graph);
            return cuda_fail(e, "capturing the decode step");
        }
        if (e2 != cudaSuccess) return cuda_fail(e2, "cudaStreamEndCapture");
        e = cudaGraphInstantiate(&exec, graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGraphInstantiate");
        kv->graphs.push_back({tokens, positions, logits, argmax, exec, now});
    }
    ER_CUDA(cudaGraphLaunch(exec, (cudaStream_t)stream));
    return ER_OK;
}

er_status er_launch_stage(er_kv *kv, int32_t stage, int32_t layer, const int32_t *tokens, const int32_t *positions,
                          float *logits, int32_t *argmax, void *stream) {
    er_status s = check_step(tokens, positions, kv);
    if (s != ER_OK) return s;
    if (stage < ER_STAGE_EMBED || stage > ER_STAGE_HEAD) return fail(ER_EINVAL, "bad stage");
    if (layer < 0 || layer >= kv->m->cfg.n_layers) return fail(ER_EINVAL, "layer out of range");
    ER_CUDA(enqueue_stage(kv, stage, layer, tokens, positions, logits, argmax, (cudaStream_t)stream, false));
    return ER_OK;
}

er_status er_prefill(er_kv *kv, int32_t seq, const int32_t *tokens, int32_t n, int32_t start, float *logits,
                     void *stream) {
    if (!kv) return fail(ER_EINVAL, "kv is NULL");
    if (kv->view) return fail(ER_EINVAL, "not a decode state");
    if (seq < 0 || seq >= kv->B) return fail(ER_EINVAL, "seq out of range");
    if (n < 0 || start < 0 || (long long)start + n > kv->cap) return fail(ER_EINVAL, "positions out of range");
    if (n == 0) return ER_OK;
    if (!tokens) return fail(ER_EINVAL, "tokens is NULL");
    if (!kv->pf) {
        er_kv *v = nullptr;
        er_status s = kv_create(kv->m, 16, kv->cap, kv->kv_type, kv, &v);
        if (s != ER_OK) return s;
        kv->pf = v;
    }
    er_kv *v = kv->pf;
    v->wide_variant = kv->wide_variant;
    const cudaStream_t st = (cudaStream_t)stream;
    const int L = kv->m->cfg.n_layers, V = kv->m->cfg.vocab;
    for (int c0 = 0; c0 < n; c0 += 16) {
        const int cols = n - c0 < 16 ? n - c0 : 16;
        const bool last = c0 + cols == n;
        v->B = cols;
        ER_CUDA(launch_prefill_setup(v->pf_pos, v->pf_seq, start + c0, seq, cols, st));
        cudaError_t e = enqueue_stage(v, ER_STAGE_EMBED, 0, tokens + c0, v->pf_pos, nullptr, nullptr, st, true);
        for (int l = 0; l < L && e == cudaSuccess; ++l)
            for (int sg = ER_STAGE_QKV; sg <= ER_STAGE_DOWN && e == cudaSuccess; ++sg)
                e = enqueue_stage(v, sg, l, tokens + c0, v->pf_pos, nullptr, nullptr, st, true);
        if (e == cudaSuccess && last && logits) {
            e = enqueue_stage(v, ER_STAGE_HEAD, 0, tokens + c0, v->pf_pos, v->pf_logits, nullptr, st, true);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(logits, v->pf_logits + (size_t)(cols - 1) * V, (size_t)V * sizeof(float),
                                    cudaMemcpyDeviceToDevice, st);
        }
        ER_CUDA(e);
    }
    return ER_OK;
}

er_status er_kv_set_schedule(er_kv *kv, int32_t schedule) {
    if (!kv) return fail(ER_EINVAL, "kv is NULL");
    int want;
    switch (schedule) {
        case ER_SCHEDULE_AUTO: want = kv->step_ok ? ER_SCHEDULE_PERSISTENT : ER_SCHEDULE_KERNELS; break;
        case ER_SCHEDULE_PERSISTENT:
            if (!kv->step_ok) return fail(ER_EUNSUPPORTED, "the persistent step cannot run this shape");
            want = ER_SCHEDULE_PERSISTENT;
            break;
        case ER_SCHEDULE_KERNELS: want = ER_SCHEDULE_KERNELS; break;
        default: return fail(ER_EINVAL, "bad schedule");
    }
    if (want != kv->schedule) {
        ER_CUDA(cudaDeviceSynchronize());
        for (auto &g : kv->graphs) cudaGraphExecDestroy(g.exec);
        kv->graphs.clear();
        kv->schedule = want;
    }
    return ER_OK;
}

int32_t er_kv_get_schedule(const er_kv *kv) { return kv ? kv->schedule : -1; }

er_status er_kv_set_wide_gemv(er_kv *kv, int32_t variant) {
    if (!kv) return fail(ER_EINVAL, "kv is NULL");
    if (variant != ER_WIDE_AUTO && variant != ER_WIDE_MMA_SYNC && variant != ER_WIDE_TCGEN05)
        return fail(ER_EINVAL, "bad batched GEMV variant");
    static_assert((int)ER_WIDE_MMA_SYNC == (int)er::WIDE_MMA_SYNC && (int)ER_WIDE_TCGEN05 == (int)er::WIDE_TCGEN05,
                  "variant codes");
    if (variant != kv->wide_variant) {
        ER_CUDA(cudaDeviceSynchronize());
        for (auto &g : kv->graphs) cudaGraphExecDestroy(g.exec);
        kv->graphs.clear();
        kv->wide_variant = variant;
    }
    return ER_OK;
}

int32_t er_kv_launches_per_step(const er_kv *kv) {
    if (!kv) return -1;
    if (kv->schedule == ER_SCHEDULE_PERSISTENT) return 1;
    const er_model *m = kv->m;
    const er_config &c = m->cfg;
    auto groups = [&](const er::Mat &w) {
        if (kv->wide_part) return 1;
        const int per = gemv_max_cols(w.qt, w.K);
        return per > 0 ? (kv->B + per - 1) / per : 0;
    };
    const er_layer_dev &L0 = m->layers[0];
    const int per_layer = groups(L0.qkv) + 1 + groups(L0.wo) + groups(L0.gateup) + groups(L0.down);
    return 1 + c.n_layers * per_layer + groups(m->head);
}

int32_t er_kv_cached_graphs(const er_kv *kv) { return kv ? (int32_t)kv->graphs.size() : -1; }

er_status er_kv_inject_wait_shortfall(er_kv *kv, int32_t extra) {
    if (!kv) return fail(ER_EINVAL, "kv is NULL");
    if (extra < 0 || extra > (1 << 20)) return fail(ER_EINVAL, "extra must be in 0..2^20");
    if ((unsigned)extra != kv->bar_extra) {
        ER_CUDA(cudaDeviceSynchronize());
        for (auto &g : kv->graphs) cudaGraphExecDestroy(g.exec);
        kv->graphs.clear();
        kv->bar_extra = (unsigned)extra;
    }
    return ER_OK;
}

er_status er_set_wait_limit_ns(uint64_t ns) {
    const unsigned long long v = ns ? (unsigned long long)ns : ER_WAIT_NS;
    cudaError_t (*set[])(unsigned long long) = {set_wait_limit_gemv, set_wait_limit_wide, set_wait_limit_tc,
                                                set_wait_limit_step_q8, set_wait_limit_step_q4, set_wait_limit_attn};
    for (auto f : set) ER_CUDA(f(v));
    return ER_OK;
}

er_status er_debug_fail_allocation(int64_t n) {
    if (n < -1) return fail(ER_EINVAL, "n must be >= -1");
    g_alloc_fail_at.store(n);
    return ER_OK;
}

int64_t er_debug_live_allocations(void) { return g_live_allocs.load(); }

er_status er_positions_increment(int32_t *positions, int32_t batch, void *stream) {
    if (!positions || batch < 1) return fail(ER_EINVAL, "bad positions/batch");
    ER_CUDA(launch_positions_increment(positions, batch, (cudaStream_t)stream));
    return ER_OK;
}

er_status er_get_device_error(er_kv *kv, int32_t *code, int32_t *non_finite) {
    if (!kv || !code || !non_finite) return fail(ER_EINVAL, "NULL argument");
    ER_CUDA(cudaDeviceSynchronize());
    int f = 0;
    ER_CUDA(cudaMemcpy(&f, kv->flags, sizeof(int), cudaMemcpyDeviceToHost));
    ER_CUDA(cudaMemset(kv->flags, 0, sizeof(int)));
    *code = f & (ER_FLAG_TOKEN | ER_FLAG_POS | ER_FLAG_WAIT);
    *non_finite = (f & ER_FLAG_NONFINITE) ? 1 : 0;
    return *code ? fail(ER_EDEVICE, "device flags 0x%x", f) : ER_OK;
}

// ---------------------------------------------------------------------------
// stand-alone matrices
// ---------------------------------------------------------------------------
er_status er_matrix_create(int32_t w_type, int32_t rows, int32_t cols, const void *blocks, void *stream,
                           er_matrix **out) {
    if (!out || !blocks) return fail(ER_EINVAL, "NULL argument");
    if (!valid_qt(w_type)) return fail(ER_EINVAL, "w_type must be ER_Q8_0 or ER_Q4_0");
    if (rows < 1 || cols < 32 || cols % 32) return fail(ER_EINVAL, "rows >= 1, cols a positive multiple of 32");
    if (gemv_max_cols(w_type, cols) < 1) return fail(ER_EUNSUPPORTED, "cols too large");
    er_matrix *x = new er_matrix();
    x->num_sms = device_sms(&x->device);
    if (x->num_sms <= 0) {
        delete x;
        return fail(ER_ECUDA, "no CUDA device");
    }
    std::vector<void *> owned;
    x->m = mat_shape(w_type, MAP_IDENT, rows, cols);
    cudaError_t e = gemv_prepare();
    if (e == cudaSuccess) e = dalloc(owned, &x->m.d, x->m.bytes);
    if (e == cudaSuccess) e = dalloc(owned, &x->part, gemv_part_floats(x->num_sms) * sizeof(float));
    if (e == cudaSuccess) e = dalloc(owned, &x->cnt, (size_t)x->m.R * sizeof(int));
    if (e == cudaSuccess) e = dalloc(owned, &x->flags, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(x->cnt, 0, (size_t)x->m.R * sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(x->flags, 0, sizeof(int));
    if (e == cudaSuccess) e = launch_repack(x->m, src1(blocks, rows), (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) {
        free_all(owned);
        delete x;
        return cuda_fail(e, "er_matrix_create");
    }
    *out = x;
    return ER_OK;
}

void er_matrix_destroy(er_matrix *x) {
    if (!x) return;
    cudaFree(x->m.d);
    cudaFree(x->part);
    cudaFree(x->cnt);
    cudaFree(x->flags);
    g_live_allocs -= 4;
    delete x;
}

er_status er_matrix_dequant(const er_matrix *x, float *out, void *stream) {
    if (!x || !out) return fail(ER_EINVAL, "NULL argument");
    ER_CUDA(launch_dequant(x->m, out, (cudaStream_t)stream));
    return ER_OK;
}

er_status er_matrix_gemv(const er_matrix *x, const float *xin, int32_t batch, float *y, void *stream) {
    if (!x || !xin || !y) return fail(ER_EINVAL, "NULL argument");
    if (batch < 1 || batch > 16) return fail(ER_EINVAL, "batch must be in 1..16");
    GemvArgs a = {};
    a.W = x->m.d;
    a.R = x->m.R;
    a.UPR = x->m.UPR;
    a.N = x->m.N;
    a.K = x->m.K;
    a.qt = x->m.qt;
    a.x = xin;
    a.y = y;
    a.part = x->part;
    a.cnt = x->cnt;
    a.flags = x->flags;
    int per = gemv_max_cols(a.qt, a.K);
    for (int b0 = 0; b0 < batch; b0 += per) {
        a.b0 = b0;
        a.B = batch - b0 < per ? batch - b0 : per;
        ER_CUDA(launch_gemv(EPI_STORE, a, x->num_sms, (cudaStream_t)stream, false));
    }
    return ER_OK;
}

}  // extern "C"
