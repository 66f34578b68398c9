// GGUF container reader (host code): parses a GGUF v2/v3 file mapped read-only
// into memory, derives the model shape from its llama.* metadata, and builds
// an er_model from its tensors ("EdgeRunner Core Architecture" section 2.2:
// the loader memory-maps the file and parses the configuration from metadata;
// "alpaca.swift" Capabilities: GGUF v2/v3, F16/Q8_0/Q4_0 tensors used in place).
//
// The file is untrusted input (as the "alpaca.swift" parser treats it): every
// count and length is bounded by the bytes actually present before anything
// is allocated or read, all size arithmetic is overflow-checked, offsets must
// respect the file's alignment, and a malformed file gives ER_EINVAL with a
// one-line reason (er_last_error) instead of a crash.
//
// Layout (little-endian): "GGUF", uint32 version, uint64 tensor count, uint64
// metadata count; metadata entries (string key, uint32 type, value); tensor
// entries (string name, uint32 n_dims, uint64 dims[n_dims] innermost first,
// uint32 type, uint64 offset from the data section); padding to the
// alignment (general.alignment, 32 by default); the data section.  A string
// is a uint64 length and that many bytes.
#include <errno.h>
#include <stdarg.h>
#include <fcntl.h>
#include <stdio.h>
#include <string.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <string>
#include <unordered_map>
#include <vector>

#include "internal.h"

namespace {

enum : uint32_t {
    GV_U8 = 0, GV_I8 = 1, GV_U16 = 2, GV_I16 = 3, GV_U32 = 4, GV_I32 = 5, GV_F32 = 6, GV_BOOL = 7,
    GV_STRING = 8, GV_ARRAY = 9, GV_U64 = 10, GV_I64 = 11, GV_F64 = 12
};

// bytes of one scalar value of a metadata type (0: not a fixed-size scalar)
uint64_t scalar_bytes(uint32_t t) {
    switch (t) {
        case GV_U8: case GV_I8: case GV_BOOL: return 1;
        case GV_U16: case GV_I16: return 2;
        case GV_U32: case GV_I32: case GV_F32: return 4;
        case GV_U64: case GV_I64: case GV_F64: return 8;
    }
    return 0;
}

// (elements per block, bytes per block) of a tensor type, from the type table
// of "EdgeRunner Core Architecture" section 1.3; {0, 0} for an unknown code
struct TypeSize { uint64_t elems, bytes; };
TypeSize type_size(uint32_t t) {
    switch (t) {
        case 0: return {1, 4};        // f32
        case 1: return {1, 2};        // f16
        case 2: return {32, 18};      // q4_0
        case 3: return {32, 20};      // q4_1
        case 6: return {32, 22};      // q5_0
        case 7: return {32, 24};      // q5_1
        case 8: return {32, 34};      // q8_0
        case 10: return {256, 84};    // q2_K
        case 11: return {256, 110};   // q3_K
        case 12: return {256, 144};   // q4_K
        case 13: return {256, 176};   // q5_K
        case 14: return {256, 210};   // q6_K
        case 16: return {1, 1};       // i8
        case 17: return {1, 2};       // i16
        case 18: return {1, 4};       // i32
        case 19: return {1, 8};       // i64
        case 20: return {1, 8};       // f64
        case 30: return {1, 2};       // bf16
    }
    return {0, 0};
}

bool mul_ok(uint64_t a, uint64_t b, uint64_t *out) {
    if (a && b > UINT64_MAX / a) return false;
    *out = a * b;
    return true;
}

// bounded cursor over the mapped bytes
struct Cursor {
    const uint8_t *p;
    uint64_t size, pos;
    bool need(uint64_t n) const { return n <= size - pos; }
    bool u32(uint32_t *v) {
        if (!need(4)) return false;
        memcpy(v, p + pos, 4);
        pos += 4;
        return true;
    }
    bool u64(uint64_t *v) {
        if (!need(8)) return false;
        memcpy(v, p + pos, 8);
        pos += 8;
        return true;
    }
    bool str(const char **s, uint64_t *len) {
        uint64_t n;
        if (!u64(&n) || !need(n)) return false;
        *s = reinterpret_cast<const char *>(p + pos);
        *len = n;
        pos += n;
        return true;
    }
    bool skip(uint64_t n) {
        if (!need(n)) return false;
        pos += n;
        return true;
    }
};

struct Meta {
    uint32_t type;
    uint64_t pos;  // file offset of the value
};

struct TensorInfo {
    std::string name;
    uint32_t type, n_dims;
    int64_t dims[4];
    uint64_t offset, bytes;
};

}  // namespace

struct er_gguf {
    int fd = -1;
    const uint8_t *map = nullptr;
    uint64_t size = 0;
    uint32_t version = 0;
    uint64_t alignment = 32, data_pos = 0;
    std::unordered_map<std::string, Meta> meta;
    std::vector<TensorInfo> tensors;
    std::unordered_map<std::string, int64_t> index;
};

namespace {

// a tensor name from the file, safe to print: printable ASCII only, at most 64 characters
std::string shown(const std::string &name) {
    std::string out;
    for (size_t i = 0; i < name.size() && i < 64; ++i) {
        const unsigned char ch = (unsigned char)name[i];
        out += (ch >= 0x20 && ch < 0x7F) ? (char)ch : '?';
    }
    if (name.size() > 64) out += "...";
    return out;
}

er_status bad(const char *fmt, ...) __attribute__((format(printf, 1, 2)));
er_status bad(const char *fmt, ...) {
    char buf[256];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    return er_fail_status(ER_EINVAL, buf);
}

// skip one metadata value of type t (arrays of arrays are refused)
bool skip_value(Cursor &c, uint32_t t, int depth) {
    if (uint64_t n = scalar_bytes(t)) return c.skip(n);
    if (t == GV_STRING) {
        const char *s;
        uint64_t len;
        return c.str(&s, &len);
    }
    if (t == GV_ARRAY && depth == 0) {
        uint32_t et;
        uint64_t count;
        if (!c.u32(&et) || !c.u64(&count)) return false;
        if (uint64_t n = scalar_bytes(et)) {
            uint64_t total;
            return mul_ok(n, count, &total) && c.skip(total);
        }
        if (et != GV_STRING) return false;
        if (count > (c.size - c.pos) / 8) return false;  // each string takes at least its 8-byte length
        for (uint64_t i = 0; i < count; ++i) {
            const char *s;
            uint64_t len;
            if (!c.str(&s, &len)) return false;
        }
        return true;
    }
    return false;
}

er_status parse(er_gguf *g) {
    Cursor c{g->map, g->size, 0};
    uint32_t magic;
    uint64_t nt, nm;
    if (!c.u32(&magic) || magic != 0x46554747u) return bad("not a GGUF file (magic)");
    if (!c.u32(&g->version) || (g->version != 2 && g->version != 3))
        return bad("GGUF version %u is not 2 or 3", g->version);
    if (!c.u64(&nt) || !c.u64(&nm)) return bad("truncated header");
    // every metadata entry takes at least 12 bytes, every tensor entry at least 24
    if (nm > (c.size - c.pos) / 12) return bad("metadata count %llu exceeds the file", (unsigned long long)nm);
    for (uint64_t i = 0; i < nm; ++i) {
        const char *k;
        uint64_t klen;
        uint32_t t;
        if (!c.str(&k, &klen) || !c.u32(&t)) return bad("truncated metadata entry %llu", (unsigned long long)i);
        Meta m{t, c.pos};
        if (!skip_value(c, t, 0)) return bad("bad or truncated metadata value %llu", (unsigned long long)i);
        if (!g->meta.emplace(std::string(k, klen), m).second) return bad("duplicate metadata key");
    }
    auto al = g->meta.find("general.alignment");
    if (al != g->meta.end()) {
        if (al->second.type != GV_U32) return bad("general.alignment is not a uint32");
        uint32_t a;
        memcpy(&a, g->map + al->second.pos, 4);
        if (a == 0 || (a & (a - 1)) || a > (1u << 16)) return bad("alignment %u is not a power of two up to 65536", a);
        g->alignment = a;
    }
    if (nt > (c.size - c.pos) / 24) return bad("tensor count %llu exceeds the file", (unsigned long long)nt);
    g->tensors.resize(nt);
    for (uint64_t i = 0; i < nt; ++i) {
        TensorInfo &ti = g->tensors[i];
        const char *n;
        uint64_t nlen;
        if (!c.str(&n, &nlen) || !c.u32(&ti.n_dims)) return bad("truncated tensor entry %llu", (unsigned long long)i);
        if (ti.n_dims < 1 || ti.n_dims > 4) return bad("tensor %llu has %u dimensions", (unsigned long long)i, ti.n_dims);
        ti.name.assign(n, nlen);
        uint64_t elems = 1;
        for (uint32_t d = 0; d < 4; ++d) ti.dims[d] = 1;
        for (uint32_t d = 0; d < ti.n_dims; ++d) {
            uint64_t v;
            if (!c.u64(&v)) return bad("truncated dimensions of %s", shown(ti.name).c_str());
            if (v == 0 || v > (1ull << 40) || !mul_ok(elems, v, &elems) || elems > (1ull << 50))
                return bad("dimensions of %s out of range", shown(ti.name).c_str());
            ti.dims[d] = (int64_t)v;
        }
        if (!c.u32(&ti.type) || !c.u64(&ti.offset)) return bad("truncated tensor entry %s", shown(ti.name).c_str());
        const TypeSize ts = type_size(ti.type);
        if (!ts.elems) return bad("tensor %s has unknown type %u", shown(ti.name).c_str(), ti.type);
        if ((uint64_t)ti.dims[0] % ts.elems) return bad("row of %s is not whole blocks", shown(ti.name).c_str());
        if (!mul_ok(elems / ts.elems, ts.bytes, &ti.bytes)) return bad("size of %s overflows", shown(ti.name).c_str());
        if (ti.offset % g->alignment) return bad("offset of %s is not aligned", shown(ti.name).c_str());
        if (!g->index.emplace(ti.name, (int64_t)i).second) return bad("duplicate tensor %s", shown(ti.name).c_str());
    }
    // data section: the next multiple of the alignment
    const uint64_t pad = (g->alignment - c.pos % g->alignment) % g->alignment;
    if (nt > 0 && !c.need(pad)) return bad("truncated before the data section");
    g->data_pos = c.pos + pad;
    for (const TensorInfo &ti : g->tensors) {
        const uint64_t avail = g->size >= g->data_pos ? g->size - g->data_pos : 0;
        if (ti.offset > avail || ti.bytes > avail - ti.offset) return bad("data of %s lies past the end", shown(ti.name).c_str());
    }
    return ER_OK;
}

// a numeric metadata value as double / uint64; false if absent or not numeric
bool meta_num(const er_gguf *g, const char *key, double *out) {
    auto it = g->meta.find(key);
    if (it == g->meta.end()) return false;
    const uint8_t *p = g->map + it->second.pos;
    switch (it->second.type) {
        case GV_U8: *out = p[0]; return true;
        case GV_I8: *out = (int8_t)p[0]; return true;
        case GV_U16: { uint16_t v; memcpy(&v, p, 2); *out = v; return true; }
        case GV_I16: { int16_t v; memcpy(&v, p, 2); *out = v; return true; }
        case GV_U32: { uint32_t v; memcpy(&v, p, 4); *out = v; return true; }
        case GV_I32: { int32_t v; memcpy(&v, p, 4); *out = v; return true; }
        case GV_U64: { uint64_t v; memcpy(&v, p, 8); *out = (double)v; return true; }
        case GV_I64: { int64_t v; memcpy(&v, p, 8); *out = (double)v; return true; }
        case GV_F32: { float v; memcpy(&v, p, 4); *out = v; return true; }
        case GV_F64: { double v; memcpy(&v, p, 8); *out = v; return true; }
    }
    return false;
}

bool meta_int(const er_gguf *g, const char *key, int32_t *out) {
    double v;
    if (!meta_num(g, key, &v) || !(v >= 1 && v <= (double)(1 << 30)) || v != (double)(int64_t)v) return false;
    *out = (int32_t)v;
    return true;
}

bool meta_str_is(const er_gguf *g, const char *key, const char *want) {
    auto it = g->meta.find(key);
    if (it == g->meta.end() || it->second.type != GV_STRING) return false;
    uint64_t len;
    memcpy(&len, g->map + it->second.pos, 8);
    return len == strlen(want) && memcmp(g->map + it->second.pos + 8, want, len) == 0;
}

const TensorInfo *find(const er_gguf *g, const std::string &name) {
    auto it = g->index.find(name);
    return it == g->index.end() ? nullptr : &g->tensors[it->second];
}

// the tensor must exist with this type and [rows x cols] (dims {cols, rows}), or [n] for rows == 0
er_status expect(const er_gguf *g, const std::string &name, uint32_t type, int64_t cols, int64_t rows,
                 const TensorInfo **out) {
    const TensorInfo *t = find(g, name);
    if (!t) return bad("tensor %s is missing", shown(name).c_str());
    if (t->type != type) return bad("tensor %s has type %u, expected %u", shown(name).c_str(), t->type, type);
    const bool ok = rows == 0 ? (t->n_dims == 1 && t->dims[0] == cols)
                              : (t->n_dims == 2 && t->dims[0] == cols && t->dims[1] == rows);
    if (!ok) return bad("tensor %s has the wrong shape", shown(name).c_str());
    if (out) *out = t;
    return ER_OK;
}

const char *LAYER_LEAF[9] = {"attn_norm", "attn_q", "attn_k", "attn_v", "attn_output",
                             "ffn_norm", "ffn_gate", "ffn_up", "ffn_down"};

}  // namespace

extern "C" {

er_status er_gguf_open(const char *path, er_gguf **out) {
    if (!path || !out) return er_fail_status(ER_EINVAL, "NULL argument");
    er_gguf *g = new er_gguf();
    g->fd = open(path, O_RDONLY);
    if (g->fd < 0) {
        delete g;
        return bad("cannot open %s: %s", path, strerror(errno));
    }
    struct stat st;
    if (fstat(g->fd, &st) != 0 || st.st_size < 0) {
        close(g->fd);
        delete g;
        return bad("cannot stat %s", path);
    }
    g->size = (uint64_t)st.st_size;
    if (g->size > 0) {
        void *m = mmap(nullptr, g->size, PROT_READ, MAP_PRIVATE, g->fd, 0);
        if (m == MAP_FAILED) {
            close(g->fd);
            delete g;
            return bad("cannot map %s", path);
        }
        g->map = static_cast<const uint8_t *>(m);
    }
    er_status s = parse(g);
    if (s != ER_OK) {
        er_gguf_close(g);
        return s;
    }
    *out = g;
    return ER_OK;
}

void er_gguf_close(er_gguf *g) {
    if (!g) return;
    if (g->map) munmap(const_cast<uint8_t *>(g->map), g->size);
    if (g->fd >= 0) close(g->fd);
    delete g;
}

int64_t er_gguf_tensor_count(const er_gguf *g) { return g ? (int64_t)g->tensors.size() : -1; }

er_status er_gguf_tensor_info(const er_gguf *g, int64_t i, const char **name, int32_t *type, int32_t *n_dims,
                              int64_t *dims, const void **data, uint64_t *bytes) {
    if (!g || i < 0 || i >= (int64_t)g->tensors.size()) return er_fail_status(ER_EINVAL, "bad handle or index");
    const TensorInfo &t = g->tensors[i];
    if (name) *name = t.name.c_str();
    if (type) *type = (int32_t)t.type;
    if (n_dims) *n_dims = (int32_t)t.n_dims;
    if (dims)
        for (int d = 0; d < 4; ++d) dims[d] = t.dims[d];
    if (data) *data = g->map + g->data_pos + t.offset;
    if (bytes) *bytes = t.bytes;
    return ER_OK;
}

er_status er_gguf_find(const er_gguf *g, const char *name, int64_t *index) {
    if (!g || !name || !index) return er_fail_status(ER_EINVAL, "NULL argument");
    auto it = g->index.find(name);
    if (it == g->index.end()) return bad("no tensor %s", shown(name).c_str());
    *index = it->second;
    return ER_OK;
}

er_status er_gguf_config(const er_gguf *g, int32_t max_batch, er_config *cfg) {
    if (!g || !cfg) return er_fail_status(ER_EINVAL, "NULL argument");
    if (!meta_str_is(g, "general.architecture", "llama")) return bad("general.architecture is not \"llama\"");
    er_config c = {};
    if (!meta_int(g, "llama.embedding_length", &c.dim) || !meta_int(g, "llama.block_count", &c.n_layers) ||
        !meta_int(g, "llama.feed_forward_length", &c.ffn_dim) ||
        !meta_int(g, "llama.attention.head_count", &c.n_heads))
        return bad("a required llama.* shape key is missing or out of range");
    if (!meta_int(g, "llama.attention.head_count_kv", &c.n_kv_heads)) c.n_kv_heads = c.n_heads;
    // head width: an explicit key length (as Qwen 3 files carry), else dim / heads (section 1.1)
    if (!meta_int(g, "llama.attention.key_length", &c.head_dim)) {
        if (c.dim % c.n_heads) return bad("embedding_length is not a multiple of head_count");
        c.head_dim = c.dim / c.n_heads;
    }
    double v;
    c.rope_base = meta_num(g, "llama.rope.freq_base", &v) ? v : 10000.0;
    c.rms_eps = meta_num(g, "llama.attention.layer_norm_rms_epsilon", &v) ? v : 1e-5;
    const TensorInfo *emb = find(g, "token_embd.weight");
    if (!emb || emb->n_dims != 2 || emb->dims[0] != c.dim || emb->dims[1] > (1 << 30))
        return bad("token_embd.weight is missing or has the wrong shape");
    c.vocab = (int32_t)emb->dims[1];
    const TensorInfo *q = find(g, "blk.0.attn_q.weight");
    if (!q) return bad("blk.0.attn_q.weight is missing");
    c.w_type = (int32_t)q->type;
    c.tied = find(g, "output.weight") ? 0 : 1;
    c.max_batch = max_batch;
    // every tensor the step reads, with the type and shape this configuration implies
    const int64_t D = c.dim, qd = (int64_t)c.n_heads * c.head_dim, kvd = (int64_t)c.n_kv_heads * c.head_dim,
                  F = c.ffn_dim, V = c.vocab;
    const uint32_t wt = (uint32_t)c.w_type;
    for (int l = 0; l < c.n_layers; ++l) {
        const std::string p = "blk." + std::to_string(l) + ".";
        er_status s = ER_OK;
        if (s == ER_OK) s = expect(g, p + "attn_norm.weight", 0, D, 0, nullptr);
        if (s == ER_OK) s = expect(g, p + "attn_q.weight", wt, D, qd, nullptr);
        if (s == ER_OK) s = expect(g, p + "attn_k.weight", wt, D, kvd, nullptr);
        if (s == ER_OK) s = expect(g, p + "attn_v.weight", wt, D, kvd, nullptr);
        if (s == ER_OK) s = expect(g, p + "attn_output.weight", wt, qd, D, nullptr);
        if (s == ER_OK) s = expect(g, p + "ffn_norm.weight", 0, D, 0, nullptr);
        if (s == ER_OK) s = expect(g, p + "ffn_gate.weight", wt, D, F, nullptr);
        if (s == ER_OK) s = expect(g, p + "ffn_up.weight", wt, D, F, nullptr);
        if (s == ER_OK) s = expect(g, p + "ffn_down.weight", wt, F, D, nullptr);
        if (s != ER_OK) return s;
    }
    if (er_status s = expect(g, "output_norm.weight", 0, D, 0, nullptr); s != ER_OK) return s;
    const uint32_t embd_type = c.tied ? wt : (uint32_t)ER_F16;
    if (er_status s = expect(g, "token_embd.weight", embd_type, D, V, nullptr); s != ER_OK) return s;
    if (!c.tied)
        if (er_status s = expect(g, "output.weight", wt, D, V, nullptr); s != ER_OK) return s;
    *cfg = c;
    return ER_OK;
}

er_status er_model_create_from_gguf(const er_gguf *g, int32_t max_batch, void *stream, er_model **out) {
    if (!g || !out) return er_fail_status(ER_EINVAL, "NULL argument");
    er_config c;
    er_status s = er_gguf_config(g, max_batch, &c);
    if (s != ER_OK) return s;
    // stage the data section on the device once, then hand the model its tensors in place
    const uint64_t data_bytes = g->size - g->data_pos;
    uint8_t *stage = nullptr;
    cudaError_t e = er::device_alloc((void **)&stage, data_bytes);
    if (e != cudaSuccess) return er_fail_cuda(e, "staging buffer for the GGUF data section");
    cudaStream_t st = (cudaStream_t)stream;
    e = cudaMemcpyAsync(stage, g->map + g->data_pos, data_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) {
        er::device_free(stage);
        return er_fail_cuda(e, "staging the GGUF data section");
    }
    auto dev = [&](const std::string &name) -> const void * { return stage + find(g, name)->offset; };
    std::vector<er_layer_weights> layers(c.n_layers);
    for (int l = 0; l < c.n_layers; ++l) {
        const std::string p = "blk." + std::to_string(l) + ".";
        const void **f = reinterpret_cast<const void **>(&layers[l]);
        for (int k = 0; k < 9; ++k) f[k] = dev(p + LAYER_LEAF[k] + ".weight");
    }
    er_weights w;
    w.tok_embd = dev("token_embd.weight");
    w.output_norm = dev("output_norm.weight");
    w.output = c.tied ? nullptr : dev("output.weight");
    w.layers = layers.data();
    s = er_model_create(&c, &w, stream, out);  // synchronises the stream before returning
    er::device_free(stage);
    return s;
}

}  // extern "C"
