// GGUF reader for the Llama model files the library runs ("量化 llama 的一次
// 前向", from_gguf：键名写死了 llama.; "生成一个 token", 读 GGUF / 建模型：按
// 名字取张量): the header (magic, version, metadata key/values, tensor
// directory) is parsed through a buffered reader without touching the weights;
// the hyperparameters come from the llama.* keys, the rotary convention from
// general.architecture, and the tensors by their GGUF names, with the head
// falling back to token_embd.weight when output.weight is absent. The weights
// are then mapped read-only and handed to llama_q8_load as host arrays.
//
// File layout (the published GGUF format, version 2 and 3): "GGUF", u32
// version, u64 tensor count, u64 key/value count; each key a string (u64
// length + bytes), a u32 value type and the value (arrays: u32 element type,
// u64 count, elements); each tensor a name, u32 rank, u64 extents (innermost
// first), u32 element type, u64 offset into the data region; the data region
// starts at the next multiple of general.alignment (32 when absent).
#include <sys/mman.h>
#include <sys/stat.h>
#include <fcntl.h>
#include <unistd.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <string>
#include <vector>

#include "llama_q8.h"

namespace {

enum GgufType : uint32_t {
    kU8 = 0, kI8 = 1, kU16 = 2, kI16 = 3, kU32 = 4, kI32 = 5, kF32 = 6, kBool = 7,
    kString = 8, kArray = 9, kU64 = 10, kI64 = 11, kF64 = 12
};
constexpr uint32_t kTensorF32 = 0;
constexpr uint32_t kTensorQ8_0 = 8;

struct Value {
    uint32_t type = 0;
    double num = 0.0;   // numeric scalars
    std::string str;    // strings
};

struct TensorInfo {
    uint32_t type = 0;
    std::vector<uint64_t> dims;  // innermost first
    uint64_t offset = 0;         // into the data region
};

struct Gguf {
    std::map<std::string, Value> kv;
    std::map<std::string, TensorInfo> tensors;
    uint64_t data_offset = 0;
    uint64_t file_bytes = 0;
};

class Reader {
   public:
    explicit Reader(FILE* f) : f_(f) {}
    bool bytes(void* dst, size_t n) { return n == 0 || std::fread(dst, 1, n, f_) == n; }
    template <typename T>
    bool pod(T* v) { return bytes(v, sizeof(T)); }
    bool str(std::string* s) {
        uint64_t n = 0;
        if (!pod(&n) || n > (1ull << 24)) return false;  // keys and string values: at most 16 MiB
        s->resize(n);
        return bytes(&(*s)[0], n);
    }
    bool skip(uint64_t n) { return std::fseek(f_, (long)n, SEEK_CUR) == 0; }
    uint64_t pos() const { return (uint64_t)std::ftell(f_); }

   private:
    FILE* f_;
};

size_t scalar_bytes(uint32_t t) {
    switch (t) {
        case kU8: case kI8: case kBool: return 1;
        case kU16: case kI16: return 2;
        case kU32: case kI32: case kF32: return 4;
        case kU64: case kI64: case kF64: return 8;
    }
    return 0;
}

bool read_scalar(Reader& r, uint32_t t, double* out) {
    switch (t) {
        case kU8: { uint8_t v; if (!r.pod(&v)) return false; *out = v; return true; }
        case kI8: { int8_t v; if (!r.pod(&v)) return false; *out = v; return true; }
        case kBool: { uint8_t v; if (!r.pod(&v)) return false; *out = v; return true; }
        case kU16: { uint16_t v; if (!r.pod(&v)) return false; *out = v; return true; }
        case kI16: { int16_t v; if (!r.pod(&v)) return false; *out = v; return true; }
        case kU32: { uint32_t v; if (!r.pod(&v)) return false; *out = v; return true; }
        case kI32: { int32_t v; if (!r.pod(&v)) return false; *out = v; return true; }
        case kF32: { float v; if (!r.pod(&v)) return false; *out = v; return true; }
        case kU64: { uint64_t v; if (!r.pod(&v)) return false; *out = (double)v; return true; }
        case kI64: { int64_t v; if (!r.pod(&v)) return false; *out = (double)v; return true; }
        case kF64: { double v; if (!r.pod(&v)) return false; *out = v; return true; }
    }
    return false;
}

// Parse the header. Arrays (the tokenizer's vocabulary, merges, types) are
// skipped: the forward pass needs none of them.
llama_q8_status parse(const char* path, Gguf* g) {
    FILE* f = std::fopen(path, "rb");
    if (!f) return LQ8_ERR_FORMAT;
    std::vector<char> buf(1 << 20);
    std::setvbuf(f, buf.data(), _IOFBF, buf.size());  // the header is many small reads
    Reader r(f);
    llama_q8_status st = LQ8_ERR_FORMAT;
    do {
        char magic[4];
        uint32_t version = 0;
        uint64_t n_tensors = 0, n_kv = 0;
        if (!r.bytes(magic, 4) || std::memcmp(magic, "GGUF", 4) != 0) break;
        if (!r.pod(&version) || (version != 2 && version != 3)) break;
        if (!r.pod(&n_tensors) || !r.pod(&n_kv) || n_tensors > (1u << 24) || n_kv > (1u << 24)) break;
        bool ok = true;
        for (uint64_t i = 0; i < n_kv && ok; ++i) {
            std::string key;
            Value v;
            ok = r.str(&key) && r.pod(&v.type);
            if (!ok) break;
            if (v.type == kString) {
                ok = r.str(&v.str);
            } else if (v.type == kArray) {
                uint32_t et = 0;
                uint64_t n = 0;
                ok = r.pod(&et) && r.pod(&n);
                if (!ok) break;
                if (et == kString) {
                    for (uint64_t j = 0; j < n && ok; ++j) {
                        uint64_t len = 0;
                        ok = r.pod(&len) && len <= (1ull << 30) && r.skip(len);
                    }
                } else {
                    const size_t b = scalar_bytes(et);
                    ok = b > 0 && n <= (1ull << 40) / b && r.skip(n * b);
                }
            } else {
                ok = read_scalar(r, v.type, &v.num);
            }
            if (ok) g->kv[key] = v;
        }
        if (!ok) break;
        for (uint64_t i = 0; i < n_tensors && ok; ++i) {
            std::string name;
            TensorInfo t;
            uint32_t rank = 0;
            ok = r.str(&name) && r.pod(&rank) && rank >= 1 && rank <= 4;
            for (uint32_t d = 0; d < rank && ok; ++d) {
                uint64_t e = 0;
                ok = r.pod(&e);
                t.dims.push_back(e);
            }
            ok = ok && r.pod(&t.type) && r.pod(&t.offset);
            if (ok) g->tensors[name] = t;
        }
        if (!ok) break;
        // general.alignment, when present, must be an integer power of two no
        // larger than 64 KiB: anything else would make the rounding below
        // undefined or let it wrap into the header.
        uint64_t align = 32;
        auto a = g->kv.find("general.alignment");
        if (a != g->kv.end()) {
            const double v = a->second.num;
            if (a->second.type == kString || a->second.type == kArray || !(v >= 1.0 && v <= 65536.0) ||
                v != (double)(uint64_t)v)
                break;
            align = (uint64_t)v;
            if (align & (align - 1)) break;
        }
        const uint64_t end = r.pos();
        g->data_offset = (end + align - 1) / align * align;
        if (std::fseek(f, 0, SEEK_END) != 0) break;
        g->file_bytes = (uint64_t)std::ftell(f);
        st = LQ8_OK;
    } while (false);
    std::fclose(f);
    return st;
}

// An integer-valued key. Values that are not finite, not integral or beyond
// +-2^53 (where a double stops holding every integer) are rejected before the
// conversion, which would otherwise be undefined.
bool get_int(const Gguf& g, const std::string& key, int64_t* out) {
    auto it = g.kv.find(key);
    if (it == g.kv.end() || it->second.type == kString || it->second.type == kArray) return false;
    const double v = it->second.num;
    if (!(v >= -9007199254740992.0 && v <= 9007199254740992.0)) return false;
    if (v != std::trunc(v)) return false;
    *out = (int64_t)v;
    return true;
}

bool get_float(const Gguf& g, const std::string& key, float* out) {
    auto it = g.kv.find(key);
    if (it == g.kv.end() || it->second.type == kString || it->second.type == kArray) return false;
    *out = (float)it->second.num;
    return true;
}

uint64_t tensor_bytes(const TensorInfo& t) {
    uint64_t n = 1;
    for (uint64_t e : t.dims) n *= e;
    return t.type == kTensorQ8_0 ? n / 32 * 34 : n * 4;
}

// A tensor the model needs: present, of the expected type and extents, inside the file.
llama_q8_status check_tensor(const Gguf& g, const std::string& name, uint32_t type, uint64_t inner,
                             uint64_t outer) {
    auto it = g.tensors.find(name);
    if (it == g.tensors.end()) return LQ8_ERR_FORMAT;
    const TensorInfo& t = it->second;
    if (t.type != type) return LQ8_ERR_UNSUPPORTED;  // matrices run as Q8_0 only, norms as F32
    const uint64_t o = t.dims.size() > 1 ? t.dims[1] : 1;
    for (size_t d = 2; d < t.dims.size(); ++d)
        if (t.dims[d] != 1) return LQ8_ERR_FORMAT;
    if (t.dims[0] != inner || o != outer) return LQ8_ERR_FORMAT;
    // inside the file, without wrapping: extents are bounded by the checked hyperparameters
    const uint64_t bytes = tensor_bytes(t);
    if (g.data_offset > g.file_bytes || t.offset > g.file_bytes - g.data_offset ||
        bytes > g.file_bytes - g.data_offset - t.offset)
        return LQ8_ERR_FORMAT;
    return LQ8_OK;
}

std::string blk(int i, const char* n) { return "blk." + std::to_string(i) + "." + n + ".weight"; }

// Hyperparameters from the llama.* keys and a check of every tensor.
llama_q8_status config_from(const Gguf& g, llama_q8_config* c) {
    int64_t n_layer, n_embd, n_head, n_head_kv = 0, n_ff;
    if (!get_int(g, "llama.block_count", &n_layer) || !get_int(g, "llama.embedding_length", &n_embd) ||
        !get_int(g, "llama.attention.head_count", &n_head) || !get_int(g, "llama.feed_forward_length", &n_ff))
        return LQ8_ERR_FORMAT;
    if (!get_int(g, "llama.attention.head_count_kv", &n_head_kv)) {
        if (g.kv.count("llama.attention.head_count_kv")) return LQ8_ERR_FORMAT;  // present but not an integer
        n_head_kv = n_head;
    }
    if (n_layer <= 0 || n_embd <= 0 || n_head <= 0 || n_head_kv <= 0 || n_ff <= 0 || n_embd % n_head)
        return LQ8_ERR_FORMAT;
    // bounds that keep every size product far from overflow (llama_q8_load checks the shapes it runs)
    if (n_layer > 4096 || n_embd > (1 << 20) || n_ff > (1 << 22) || n_head > 4096 || n_head_kv > n_head)
        return LQ8_ERR_FORMAT;
    std::memset(c, 0, sizeof(*c));
    c->n_layer = (int32_t)n_layer;
    c->n_embd = (int32_t)n_embd;
    c->n_head = (int32_t)n_head;
    c->n_head_kv = (int32_t)n_head_kv;
    c->head_dim = (int32_t)(n_embd / n_head);
    c->n_ff = (int32_t)n_ff;
    c->max_seq = 4096;  // the rotary table size on the pages, a constant of the loader
    c->rms_eps = 1e-5f;
    get_float(g, "llama.attention.layer_norm_rms_epsilon", &c->rms_eps);
    c->rope_theta = 10000.0f;
    get_float(g, "llama.rope.freq_base", &c->rope_theta);
    auto arch = g.kv.find("general.architecture");
    c->rope_style = (arch != g.kv.end() && arch->second.type == kString)
                        ? llama_q8_rope_style_for_arch(arch->second.str.c_str())
                        : 0;
    auto e = g.tensors.find("token_embd.weight");
    if (e == g.tensors.end() || e->second.dims.size() < 2 || e->second.dims[1] == 0 ||
        e->second.dims[1] > (1u << 24))
        return LQ8_ERR_FORMAT;
    c->n_vocab = (int32_t)e->second.dims[1];
    c->tied_output = g.tensors.count("output.weight") ? 0 : 1;
    const uint64_t h = (uint64_t)n_embd, V = (uint64_t)c->n_vocab, F = (uint64_t)n_ff;
    const uint64_t qd = (uint64_t)n_head * c->head_dim, kvd = (uint64_t)n_head_kv * c->head_dim;
    llama_q8_status st = check_tensor(g, "token_embd.weight", kTensorQ8_0, h, V);
    if (st == LQ8_OK) st = check_tensor(g, "output_norm.weight", kTensorF32, h, 1);
    if (st == LQ8_OK && !c->tied_output) st = check_tensor(g, "output.weight", kTensorQ8_0, h, V);
    for (int i = 0; i < c->n_layer && st == LQ8_OK; ++i) {
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "attn_norm"), kTensorF32, h, 1);
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "ffn_norm"), kTensorF32, h, 1);
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "attn_q"), kTensorQ8_0, h, qd);
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "attn_k"), kTensorQ8_0, h, kvd);
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "attn_v"), kTensorQ8_0, h, kvd);
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "attn_output"), kTensorQ8_0, qd, h);
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "ffn_gate"), kTensorQ8_0, h, F);
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "ffn_up"), kTensorQ8_0, h, F);
        if (st == LQ8_OK) st = check_tensor(g, blk(i, "ffn_down"), kTensorQ8_0, F, h);
    }
    return st;
}

}  // namespace

extern "C" {

llama_q8_status llama_q8_gguf_config(const char* path, llama_q8_config* cfg, int64_t* n_tensors,
                                     int64_t* data_offset) {
    if (!path || !cfg) return LQ8_ERR_ARG;
    Gguf g;
    llama_q8_status st = parse(path, &g);
    if (st != LQ8_OK) return st;
    if (n_tensors) *n_tensors = (int64_t)g.tensors.size();
    if (data_offset) *data_offset = (int64_t)g.data_offset;
    return config_from(g, cfg);
}

llama_q8_status llama_q8_load_gguf(const char* path, int32_t device, int32_t decode_kernel, llama_q8_ctx** out) {
    if (!path || !out) return LQ8_ERR_ARG;
    *out = nullptr;
    Gguf g;
    llama_q8_status st = parse(path, &g);
    llama_q8_config cfg;
    if (st == LQ8_OK) st = config_from(g, &cfg);
    if (st != LQ8_OK) return st;
    cfg.decode_kernel = decode_kernel;
    const int fd = open(path, O_RDONLY);
    if (fd < 0) return LQ8_ERR_FORMAT;
    void* map = mmap(nullptr, (size_t)g.file_bytes, PROT_READ, MAP_PRIVATE, fd, 0);
    close(fd);
    if (map == MAP_FAILED) return LQ8_ERR_FORMAT;
    const uint8_t* data = static_cast<const uint8_t*>(map) + g.data_offset;
    auto ptr = [&](const std::string& name) -> const void* { return data + g.tensors.at(name).offset; };
    std::vector<llama_q8_layer_weights> layers((size_t)cfg.n_layer);
    for (int i = 0; i < cfg.n_layer; ++i) {
        llama_q8_layer_weights& L = layers[i];
        L.attn_norm = static_cast<const float*>(ptr(blk(i, "attn_norm")));
        L.ffn_norm = static_cast<const float*>(ptr(blk(i, "ffn_norm")));
        L.attn_q = ptr(blk(i, "attn_q"));
        L.attn_k = ptr(blk(i, "attn_k"));
        L.attn_v = ptr(blk(i, "attn_v"));
        L.attn_output = ptr(blk(i, "attn_output"));
        L.ffn_gate = ptr(blk(i, "ffn_gate"));
        L.ffn_up = ptr(blk(i, "ffn_up"));
        L.ffn_down = ptr(blk(i, "ffn_down"));
    }
    llama_q8_weights w;
    std::memset(&w, 0, sizeof(w));
    w.token_embd = ptr("token_embd.weight");
    w.output_norm = static_cast<const float*>(ptr("output_norm.weight"));
    w.output = cfg.tied_output ? nullptr : ptr("output.weight");
    w.layers = layers.data();
    w.on_device = 0;
    st = llama_q8_load(&cfg, &w, device, out);  // copies every tensor to the device
    munmap(map, (size_t)g.file_bytes);
    return st;
}

}  // extern "C"
