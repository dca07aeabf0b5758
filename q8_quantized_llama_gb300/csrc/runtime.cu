// Host runtime behind include/llama_q8.h: context, weight repacking, KV cache,
// the prefill launch sequence and the CUDA-graph decode step.
//
// The forward follows ModelWeights::forward on "量化 llama 的一次前向"
// (forward：mask 什么时候建): embedding, per layer RMSNorm -> attention with
// the KV cache -> O projection + residual -> RMSNorm -> SiLU-gated MLP +
// residual, final RMSNorm of the last row, output head. Differences in form
// (not in result): Q/K/V are one concatenated projection, gate/up one
// row-interleaved projection, RoPE and the KV append run in the projection
// epilogue, the cache is preallocated and written in place, and the decode
// step is one CUDA graph whose position and input token live in device memory.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "kernels.cuh"
#include "llama_q8.h"

using namespace lq8;

namespace lq8 {
cudaError_t init_gemv_attributes();
cudaError_t init_attention_attributes();

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_init_mu;
bool g_init_done[kMaxDevices] = {};
}  // namespace

// Kernel attributes (shared-memory limits, cluster permissions) of every
// kernel, set once per device under one lock.
cudaError_t ensure_kernel_attributes() {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_init_mu);
    if (g_init_done[dev]) return cudaSuccess;
    err = init_gemv_attributes();
    if (err == cudaSuccess) err = init_attention_attributes();
    if (err == cudaSuccess) err = init_gemm_tc_attributes();
    if (err == cudaSuccess) err = init_gemv_fmt_attributes();
    if (err == cudaSuccess) g_init_done[dev] = true;
    return err;
}
}  // namespace lq8

namespace {

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// Layout of one decode step for llama_q8_profile_decode: the family and the
// algorithmic bytes of each launch, in launch order (K/V bytes are per cached
// position and scaled by the step's cache length when the timeline is read).
struct StepLayout {
    struct Rec {
        int family;
        double bytes;       // algorithmic bytes of the launch, fixed part
        double kv_per_pos;  // plus this many bytes per cached position (K/V reads)
    };
    std::vector<Rec> recs;
};

enum Family {
    F_EMBED = 0, F_QKV, F_ATTN, F_OPROJ, F_GATEUP, F_DOWN, F_HEAD, F_ATTN_O, F_FRONT, F_MLP, F_COUNT
};
const char* kFamilyNames[F_COUNT] = {"embed", "gemv_qkv_rope_kv", "attn_decode", "gemv_o_residual",
                                     "gemv_gate_up_silu", "gemv_down_residual", "gemv_head_argmax",
                                     "attn_oproj_residual", "layer_front_qkv_attn_o", "decode_mlp"};

struct LayerDev {
    const float* attn_norm;
    const float* ffn_norm;
    PackedQ8 qkv, o, gu, down;
};

}  // namespace

struct llama_q8_ctx {
    llama_q8_config cfg{};
    int device = 0;
    cudaStream_t stream = nullptr;
    bool failed = false;
    int q_rows = 0, kv_rows = 0;

    uint8_t* d_weights = nullptr;
    float* d_norms = nullptr;
    float* d_rope_cos = nullptr;
    float* d_rope_sin = nullptr;
    float* d_kcache = nullptr;
    float* d_vcache = nullptr;
    float* d_x = nullptr;
    float* d_y = nullptr;
    float* d_q = nullptr;
    float* d_o = nullptr;
    float* d_a = nullptr;
    float* d_part = nullptr;  // decode: per-KV-head partials of W_o o
    float* d_xsum = nullptr;  // decode: x + W_o o, the residual of the down projection
    float* d_xr = nullptr;    // decode with the MLP kernel: x + W_o o of the last layer
    float* d_mlp = nullptr;   // decode with the MLP kernel: per-cluster partials of W_down a
    float* d_logits = nullptr;
    int32_t* d_ids = nullptr;
    int32_t* d_out_ids = nullptr;
    DevState* d_state = nullptr;
    unsigned long long* d_best = nullptr;
    unsigned int* d_done = nullptr;
    void* d_attn_ws = nullptr;
    float* d_rowmax = nullptr;  // prefill products on the tensor cores: each token row's largest |x|
    __half* d_hl = nullptr;     // and its rows scaled and split into f16 hi / lo (max_seq x 2 x widest k)

    int32_t* h_ids = nullptr;
    int32_t* h_out = nullptr;
    float* h_logits = nullptr;
    DevState* h_state = nullptr;

    std::vector<LayerDev> layers;
    PackedQ8 embd{}, head{};
    const float* out_norm = nullptr;

    int len = 0;
    int64_t launches = 0;
    bool fuse_o = false;                 // decode attention kernel also applies W_o and the residual
    int front_cl = 0;                    // > 0: norm + QKV + attention + W_o as one kernel (this cluster size)
    int mlp_clusters = 0;                // > 0: gate/up + down as one kernel with this many 16-CTA clusters
    cudaGraph_t decode_graph = nullptr;
    cudaGraphExec_t decode_exec = nullptr;
    // kMultiSteps decode steps in one graph: the programmatic dependent launches
    // chain across the steps too (no gap between graph launches)
    cudaGraph_t multi_graph = nullptr;
    cudaGraphExec_t multi_exec = nullptr;
    int decode_kernels = 0;

    size_t layer_cache_floats() const { return (size_t)cfg.n_head_kv * cfg.max_seq * cfg.head_dim; }
    float* kcache(int l) const { return d_kcache + (size_t)l * layer_cache_floats(); }
    float* vcache(int l) const { return d_vcache + (size_t)l * layer_cache_floats(); }
};

#define LQ8_CK(ctx, call)                           \
    do {                                            \
        cudaError_t e_ = (call);                    \
        if (e_ != cudaSuccess) {                    \
            if (ctx) (ctx)->failed = true;          \
            return LQ8_ERR_CUDA;                    \
        }                                           \
    } while (0)

namespace {

void free_ctx_memory(llama_q8_ctx* c) {
    if (c->decode_exec) cudaGraphExecDestroy(c->decode_exec);
    if (c->decode_graph) cudaGraphDestroy(c->decode_graph);
    if (c->multi_exec) cudaGraphExecDestroy(c->multi_exec);
    if (c->multi_graph) cudaGraphDestroy(c->multi_graph);
    void* dev[] = {c->d_weights, c->d_norms, c->d_rope_cos, c->d_rope_sin, c->d_kcache, c->d_vcache,
                   c->d_x, c->d_y, c->d_q, c->d_o, c->d_a, c->d_part, c->d_xsum, c->d_xr, c->d_mlp, c->d_logits, c->d_ids,
                   c->d_out_ids,
                   c->d_state, c->d_best, c->d_done, c->d_attn_ws, c->d_rowmax, c->d_hl};
    for (void* p : dev)
        if (p) cudaFree(p);
    void* host[] = {c->h_ids, c->h_out, c->h_logits, c->h_state};
    for (void* p : host)
        if (p) cudaFreeHost(p);
    if (c->stream) cudaStreamDestroy(c->stream);
}

EpiArgs qkv_epi(const llama_q8_ctx* c, int l) {
    EpiArgs e;
    e.q_out = c->d_q;
    e.k_cache = c->kcache(l);
    e.v_cache = c->vcache(l);
    e.q_rows = c->q_rows;
    e.kv_rows = c->kv_rows;
    e.head_dim = c->cfg.head_dim;
    e.max_seq = c->cfg.max_seq;
    e.rope_cos = c->d_rope_cos;
    e.rope_sin = c->d_rope_sin;
    return e;
}

EpiArgs head_epi(const llama_q8_ctx* c, int pos_after) {
    EpiArgs e;
    e.logits = c->d_logits;
    e.best_key = c->d_best;
    e.done_count = c->d_done;
    e.st = c->d_state;
    e.out_ids = c->d_out_ids;
    e.pos_after = pos_after;
    return e;
}

// Bytes of a Q8_0 matrix: 34 per 32 weights.
double q8_bytes(int64_t rows, int64_t k) { return (double)rows * (double)k * 34.0 / 32.0; }

// One decode step (T = 1): position and token come from the device state, so
// the same launch sequence serves every position and can be captured once.
// With a profiler, each launch is bracketed by events and tagged with its
// algorithmic bytes (attention bytes are per cached position, scaled by the
// step's cache length when the times are read); launches are then plain, since
// an event node between two kernels leaves nothing for PDL to overlap.
FrontArgs front_args(llama_q8_ctx* c, int l) {
    const llama_q8_config& cfg = c->cfg;
    const LayerDev& L = c->layers[l];
    FrontArgs fa{};
    fa.x = c->d_x;
    if (c->mlp_clusters > 0 && l > 0) {  // x = the MLP's residual base + its cluster partials
        fa.x = c->d_xr;
        fa.xparts = c->d_mlp;
        fa.n_xparts = c->mlp_clusters;
        fa.x_store = c->d_x;
    }
    fa.g = L.attn_norm;
    fa.eps = cfg.rms_eps;
    fa.wqkv = L.qkv;
    fa.wo = L.o;
    fa.kc = c->kcache(l);
    fa.vc = c->vcache(l);
    fa.rope_cos = c->d_rope_cos;
    fa.rope_sin = c->d_rope_sin;
    fa.n_head = cfg.n_head;
    fa.n_kv = cfg.n_head_kv;
    fa.stride = cfg.max_seq;
    fa.st = c->d_state;
    fa.scale = 1.0f / sqrtf((float)cfg.head_dim);
    fa.part = c->d_part;
    fa.part_stride = cfg.n_embd;
    fa.err = &c->d_state->err;
    return fa;
}

cudaError_t enqueue_decode_step(llama_q8_ctx* c, int* n_kernels, StepLayout* layout = nullptr,
                                unsigned long long* stamps = nullptr) {
    const llama_q8_config& cfg = c->cfg;
    cudaStream_t s = c->stream;
    const bool pdl = true;
    const int64_t h = cfg.n_embd, F = cfg.n_ff, qr = c->q_rows, kvr = c->kv_rows;
    int n = 0;
    cudaError_t err = cudaSuccess;
    unsigned long long* stp = nullptr;  // this launch's two stamps (instrumented graph only)
    auto run = [&](int fam, double bytes, double kv_per_pos, auto&& launch) {
        if (err != cudaSuccess) return;
        stp = stamps ? stamps + 2 * n : nullptr;
        if (layout) layout->recs.push_back({fam, bytes, kv_per_pos});
        err = launch();
        ++n;
    };
    auto stamped = [&](EpiArgs x) {
        x.stamp = stp;
        return x;
    };
    run(F_EMBED, q8_bytes(1, h) + 4.0 * h, 0.0, [&] {
        return launch_embed(c->embd, nullptr, 1, c->d_state, c->d_state, c->d_x, cfg.n_vocab, pdl, s, stp);
    });
    for (int l = 0; l < cfg.n_layer; ++l) {
        const LayerDev& L = c->layers[l];
        EpiArgs e = qkv_epi(c, l);
        e.state = c->d_state;
        EpiArgs r;
        r.y = c->d_x;
        if (c->front_cl > 0 || c->fuse_o) {
            // attention + W_o per KV head (partials), the sum folded into the gate/up kernel's norm,
            // and the down projection's residual taken from that sum
            if (c->front_cl > 0) {
                FrontArgs fa = front_args(c, l);
                run(F_FRONT, q8_bytes(qr + 2 * kvr, h) + q8_bytes(h, qr) + 8.0 * h + 4.0 * h * cfg.n_head_kv,
                    8.0 * (double)cfg.n_head_kv * cfg.head_dim, [&] {
                        fa.stamp = stp;
                        return launch_layer_front(fa, cfg.head_dim, c->front_cl, pdl, s);
                    });
            } else {
                run(F_QKV, q8_bytes(qr + 2 * kvr, h) + 8.0 * h + 4.0 * (qr + 2 * kvr), 0.0, [&] {
                    return launch_gemv(L.qkv, c->d_x, L.attn_norm, cfg.rms_eps, EPI_QKV, stamped(e), pdl,
                                       &c->d_state->err, s);
                });
                run(F_ATTN_O, 4.0 * qr + q8_bytes(h, qr) + 4.0 * h * cfg.n_head_kv,
                    8.0 * (double)cfg.n_head_kv * cfg.head_dim, [&] {
                        return launch_attn_oproj(c->d_q, c->kcache(l), c->vcache(l), cfg.n_head, cfg.n_head_kv,
                                                 cfg.head_dim, cfg.max_seq, c->d_state, L.o, c->d_part, (int)h, pdl,
                                                 &c->d_state->err, s, stp);
                    });
            }
            if (c->mlp_clusters > 0) {
                MlpArgs ma{};
                ma.x = c->d_x;
                ma.attn_part = c->d_part;
                ma.n_attn_part = cfg.n_head_kv;
                ma.g = L.ffn_norm;
                ma.eps = cfg.rms_eps;
                ma.wgu = L.gu;
                ma.wdown = L.down;
                ma.xr_out = c->d_xr;
                ma.mlp_part = c->d_mlp;
                ma.err = &c->d_state->err;
                run(F_MLP, q8_bytes(2 * F, h) + q8_bytes(h, F) + 4.0 * h * (3 + cfg.n_head_kv + c->mlp_clusters), 0.0,
                    [&] {
                        ma.stamp = stp;
                        return launch_decode_mlp(ma, pdl, s);
                    });
                continue;
            }
            EpiArgs g;
            g.a_out = c->d_a;
            GemvPreSum pre;
            pre.part = c->d_part;
            pre.n_part = cfg.n_head_kv;
            pre.part_stride = (int)h;
            pre.x_sum_out = c->d_xsum;
            run(F_GATEUP, q8_bytes(2 * F, h) + 4.0 * h * (2 + cfg.n_head_kv) + 4.0 * F, 0.0, [&] {
                return launch_gemv(L.gu, c->d_x, L.ffn_norm, cfg.rms_eps, EPI_SILU, stamped(g), pdl,
                                   &c->d_state->err, s, &pre);
            });
            EpiArgs rd;
            rd.y = c->d_x;
            rd.res = c->d_xsum;
            run(F_DOWN, q8_bytes(h, F) + 4.0 * F + 8.0 * h, 0.0,
                [&] {
                    return launch_gemv(L.down, c->d_a, nullptr, 0.f, EPI_RESIDUAL, stamped(rd), pdl, &c->d_state->err, s);
                });
        } else {
            run(F_QKV, q8_bytes(qr + 2 * kvr, h) + 8.0 * h + 4.0 * (qr + 2 * kvr), 0.0,
                [&] {
                    return launch_gemv(L.qkv, c->d_x, L.attn_norm, cfg.rms_eps, EPI_QKV, stamped(e), pdl,
                                       &c->d_state->err, s);
                });
            run(F_ATTN, 8.0 * qr, 8.0 * (double)cfg.n_head_kv * cfg.head_dim, [&] {
                return launch_attn_decode_cluster(c->d_q, c->kcache(l), c->vcache(l), cfg.n_head, cfg.n_head_kv,
                                                  cfg.head_dim, cfg.max_seq, 0, c->d_state, c->d_o, pdl,
                                                  &c->d_state->err, s, stp);
            });
            run(F_OPROJ, q8_bytes(h, qr) + 4.0 * qr + 8.0 * h, 0.0,
                [&] {
                    return launch_gemv(L.o, c->d_o, nullptr, 0.f, EPI_RESIDUAL, stamped(r), pdl, &c->d_state->err, s);
                });
            EpiArgs g;
            g.a_out = c->d_a;
            run(F_GATEUP, q8_bytes(2 * F, h) + 8.0 * h + 4.0 * F, 0.0, [&] {
                return launch_gemv(L.gu, c->d_x, L.ffn_norm, cfg.rms_eps, EPI_SILU, stamped(g), pdl,
                                   &c->d_state->err, s);
            });
            run(F_DOWN, q8_bytes(h, F) + 4.0 * F + 8.0 * h, 0.0,
                [&] {
                    return launch_gemv(L.down, c->d_a, nullptr, 0.f, EPI_RESIDUAL, stamped(r), pdl, &c->d_state->err, s);
                });
        }
    }
    if (c->mlp_clusters > 0) {  // the last layer's residual = its base + the MLP's cluster partials
        GemvPreSum pre;
        pre.part = c->d_mlp;
        pre.n_part = c->mlp_clusters;
        pre.part_stride = (int)h;
        run(F_HEAD, q8_bytes(cfg.n_vocab, h) + 8.0 * h + 4.0 * h * c->mlp_clusters + 4.0 * cfg.n_vocab, 0.0, [&] {
            return launch_gemv(c->head, c->d_xr, c->out_norm, cfg.rms_eps, EPI_ARGMAX, stamped(head_epi(c, -1)), pdl,
                               &c->d_state->err, s, &pre, cfg.head_splits);
        });
    } else {
        run(F_HEAD, q8_bytes(cfg.n_vocab, h) + 8.0 * h + 4.0 * cfg.n_vocab, 0.0, [&] {
            return launch_gemv(c->head, c->d_x, c->out_norm, cfg.rms_eps, EPI_ARGMAX, stamped(head_epi(c, -1)), pdl,
                               &c->d_state->err, s, nullptr, cfg.head_splits);
        });
    }
    // the instrumented graph ends with a stamp kernel whose wait returns when the lm_head has completed
    if (err == cudaSuccess && stamps) err = launch_stamp(stamps + 2 * n, s);
    if (n_kernels) *n_kernels = n;
    return err;
}

// Prefill of T > 1 tokens already in device memory at positions
// [index_pos, index_pos + T); ends with the lm_head + argmax of the last row.
cudaError_t enqueue_prefill(llama_q8_ctx* c, const int32_t* d_ids, int T, int index_pos) {
    const llama_q8_config& cfg = c->cfg;
    cudaStream_t s = c->stream;
    const int h = cfg.n_embd;
    cudaError_t err = launch_embed(c->embd, d_ids, T, nullptr, c->d_state, c->d_x, cfg.n_vocab, true, s);
    // the tensor-core operand of every product (rows scaled and split), one
    // buffer reused in stream order; the RMSNorms write it for the Q/K/V and
    // gate/up products in place of y when those run on the tensor cores
    const SplitRows sp{c->d_rowmax, c->d_hl};
    const bool tc_norm = matmul_on_tensor_cores(T, 0, h, MATMUL_AUTO);
    float* y = tc_norm ? nullptr : c->d_y;
    const SplitRows* norm_split = tc_norm ? &sp : nullptr;
    for (int l = 0; l < cfg.n_layer && err == cudaSuccess; ++l) {
        const LayerDev& L = c->layers[l];
        err = launch_rmsnorm(c->d_x, L.attn_norm, cfg.rms_eps, T, h, y, true, s, norm_split);
        EpiArgs e = qkv_epi(c, l);
        e.pos0 = index_pos;
        if (err == cudaSuccess) err = launch_matmul_rows(L.qkv, c->d_y, T, h, EPI_QKV, e, true, &c->d_state->err, s, sp,
                                                         MATMUL_AUTO, true);
        if (err == cudaSuccess)
            err = launch_attn_prefill(c->d_q, c->kcache(l), c->vcache(l), T, index_pos, cfg.n_head, cfg.n_head_kv,
                                      cfg.head_dim, cfg.max_seq, c->d_o, true, s);
        EpiArgs r;
        r.y = c->d_x;
        r.ldy = h;
        if (err == cudaSuccess) err = launch_matmul_rows(L.o, c->d_o, T, c->q_rows, EPI_RESIDUAL, r, true, &c->d_state->err, s, sp);
        if (err == cudaSuccess) err = launch_rmsnorm(c->d_x, L.ffn_norm, cfg.rms_eps, T, h, y, true, s, norm_split);
        EpiArgs g;
        g.a_out = c->d_a;
        g.lda = cfg.n_ff;
        if (err == cudaSuccess) err = launch_matmul_rows(L.gu, c->d_y, T, h, EPI_SILU, g, true, &c->d_state->err, s, sp,
                                                         MATMUL_AUTO, true);
        if (err == cudaSuccess) err = launch_matmul_rows(L.down, c->d_a, T, cfg.n_ff, EPI_RESIDUAL, r, true, &c->d_state->err, s, sp);
    }
    if (err == cudaSuccess)
        err = launch_gemv(c->head, c->d_x + (size_t)(T - 1) * h, c->out_norm, cfg.rms_eps, EPI_ARGMAX,
                          head_epi(c, index_pos + T), true, &c->d_state->err, s, nullptr, cfg.head_splits);
    return err;
}

// Status raised on the device (read back into h_state): an out-of-range id in
// device memory (LQ8_ERR_TOKEN, the context stays usable), or a bounded wait
// that timed out inside a kernel (the context is marked failed).
llama_q8_status device_status(llama_q8_ctx* c) {
    const int e = c->h_state->err;
    if (e == 0) return LQ8_OK;
    if (e == LQ8_ERR_TOKEN) return LQ8_ERR_TOKEN;
    c->failed = true;
    return LQ8_ERR_CUDA;
}

// embed, per layer two norms, attention and four products (on the tensor
// cores, W_o and the down projection after a row-maximum pass each; the
// norms give Q/K/V and gate/up theirs), the lm_head
int prefill_kernel_count(const llama_q8_ctx* c, int T) {
    const int per_layer = 7 + (matmul_on_tensor_cores(T, 0, 0, MATMUL_AUTO) ? 2 : 0);
    return 1 + per_layer * c->cfg.n_layer + 1;
}

constexpr int kMultiSteps = 8;

// Capture `steps` decode steps back to back into one instantiated graph.
cudaError_t capture_decode_steps(llama_q8_ctx* c, int steps, cudaGraph_t* graph, cudaGraphExec_t* exec, int* n_kernels) {
    cudaError_t err = cudaStreamBeginCapture(c->stream, cudaStreamCaptureModeThreadLocal);
    if (err != cudaSuccess) return err;
    cudaError_t lerr = cudaSuccess;
    for (int i = 0; i < steps && lerr == cudaSuccess; ++i) lerr = enqueue_decode_step(c, n_kernels);
    cudaGraph_t g = nullptr;
    err = cudaStreamEndCapture(c->stream, &g);
    if (lerr != cudaSuccess) {
        if (g) cudaGraphDestroy(g);
        return lerr;
    }
    if (err != cudaSuccess) return err;
    err = cudaGraphInstantiate(exec, g, 0);
    if (err != cudaSuccess) {
        cudaGraphDestroy(g);
        return err;
    }
    *graph = g;
    return cudaSuccess;
}

cudaError_t ensure_decode_graph(llama_q8_ctx* c) {
    if (c->decode_exec) return cudaSuccess;
    int n = 0;
    cudaError_t err = capture_decode_steps(c, 1, &c->decode_graph, &c->decode_exec, &n);
    if (err != cudaSuccess) return err;
    c->decode_kernels = n;
    int n8 = 0;
    return capture_decode_steps(c, kMultiSteps, &c->multi_graph, &c->multi_exec, &n8);
}

// n decode steps on the context stream: the multi-step graph while it fits,
// then single steps. Returns the number of kernel launches enqueued.
cudaError_t launch_decode_steps(llama_q8_ctx* c, int n) {
    cudaError_t err = cudaSuccess;
    for (; n >= kMultiSteps && err == cudaSuccess; n -= kMultiSteps) err = cudaGraphLaunch(c->multi_exec, c->stream);
    for (; n > 0 && err == cudaSuccess; --n) err = cudaGraphLaunch(c->decode_exec, c->stream);
    return err;
}

llama_q8_status check_positions(const llama_q8_ctx* c, int T, int index_pos) {
    if (index_pos < 0) return LQ8_ERR_POS;
    if ((int64_t)index_pos + T > c->cfg.max_seq) return LQ8_ERR_CTX;
    if (index_pos != 0 && index_pos != c->len) return LQ8_ERR_POS;
    return LQ8_OK;
}

// Runs one forward of host ids (T >= 1) and leaves the logits and greedy
// token on the device (d_logits, d_out_ids[0], state.token).
llama_q8_status run_forward(llama_q8_ctx* c, const int32_t* ids, int T, int index_pos) {
    if (!c || !ids) return LQ8_ERR_ARG;
    if (c->failed) return LQ8_ERR_STATE;
    if (T <= 0) return LQ8_ERR_ARG;
    for (int i = 0; i < T; ++i)
        if (ids[i] < 0 || ids[i] >= c->cfg.n_vocab) return LQ8_ERR_TOKEN;
    llama_q8_status st = check_positions(c, T, index_pos);
    if (st != LQ8_OK) return st;
    LQ8_CK(c, cudaSetDevice(c->device));
    if (T == 1) {
        LQ8_CK(c, ensure_decode_graph(c));
        LQ8_CK(c, launch_set_state(c->d_state, index_pos, ids[0], 0, c->stream));
        LQ8_CK(c, cudaGraphLaunch(c->decode_exec, c->stream));
        c->launches += 1 + c->decode_kernels;
    } else {
        std::memcpy(c->h_ids, ids, sizeof(int32_t) * T);
        LQ8_CK(c, cudaMemcpyAsync(c->d_ids, c->h_ids, sizeof(int32_t) * T, cudaMemcpyHostToDevice, c->stream));
        LQ8_CK(c, launch_set_state(c->d_state, index_pos, -1, 0, c->stream));
        LQ8_CK(c, enqueue_prefill(c, c->d_ids, T, index_pos));
        c->launches += 1 + prefill_kernel_count(c, T);
    }
    c->len = index_pos + T;
    return LQ8_OK;
}

}  // namespace

extern "C" {

llama_q8_status llama_q8_selftest_wait_timeout(int32_t* code) {
    if (!code) return LQ8_ERR_ARG;
    int* d = nullptr;
    if (cudaMalloc(&d, sizeof(int)) != cudaSuccess) return LQ8_ERR_OOM;
    cudaError_t e = cudaMemset(d, 0, sizeof(int));
    if (e == cudaSuccess) e = launch_wait_timeout(d, 41, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    int h = 0;
    if (e == cudaSuccess) e = cudaMemcpy(&h, d, sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return LQ8_ERR_CUDA;
    *code = h;
    return LQ8_OK;
}

const char* llama_q8_status_str(llama_q8_status s) {
    switch (s) {
        case LQ8_OK: return "ok";
        case LQ8_ERR_ARG: return "invalid argument";
        case LQ8_ERR_POS: return "index_pos is neither 0 nor the cached length";
        case LQ8_ERR_CTX: return "index_pos + T exceeds max_seq";
        case LQ8_ERR_TOKEN: return "token id out of range";
        case LQ8_ERR_CUDA: return "CUDA error";
        case LQ8_ERR_OOM: return "out of memory";
        case LQ8_ERR_STATE: return "context unusable or call out of order";
        case LQ8_ERR_UNSUPPORTED: return "unsupported shape";
        case LQ8_ERR_FORMAT: return "not a readable GGUF Llama file";
    }
    return "unknown status";
}

llama_q8_status llama_q8_load(const llama_q8_config* cfg, const llama_q8_weights* w, int32_t device,
                              llama_q8_ctx** out) {
    if (!cfg || !w || !out || !w->layers || !w->token_embd || !w->output_norm) return LQ8_ERR_ARG;
    *out = nullptr;
    const llama_q8_config& C = *cfg;
    if (C.n_layer <= 0 || C.n_embd <= 0 || C.n_head <= 0 || C.n_head_kv <= 0 || C.n_ff <= 0 ||
        C.n_vocab <= 0 || C.max_seq <= 0 || C.head_dim <= 0 || !(C.rms_eps >= 0.f) || !(C.rope_theta > 0.f))
        return LQ8_ERR_ARG;
    if (C.n_head % C.n_head_kv != 0) return LQ8_ERR_ARG;
    if (C.decode_kernel < 0 || C.decode_kernel > 5) return LQ8_ERR_ARG;
    // 2 and 5 (one cluster kernel for the whole step / per layer) were measured
    // slower than the per-layer kernels and are not built
    if (C.decode_kernel == 2 || C.decode_kernel == 5) return LQ8_ERR_UNSUPPORTED;
    if (C.rope_style != 0 && C.rope_style != 1) return LQ8_ERR_ARG;
    if (C.head_splits < 0 || C.head_splits == 1 || C.head_splits > 8 ||
        (C.head_splits > 0 && C.n_embd > 0 && C.n_embd / 32 < C.head_splits))
        return LQ8_ERR_ARG;
    if (!C.tied_output && !w->output) return LQ8_ERR_ARG;
    for (int l = 0; l < C.n_layer; ++l) {
        const llama_q8_layer_weights& L = w->layers[l];
        if (!L.attn_norm || !L.ffn_norm || !L.attn_q || !L.attn_k || !L.attn_v || !L.attn_output ||
            !L.ffn_gate || !L.ffn_up || !L.ffn_down)
            return LQ8_ERR_ARG;
    }
    if (C.head_dim != 64 && C.head_dim != 128) return LQ8_ERR_UNSUPPORTED;
    if (C.n_embd % 32 || C.n_ff % 32 || C.n_head / C.n_head_kv > 8) return LQ8_ERR_UNSUPPORTED;
    if (C.n_embd > 51200 || C.n_ff > 51200 || C.n_head * C.head_dim > 51200) return LQ8_ERR_UNSUPPORTED;

    llama_q8_ctx* c = new (std::nothrow) llama_q8_ctx();
    if (!c) return LQ8_ERR_OOM;
    c->cfg = C;
    c->device = device;
    c->q_rows = C.n_head * C.head_dim;
    c->kv_rows = C.n_head_kv * C.head_dim;
    const int h = C.n_embd, F = C.n_ff, V = C.n_vocab, L = C.n_layer, hd = C.head_dim;
    const int qkv_rows = c->q_rows + 2 * c->kv_rows;

#define LOAD_CK(call)                          \
    do {                                       \
        cudaError_t e_ = (call);               \
        if (e_ != cudaSuccess) {               \
            free_ctx_memory(c);                \
            delete c;                          \
            return e_ == cudaErrorMemoryAllocation ? LQ8_ERR_OOM : LQ8_ERR_CUDA; \
        }                                      \
    } while (0)

    LOAD_CK(cudaSetDevice(device));
    LOAD_CK(ensure_kernel_attributes());
    LOAD_CK(cudaStreamCreateWithFlags(&c->stream, cudaStreamNonBlocking));

    // --- weight arena ---------------------------------------------------
    const size_t b_qkv = align256(packed_total_bytes(qkv_rows, h));
    const size_t b_o = align256(packed_total_bytes(h, c->q_rows));
    const size_t b_gu = align256(packed_total_bytes(2 * (int64_t)F, h));
    const size_t b_down = align256(packed_total_bytes(h, F));
    const size_t b_layer = b_qkv + b_o + b_gu + b_down;
    const size_t b_embd = align256(packed_total_bytes(V, h));
    const size_t b_head = C.tied_output ? 0 : b_embd;
    const size_t w_bytes = b_layer * L + b_embd + b_head;
    LOAD_CK(cudaMalloc(&c->d_weights, w_bytes));
    LOAD_CK(cudaMemsetAsync(c->d_weights, 0, w_bytes, c->stream));
    LOAD_CK(cudaMalloc(&c->d_norms, sizeof(float) * (size_t)(2 * L + 1) * h));

    // staging for host Q8_0 blocks (largest matrix)
    size_t max_aos = (size_t)V * (h / 32) * 34;
    max_aos = std::max(max_aos, (size_t)F * (h / 32) * 34);
    max_aos = std::max(max_aos, (size_t)h * (F / 32) * 34);
    max_aos = std::max(max_aos, (size_t)h * (c->q_rows / 32) * 34);
    uint8_t* staging = nullptr;
    if (!w->on_device) LOAD_CK(cudaMalloc(&staging, max_aos));

    // neox_heads > 0: rows are that many heads of head_dim rows; row i and row
    // i + head_dim/2 of each head go to rows 2i and 2i+1 (the NEOX pairs side by side)
    auto pack = [&](const void* src, int64_t rows, int64_t k, uint8_t* dst, int64_t dst_rows, int64_t off,
                    int64_t stride, int neox_heads = 0) -> cudaError_t {
        const uint8_t* s = reinterpret_cast<const uint8_t*>(src);
        cudaError_t err = cudaSuccess;
        if (!w->on_device) {
            err = cudaMemcpyAsync(staging, src, (size_t)rows * (k / 32) * 34, cudaMemcpyHostToDevice, c->stream);
            if (err != cudaSuccess) return err;
            s = staging;
        }
        if (neox_heads > 0) {
            const int64_t hd = C.head_dim, half = hd / 2, row_bytes = (k / 32) * 34;
            for (int hh = 0; hh < neox_heads && err == cudaSuccess; ++hh) {
                err = launch_pack(s + hh * hd * row_bytes, half, k, dst, dst_rows, off + hh * hd, 2, c->stream);
                if (err == cudaSuccess)
                    err = launch_pack(s + (hh * hd + half) * row_bytes, half, k, dst, dst_rows, off + hh * hd + 1, 2,
                                      c->stream);
            }
        } else {
            err = launch_pack(s, rows, k, dst, dst_rows, off, stride, c->stream);
        }
        if (err != cudaSuccess) return err;
        if (!w->on_device) err = cudaStreamSynchronize(c->stream);  // staging is reused
        return err;
    };
    const cudaMemcpyKind nk = w->on_device ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;

    c->layers.resize(L);
    for (int l = 0; l < L; ++l) {
        const llama_q8_layer_weights& LW = w->layers[l];
        uint8_t* base = c->d_weights + b_layer * l;
        uint8_t* p_qkv = base;
        uint8_t* p_o = p_qkv + b_qkv;
        uint8_t* p_gu = p_o + b_o;
        uint8_t* p_down = p_gu + b_gu;
        const int neox = C.rope_style == 1;
        cudaError_t err = pack(LW.attn_q, c->q_rows, h, p_qkv, qkv_rows, 0, 1, neox ? C.n_head : 0);
        if (err == cudaSuccess)
            err = pack(LW.attn_k, c->kv_rows, h, p_qkv, qkv_rows, c->q_rows, 1, neox ? C.n_head_kv : 0);
        if (err == cudaSuccess) err = pack(LW.attn_v, c->kv_rows, h, p_qkv, qkv_rows, c->q_rows + c->kv_rows, 1);
        if (err == cudaSuccess) err = pack(LW.attn_output, h, c->q_rows, p_o, h, 0, 1);
        if (err == cudaSuccess) err = pack(LW.ffn_gate, F, h, p_gu, 2 * (int64_t)F, 0, 2);
        if (err == cudaSuccess) err = pack(LW.ffn_up, F, h, p_gu, 2 * (int64_t)F, 1, 2);
        if (err == cudaSuccess) err = pack(LW.ffn_down, h, F, p_down, h, 0, 1);
        float* n_attn = c->d_norms + (size_t)(2 * l) * h;
        float* n_ffn = n_attn + h;
        if (err == cudaSuccess) err = cudaMemcpyAsync(n_attn, LW.attn_norm, sizeof(float) * h, nk, c->stream);
        if (err == cudaSuccess) err = cudaMemcpyAsync(n_ffn, LW.ffn_norm, sizeof(float) * h, nk, c->stream);
        if (err != cudaSuccess) {
            if (staging) cudaFree(staging);
            LOAD_CK(err);
        }
        LayerDev& D = c->layers[l];
        D.attn_norm = n_attn;
        D.ffn_norm = n_ffn;
        D.qkv = packed_view(p_qkv, qkv_rows, h);
        D.o = packed_view(p_o, h, c->q_rows);
        D.gu = packed_view(p_gu, 2 * (int64_t)F, h);
        D.down = packed_view(p_down, h, F);
    }
    uint8_t* p_embd = c->d_weights + b_layer * L;
    cudaError_t err = pack(w->token_embd, V, h, p_embd, V, 0, 1);
    c->embd = packed_view(p_embd, V, h);
    c->head = c->embd;
    if (err == cudaSuccess && !C.tied_output) {
        uint8_t* p_head = p_embd + b_embd;
        err = pack(w->output, V, h, p_head, V, 0, 1);
        c->head = packed_view(p_head, V, h);
    }
    float* n_out = c->d_norms + (size_t)(2 * L) * h;
    if (err == cudaSuccess) err = cudaMemcpyAsync(n_out, w->output_norm, sizeof(float) * h, nk, c->stream);
    c->out_norm = n_out;
    if (err == cudaSuccess) err = cudaStreamSynchronize(c->stream);
    if (staging) cudaFree(staging);
    LOAD_CK(err);

    // --- rotary table: angle p * theta^(-2i/hd) in double, stored f32 ---
    {
        const int half = hd / 2;
        std::vector<float> cs((size_t)C.max_seq * half), sn((size_t)C.max_seq * half);
        for (int i = 0; i < half; ++i) {
            const double f = std::pow((double)C.rope_theta, -2.0 * i / hd);
            for (int p = 0; p < C.max_seq; ++p) {
                const double a = (double)p * f;
                cs[(size_t)p * half + i] = (float)std::cos(a);
                sn[(size_t)p * half + i] = (float)std::sin(a);
            }
        }
        LOAD_CK(cudaMalloc(&c->d_rope_cos, sizeof(float) * cs.size()));
        LOAD_CK(cudaMalloc(&c->d_rope_sin, sizeof(float) * sn.size()));
        LOAD_CK(cudaMemcpy(c->d_rope_cos, cs.data(), sizeof(float) * cs.size(), cudaMemcpyHostToDevice));
        LOAD_CK(cudaMemcpy(c->d_rope_sin, sn.data(), sizeof(float) * sn.size(), cudaMemcpyHostToDevice));
    }

    // --- KV cache, activations, scratch, host staging ------------------
    const size_t cache_floats = (size_t)L * c->layer_cache_floats();
    LOAD_CK(cudaMalloc(&c->d_kcache, sizeof(float) * cache_floats));
    LOAD_CK(cudaMalloc(&c->d_vcache, sizeof(float) * cache_floats));
    LOAD_CK(cudaMemsetAsync(c->d_kcache, 0, sizeof(float) * cache_floats, c->stream));
    LOAD_CK(cudaMemsetAsync(c->d_vcache, 0, sizeof(float) * cache_floats, c->stream));
    const size_t T = (size_t)C.max_seq;
    LOAD_CK(cudaMalloc(&c->d_x, sizeof(float) * T * h));
    LOAD_CK(cudaMalloc(&c->d_y, sizeof(float) * T * h));
    LOAD_CK(cudaMalloc(&c->d_q, sizeof(float) * T * c->q_rows));
    LOAD_CK(cudaMalloc(&c->d_o, sizeof(float) * T * c->q_rows));
    LOAD_CK(cudaMalloc(&c->d_a, sizeof(float) * T * F));
    LOAD_CK(cudaMalloc(&c->d_rowmax, sizeof(float) * T));
    LOAD_CK(cudaMalloc(&c->d_hl, sizeof(__half) * T * 2 * std::max({(size_t)h, (size_t)c->q_rows, (size_t)F})));
    LOAD_CK(cudaMalloc(&c->d_part, sizeof(float) * C.n_head_kv * h));
    LOAD_CK(cudaMalloc(&c->d_xsum, sizeof(float) * h));
    LOAD_CK(cudaMalloc(&c->d_xr, sizeof(float) * h));
    LOAD_CK(cudaMalloc(&c->d_mlp, sizeof(float) * h * (F / 32 / 8 + 1)));
    LOAD_CK(cudaMalloc(&c->d_logits, sizeof(float) * V));
    LOAD_CK(cudaMalloc(&c->d_ids, sizeof(int32_t) * T));
    LOAD_CK(cudaMalloc(&c->d_out_ids, sizeof(int32_t) * (T + 1)));
    LOAD_CK(cudaMalloc(&c->d_state, sizeof(DevState)));
    LOAD_CK(cudaMalloc(&c->d_best, sizeof(unsigned long long)));
    LOAD_CK(cudaMalloc(&c->d_done, sizeof(unsigned int)));
    const size_t ws = attn_workspace_bytes(C.n_head, C.n_head_kv, hd, C.max_seq);
    LOAD_CK(cudaMalloc(&c->d_attn_ws, ws));
    LOAD_CK(cudaMemsetAsync(c->d_attn_ws, 0, ws, c->stream));
    LOAD_CK(cudaMemsetAsync(c->d_state, 0, sizeof(DevState), c->stream));
    LOAD_CK(cudaMemsetAsync(c->d_best, 0, sizeof(unsigned long long), c->stream));
    LOAD_CK(cudaMemsetAsync(c->d_done, 0, sizeof(unsigned int), c->stream));
    LOAD_CK(cudaMallocHost(&c->h_ids, sizeof(int32_t) * T));
    LOAD_CK(cudaMallocHost(&c->h_out, sizeof(int32_t) * (T + 1)));
    LOAD_CK(cudaMallocHost(&c->h_logits, sizeof(float) * V));
    LOAD_CK(cudaMallocHost(&c->h_state, sizeof(DevState)));
    LOAD_CK(cudaStreamSynchronize(c->stream));
    // decode_kernel: 0 automatic (two per layer when the model fits, else three, four or five),
    // 1 five per layer, 3 four per layer, 4 three per layer
    bool unsupported = false;
    if (C.decode_kernel == 0 || C.decode_kernel == 3 || C.decode_kernel == 4) {
        c->fuse_o = attn_oproj_fused_supported(C.n_head, C.n_head_kv, hd, c->layers[0].o);
        cudaGetLastError();
        if (C.decode_kernel != 3 && c->fuse_o) c->front_cl = layer_front_cluster_size(front_args(c, 0), hd);
        cudaGetLastError();
        if (C.decode_kernel == 0 && c->front_cl > 0) c->mlp_clusters = decode_mlp_clusters(h, F, c->layers[0].gu.rows);
        // the front and MLP kernels read at most 8 partials of their input
        if (c->mlp_clusters > 8 || C.n_head_kv > 8) c->mlp_clusters = 0;
        cudaGetLastError();
        unsupported = (C.decode_kernel == 3 && !c->fuse_o) || (C.decode_kernel == 4 && c->front_cl == 0);
    }
    if (unsupported) {
        free_ctx_memory(c);
        delete c;
        return LQ8_ERR_UNSUPPORTED;
    }
    LOAD_CK(ensure_decode_graph(c));
#undef LOAD_CK
    c->len = 0;
    *out = c;
    return LQ8_OK;
}

llama_q8_status llama_q8_forward(llama_q8_ctx* ctx, const int32_t* ids, int32_t T, int32_t index_pos,
                                 float* logits) {
    if (!logits) return LQ8_ERR_ARG;
    llama_q8_status st = run_forward(ctx, ids, T, index_pos);
    if (st != LQ8_OK) return st;
    LQ8_CK(ctx, cudaMemcpyAsync(ctx->h_logits, ctx->d_logits, sizeof(float) * ctx->cfg.n_vocab,
                                cudaMemcpyDeviceToHost, ctx->stream));
    LQ8_CK(ctx, cudaMemcpyAsync(ctx->h_state, ctx->d_state, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    LQ8_CK(ctx, cudaStreamSynchronize(ctx->stream));
    std::memcpy(logits, ctx->h_logits, sizeof(float) * ctx->cfg.n_vocab);
    return device_status(ctx);
}

llama_q8_status llama_q8_forward_argmax(llama_q8_ctx* ctx, const int32_t* ids, int32_t T, int32_t index_pos,
                                        int32_t* next) {
    if (!next) return LQ8_ERR_ARG;
    llama_q8_status st = run_forward(ctx, ids, T, index_pos);
    if (st != LQ8_OK) return st;
    LQ8_CK(ctx, cudaMemcpyAsync(ctx->h_state, ctx->d_state, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    LQ8_CK(ctx, cudaStreamSynchronize(ctx->stream));
    *next = ctx->h_state->token;
    return device_status(ctx);
}

llama_q8_status llama_q8_generate(llama_q8_ctx* ctx, const int32_t* prompt, int32_t T, int32_t n_decode,
                                  int32_t* out_ids) {
    if (!ctx || !prompt || !out_ids || T <= 0 || n_decode < 0) return LQ8_ERR_ARG;
    if (ctx->failed) return LQ8_ERR_STATE;
    for (int i = 0; i < T; ++i)
        if (prompt[i] < 0 || prompt[i] >= ctx->cfg.n_vocab) return LQ8_ERR_TOKEN;
    if ((int64_t)T + n_decode > ctx->cfg.max_seq) return LQ8_ERR_CTX;
    LQ8_CK(ctx, cudaSetDevice(ctx->device));
    LQ8_CK(ctx, ensure_decode_graph(ctx));
    if (T == 1) {
        LQ8_CK(ctx, launch_set_state(ctx->d_state, 0, prompt[0], 0, ctx->stream));
        LQ8_CK(ctx, cudaGraphLaunch(ctx->decode_exec, ctx->stream));
        ctx->launches += 1 + ctx->decode_kernels;
    } else {
        std::memcpy(ctx->h_ids, prompt, sizeof(int32_t) * T);
        LQ8_CK(ctx, cudaMemcpyAsync(ctx->d_ids, ctx->h_ids, sizeof(int32_t) * T, cudaMemcpyHostToDevice, ctx->stream));
        LQ8_CK(ctx, launch_set_state(ctx->d_state, 0, -1, 0, ctx->stream));
        LQ8_CK(ctx, enqueue_prefill(ctx, ctx->d_ids, T, 0));
        ctx->launches += 1 + prefill_kernel_count(ctx, T);
    }
    LQ8_CK(ctx, launch_decode_steps(ctx, n_decode));
    ctx->launches += (int64_t)n_decode * ctx->decode_kernels;
    LQ8_CK(ctx, cudaMemcpyAsync(ctx->h_out, ctx->d_out_ids, sizeof(int32_t) * (n_decode + 1), cudaMemcpyDeviceToHost,
                                ctx->stream));
    LQ8_CK(ctx, cudaMemcpyAsync(ctx->h_state, ctx->d_state, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    LQ8_CK(ctx, cudaStreamSynchronize(ctx->stream));
    std::memcpy(out_ids, ctx->h_out, sizeof(int32_t) * (n_decode + 1));
    ctx->len = T + n_decode;
    return device_status(ctx);
}

llama_q8_status llama_q8_prefill_async(llama_q8_ctx* ctx, const int32_t* d_ids, int32_t T, int32_t index_pos,
                                       int32_t* d_next) {
    if (!ctx || !d_ids || !d_next || T <= 0) return LQ8_ERR_ARG;
    if (ctx->failed) return LQ8_ERR_STATE;
    llama_q8_status st = check_positions(ctx, T, index_pos);
    if (st != LQ8_OK) return st;
    LQ8_CK(ctx, cudaSetDevice(ctx->device));
    LQ8_CK(ctx, ensure_decode_graph(ctx));
    LQ8_CK(ctx, launch_set_state(ctx->d_state, index_pos, -1, 0, ctx->stream));
    if (T == 1) {
        LQ8_CK(ctx, cudaMemcpyAsync(&ctx->d_state->token, d_ids, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                    ctx->stream));
        LQ8_CK(ctx, cudaGraphLaunch(ctx->decode_exec, ctx->stream));
        ctx->launches += 1 + ctx->decode_kernels;
    } else {
        LQ8_CK(ctx, enqueue_prefill(ctx, d_ids, T, index_pos));
        ctx->launches += 1 + prefill_kernel_count(ctx, T);
    }
    LQ8_CK(ctx, cudaMemcpyAsync(d_next, ctx->d_out_ids, sizeof(int32_t), cudaMemcpyDeviceToDevice, ctx->stream));
    ctx->len = index_pos + T;
    return LQ8_OK;
}

llama_q8_status llama_q8_decode_async(llama_q8_ctx* ctx, int32_t n_steps, int32_t* d_out) {
    if (!ctx || !d_out || n_steps < 0) return LQ8_ERR_ARG;
    if (ctx->failed) return LQ8_ERR_STATE;
    if (ctx->len == 0) return LQ8_ERR_STATE;
    if ((int64_t)ctx->len + n_steps > ctx->cfg.max_seq) return LQ8_ERR_CTX;
    if (n_steps == 0) return LQ8_OK;
    LQ8_CK(ctx, cudaSetDevice(ctx->device));
    LQ8_CK(ctx, ensure_decode_graph(ctx));
    LQ8_CK(ctx, launch_set_state(ctx->d_state, -1, -1, 0, ctx->stream));
    LQ8_CK(ctx, launch_decode_steps(ctx, n_steps));
    ctx->launches += 1 + (int64_t)n_steps * ctx->decode_kernels;
    LQ8_CK(ctx, cudaMemcpyAsync(d_out, ctx->d_out_ids, sizeof(int32_t) * n_steps, cudaMemcpyDeviceToDevice,
                                ctx->stream));
    ctx->len += n_steps;
    return LQ8_OK;
}

int64_t llama_q8_launch_count(const llama_q8_ctx* ctx) { return ctx ? ctx->launches : 0; }

llama_q8_status llama_q8_profile_decode(llama_q8_ctx* ctx, int32_t n_steps, llama_q8_kernel_stat* stats,
                                        int32_t max_stats, int32_t* n_stats) {
    if (!ctx || !stats || !n_stats || n_steps <= 0 || max_stats < F_COUNT) return LQ8_ERR_ARG;
    if (ctx->failed) return LQ8_ERR_STATE;
    if (ctx->len == 0) return LQ8_ERR_STATE;
    if ((int64_t)ctx->len + n_steps > ctx->cfg.max_seq) return LQ8_ERR_CTX;
    LQ8_CK(ctx, cudaSetDevice(ctx->device));
    // the instrumented copy of the decode graph: the same launches with their stamp slots set
    const int nk = ctx->decode_kernels;
    const size_t slots = 2 * (size_t)(nk + 1);
    const size_t sbytes = slots * sizeof(unsigned long long);
    unsigned long long* d_st = nullptr;
    unsigned long long* h_st = nullptr;
    LQ8_CK(ctx, cudaMalloc(&d_st, sbytes));
    if (cudaMallocHost(&h_st, sbytes * (size_t)n_steps) != cudaSuccess) {
        cudaFree(d_st);
        return LQ8_ERR_OOM;
    }
    StepLayout layout;
    int n = 0;
    cudaGraphExec_t exec = nullptr;
    cudaError_t err = cudaStreamBeginCapture(ctx->stream, cudaStreamCaptureModeThreadLocal);
    if (err == cudaSuccess) {
        cudaError_t lerr = enqueue_decode_step(ctx, &n, &layout, d_st);
        cudaGraph_t g = nullptr;
        err = cudaStreamEndCapture(ctx->stream, &g);
        if (err == cudaSuccess) err = lerr;
        if (err == cudaSuccess && n != nk) err = cudaErrorUnknown;
        if (err == cudaSuccess) err = cudaGraphInstantiate(&exec, g, 0);
        if (g) cudaGraphDestroy(g);
    }
    if (err == cudaSuccess) err = launch_set_state(ctx->d_state, -1, -1, 0, ctx->stream);
    ctx->launches += 1;
    for (int i = 0; i < n_steps && err == cudaSuccess; ++i) {
        err = cudaMemsetAsync(d_st, 0xff, sbytes, ctx->stream);
        if (err == cudaSuccess) err = cudaGraphLaunch(exec, ctx->stream);
        if (err == cudaSuccess)
            err = cudaMemcpyAsync(h_st + (size_t)i * slots, d_st, sbytes, cudaMemcpyDeviceToHost, ctx->stream);
        ctx->launches += nk + 1;
    }
    if (err == cudaSuccess) err = cudaStreamSynchronize(ctx->stream);
    if (exec) cudaGraphExecDestroy(exec);
    cudaFree(d_st);
    if (err != cudaSuccess) {
        cudaFreeHost(h_st);
        ctx->failed = true;
        return LQ8_ERR_CUDA;
    }
    for (int f = 0; f < F_COUNT; ++f) {
        std::memset(stats[f].name, 0, sizeof(stats[f].name));
        std::strncpy(stats[f].name, kFamilyNames[f], sizeof(stats[f].name) - 1);
        stats[f].launches = 0;
        stats[f].ms = 0.0;
        stats[f].span_ms = 0.0;
        stats[f].bytes = 0.0;
    }
    // Launch k's exclusive time runs from the first return of its dependency
    // wait (its predecessor has completed) to that of launch k + 1 (it has
    // completed); its span starts at its first CTA's entry instead.
    bool complete = true;
    for (int i = 0; i < n_steps; ++i) {
        const unsigned long long* t = h_st + (size_t)i * slots;
        const double kv_len = (double)(ctx->len + i + 1);  // the step's token sits at len + i
        for (int k = 0; k < nk; ++k) {
            const unsigned long long e0 = t[2 * k], w0 = t[2 * k + 1], w1 = t[2 * k + 3];
            if (e0 == ~0ull || w0 == ~0ull || w1 == ~0ull || w1 < w0 || w1 < e0) {
                complete = false;
                continue;
            }
            const StepLayout::Rec& r = layout.recs[k];
            stats[r.family].launches += 1;
            stats[r.family].ms += (double)(w1 - w0) * 1e-6;
            stats[r.family].span_ms += (double)(w1 - e0) * 1e-6;
            stats[r.family].bytes += r.bytes + r.kv_per_pos * kv_len;
        }
    }
    cudaFreeHost(h_st);
    ctx->len += n_steps;
    if (!complete) return LQ8_ERR_STATE;
    *n_stats = F_COUNT;
    return device_status(ctx);
}

llama_q8_status llama_q8_sync(llama_q8_ctx* ctx) {
    if (!ctx) return LQ8_ERR_ARG;
    if (ctx->failed) return LQ8_ERR_STATE;
    LQ8_CK(ctx, cudaSetDevice(ctx->device));
    LQ8_CK(ctx, cudaMemcpyAsync(ctx->h_state, ctx->d_state, sizeof(DevState), cudaMemcpyDeviceToHost, ctx->stream));
    LQ8_CK(ctx, cudaStreamSynchronize(ctx->stream));
    if (ctx->h_state->err) {
        llama_q8_status st = device_status(ctx);
        if (st == LQ8_ERR_TOKEN) {
            ctx->h_state->err = 0;
            LQ8_CK(ctx, cudaMemsetAsync(&ctx->d_state->err, 0, sizeof(int32_t), ctx->stream));
            LQ8_CK(ctx, cudaStreamSynchronize(ctx->stream));
        }
        return st;
    }
    return LQ8_OK;
}

llama_q8_status llama_q8_reset(llama_q8_ctx* ctx) {
    if (!ctx) return LQ8_ERR_ARG;
    if (ctx->failed) return LQ8_ERR_STATE;
    ctx->len = 0;
    return LQ8_OK;
}

llama_q8_status llama_q8_free(llama_q8_ctx* ctx) {
    if (!ctx) return LQ8_OK;
    cudaSetDevice(ctx->device);
    if (ctx->stream) cudaStreamSynchronize(ctx->stream);
    free_ctx_memory(ctx);
    delete ctx;
    return LQ8_OK;
}

llama_q8_status llama_q8_cache_len(const llama_q8_ctx* ctx, int32_t* len) {
    if (!ctx || !len) return LQ8_ERR_ARG;
    *len = ctx->len;
    return LQ8_OK;
}

llama_q8_status llama_q8_read_kv(llama_q8_ctx* ctx, int32_t layer, int32_t pos0, int32_t n, float* k_out,
                                 float* v_out) {
    if (!ctx || !k_out || !v_out || layer < 0 || layer >= ctx->cfg.n_layer || pos0 < 0 || n <= 0)
        return LQ8_ERR_ARG;
    if (ctx->failed) return LQ8_ERR_STATE;
    if (pos0 + n > ctx->len) return LQ8_ERR_ARG;
    LQ8_CK(ctx, cudaSetDevice(ctx->device));
    const int hd = ctx->cfg.head_dim;
    for (int kh = 0; kh < ctx->cfg.n_head_kv; ++kh) {
        const size_t off = ((size_t)kh * ctx->cfg.max_seq + pos0) * hd;
        LQ8_CK(ctx, cudaMemcpyAsync(k_out + (size_t)kh * n * hd, ctx->kcache(layer) + off, sizeof(float) * n * hd,
                                    cudaMemcpyDeviceToHost, ctx->stream));
        LQ8_CK(ctx, cudaMemcpyAsync(v_out + (size_t)kh * n * hd, ctx->vcache(layer) + off, sizeof(float) * n * hd,
                                    cudaMemcpyDeviceToHost, ctx->stream));
    }
    LQ8_CK(ctx, cudaStreamSynchronize(ctx->stream));
    if (ctx->cfg.rope_style == 1) {  // K rows are stored with the NEOX pairs interleaved: undo it
        std::vector<float> row(hd);
        for (size_t r = 0; r < (size_t)ctx->cfg.n_head_kv * n; ++r) {
            float* kr = k_out + r * hd;
            for (int i = 0; i < hd / 2; ++i) {
                row[i] = kr[2 * i];
                row[i + hd / 2] = kr[2 * i + 1];
            }
            std::copy(row.begin(), row.end(), kr);
        }
    }
    return LQ8_OK;
}

void* llama_q8_stream(llama_q8_ctx* ctx) { return ctx ? (void*)ctx->stream : nullptr; }

int32_t llama_q8_rope_style_for_arch(const char* arch) {
    if (!arch) return -1;
    static const char* const kNeox[] = {"qwen", "qwen2", "falcon", "phi3", "stablelm"};
    for (const char* a : kNeox)
        if (std::strcmp(arch, a) == 0) return 1;
    return 0;
}

int32_t llama_q8_decode_kernel_count(const llama_q8_ctx* ctx) { return ctx ? ctx->decode_kernels : 0; }

// ---------------------------------------------------------------------------
// Device-level entry points
// ---------------------------------------------------------------------------

llama_q8_status llama_q8_quantize(const float* w, int64_t rows, int64_t k, void* out, void* stream) {
    if (!w || !out || rows < 0 || k <= 0 || k % 32) return LQ8_ERR_ARG;
    if (launch_quantize(w, rows, k, reinterpret_cast<uint8_t*>(out), (cudaStream_t)stream) != cudaSuccess)
        return LQ8_ERR_CUDA;
    return LQ8_OK;
}

size_t llama_q8_packed_bytes(int64_t rows, int64_t k) {
    if (rows <= 0 || k <= 0 || k % 32) return 0;
    return (size_t)packed_total_bytes(rows, k);
}

llama_q8_status llama_q8_pack(const void* q8, int64_t rows, int64_t k, void* packed, void* stream) {
    if (!q8 || !packed || rows <= 0 || k <= 0 || k % 32) return LQ8_ERR_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(packed, 0, (size_t)packed_total_bytes(rows, k), s) != cudaSuccess) return LQ8_ERR_CUDA;
    if (launch_pack(reinterpret_cast<const uint8_t*>(q8), rows, k, reinterpret_cast<uint8_t*>(packed), rows, 0, 1,
                    s) != cudaSuccess)
        return LQ8_ERR_CUDA;
    return LQ8_OK;
}

llama_q8_status llama_q8_matmul(const void* packed, int64_t rows, int64_t k, const float* x, int64_t m, float* y,
                                void* stream) {
    return llama_q8_matmul_ex(packed, rows, k, x, m, y, 0, stream);
}

llama_q8_status llama_q8_matmul_ex(const void* packed, int64_t rows, int64_t k, const float* x, int64_t m, float* y,
                                   int32_t flags, void* stream) {
    if (!packed || !x || !y || rows <= 0 || k <= 0 || k % 32 || m <= 0) return LQ8_ERR_ARG;
    if (flags & ~(LQ8_MATMUL_EARLY_WEIGHTS | LQ8_MATMUL_TENSOR_CORES | LQ8_MATMUL_CUDA_CORES)) return LQ8_ERR_ARG;
    if ((flags & LQ8_MATMUL_TENSOR_CORES) && (flags & LQ8_MATMUL_CUDA_CORES)) return LQ8_ERR_ARG;
    const int path = (flags & LQ8_MATMUL_TENSOR_CORES) ? MATMUL_TENSOR_CORES
                     : (flags & LQ8_MATMUL_CUDA_CORES) ? MATMUL_CUDA_CORES : MATMUL_AUTO;
    // W and x are fetched by bulk and tensor copies: 16-byte aligned only
    if (((uintptr_t)packed | (uintptr_t)x) & 15) return LQ8_ERR_ARG;
    const bool early = (flags & LQ8_MATMUL_EARLY_WEIGHTS) != 0;
    if (rows > (1 << 30) || m > (1 << 30)) return LQ8_ERR_UNSUPPORTED;
    if (ensure_kernel_attributes() != cudaSuccess) return LQ8_ERR_CUDA;
    PackedQ8 W = packed_view(reinterpret_cast<const uint8_t*>(packed), rows, k);
    EpiArgs e;
    e.y = y;
    e.ldy = (int)rows;
    cudaError_t err;
    if (m == 1) {
        if ((size_t)k > gemv_max_k()) return LQ8_ERR_UNSUPPORTED;
        err = launch_gemv(W, x, nullptr, 0.f, EPI_STORE, e, early, nullptr, (cudaStream_t)stream);
    } else {
        const bool tc = matmul_on_tensor_cores((int)m, (int)rows, (int)k, path);
        if (!tc && !gemv_rows_fits(m, k)) return LQ8_ERR_UNSUPPORTED;
        // tensor cores: the rows' largest |x| and the scaled, split rows, in
        // stream-ordered scratch (one allocation: m floats, then m x 2k halves)
        SplitRows sp;
        void* scratch = nullptr;
        const size_t rm_bytes = ((size_t)m * sizeof(float) + 255) / 256 * 256;
        if (tc) {
            if (cudaMallocAsync(&scratch, rm_bytes + (size_t)m * 2 * (size_t)k * sizeof(__half),
                                (cudaStream_t)stream) != cudaSuccess)
                return LQ8_ERR_OOM;
            sp.rowmax = reinterpret_cast<float*>(scratch);
            sp.hl = reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(scratch) + rm_bytes);
        }
        err = launch_matmul_rows(W, x, (int)m, (int)k, EPI_STORE, e, early, nullptr, (cudaStream_t)stream, sp, path);
        if (scratch) {
            const cudaError_t ferr = cudaFreeAsync(scratch, (cudaStream_t)stream);
            if (err == cudaSuccess) err = ferr;
        }
    }
    return err == cudaSuccess ? LQ8_OK : LQ8_ERR_CUDA;
}

size_t llama_q8_packed_bytes_fmt(int32_t gguf_type, int64_t rows, int64_t k) {
    if (gguf_type == kGgufQ8_0) return llama_q8_packed_bytes(rows, k);
    if (!fmt_supported(gguf_type) || rows <= 0 || k <= 0 || k % fmt_block_weights(gguf_type)) return 0;
    return (size_t)fmt_packed_bytes(gguf_type, rows, k);
}

llama_q8_status llama_q8_pack_fmt(int32_t gguf_type, const void* blocks, int64_t rows, int64_t k, void* packed,
                                  void* stream) {
    if (gguf_type == kGgufQ8_0) return llama_q8_pack(blocks, rows, k, packed, stream);
    if (!blocks || !packed || rows <= 0 || k <= 0) return LQ8_ERR_ARG;
    if (!fmt_supported(gguf_type)) return LQ8_ERR_UNSUPPORTED;
    if (k % fmt_block_weights(gguf_type)) return LQ8_ERR_ARG;
    if (rows > (1 << 30) || k > (1 << 30)) return LQ8_ERR_UNSUPPORTED;
    return launch_pack_fmt(gguf_type, reinterpret_cast<const uint8_t*>(blocks), rows, k,
                           reinterpret_cast<uint8_t*>(packed), (cudaStream_t)stream) == cudaSuccess
               ? LQ8_OK
               : LQ8_ERR_CUDA;
}

llama_q8_status llama_q8_matvec_fmt(int32_t gguf_type, const void* packed, int64_t rows, int64_t k, const float* x,
                                    float* y, int32_t flags, void* stream) {
    if (gguf_type == kGgufQ8_0) return llama_q8_matmul_ex(packed, rows, k, x, 1, y, flags, stream);
    if (!packed || !x || !y || rows <= 0 || k <= 0) return LQ8_ERR_ARG;
    if (!fmt_supported(gguf_type)) return LQ8_ERR_UNSUPPORTED;
    if (k % fmt_block_weights(gguf_type)) return LQ8_ERR_ARG;
    if (flags & ~LQ8_MATMUL_EARLY_WEIGHTS) return LQ8_ERR_ARG;
    // records and x are fetched by bulk async copies: 16-byte aligned only
    if (((uintptr_t)packed | (uintptr_t)x) & 15) return LQ8_ERR_ARG;
    if (rows > (1 << 30) || k > fmt_max_k(gguf_type)) return LQ8_ERR_UNSUPPORTED;
    if (ensure_kernel_attributes() != cudaSuccess) return LQ8_ERR_CUDA;
    const bool early = (flags & LQ8_MATMUL_EARLY_WEIGHTS) != 0;
    return launch_gemv_fmt(gguf_type, reinterpret_cast<const uint8_t*>(packed), (int)rows, (int)k, x, y, early,
                           nullptr, (cudaStream_t)stream) == cudaSuccess
               ? LQ8_OK
               : LQ8_ERR_CUDA;
}

llama_q8_status llama_q8_attention_decode(const float* q, const float* k_cache, const float* v_cache, int32_t kv_len,
                                         int32_t n_head, int32_t n_head_kv, int32_t head_dim, int32_t cache_stride,
                                         float* out, void* stream) {
    if (!q || !k_cache || !v_cache || !out || kv_len <= 0 || n_head <= 0 || n_head_kv <= 0 ||
        n_head % n_head_kv || cache_stride <= 0)
        return LQ8_ERR_ARG;
    if (kv_len > cache_stride) return LQ8_ERR_CTX;
    if (head_dim != 64 && head_dim != 128) return LQ8_ERR_UNSUPPORTED;
    if (n_head / n_head_kv > 8) return LQ8_ERR_UNSUPPORTED;
    // K/V rows and q are fetched by bulk async copies or 16-byte loads: 16-byte aligned buffers only
    if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)out) & 15) return LQ8_ERR_ARG;
    if (ensure_kernel_attributes() != cudaSuccess) return LQ8_ERR_CUDA;
    cudaError_t err = launch_attn_decode_cluster(q, k_cache, v_cache, n_head, n_head_kv, head_dim, cache_stride,
                                                 kv_len, nullptr, out, false, nullptr, (cudaStream_t)stream);
    return err == cudaSuccess ? LQ8_OK : LQ8_ERR_CUDA;
}

size_t llama_q8_attention_workspace_bytes(int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                                          int32_t cache_stride) {
    if (n_head <= 0 || n_head_kv <= 0 || n_head % n_head_kv || head_dim <= 0 || cache_stride <= 0) return 0;
    return attn_workspace_bytes(n_head, n_head_kv, head_dim, cache_stride);
}

llama_q8_status llama_q8_attention(const float* q, const float* k_cache, const float* v_cache, int32_t T,
                                   int32_t index_pos, int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                                   int32_t cache_stride, float* out, void* workspace, size_t workspace_bytes,
                                   void* stream) {
    if (!q || !k_cache || !v_cache || !out || T <= 0 || index_pos < 0 || n_head <= 0 || n_head_kv <= 0 ||
        n_head % n_head_kv || cache_stride <= 0)
        return LQ8_ERR_ARG;
    if ((int64_t)index_pos + T > cache_stride) return LQ8_ERR_CTX;
    if (head_dim != 64 && head_dim != 128) return LQ8_ERR_UNSUPPORTED;
    if (n_head / n_head_kv > 8) return LQ8_ERR_UNSUPPORTED;
    // q, K/V rows and outputs move in 16-byte pieces: 16-byte aligned buffers only
    if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)out) & 15) return LQ8_ERR_ARG;
    if (ensure_kernel_attributes() != cudaSuccess) return LQ8_ERR_CUDA;
    cudaError_t err;
    if (T == 1) {
        if (!workspace || workspace_bytes < attn_workspace_bytes(n_head, n_head_kv, head_dim, cache_stride))
            return LQ8_ERR_ARG;
        err = launch_attn_decode(q, k_cache, v_cache, n_head, n_head_kv, head_dim, cache_stride, index_pos + 1,
                                 nullptr, out, workspace, false, (cudaStream_t)stream);
    } else {
        err = launch_attn_prefill(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, head_dim, cache_stride, out,
                                  false, (cudaStream_t)stream);
    }
    return err == cudaSuccess ? LQ8_OK : LQ8_ERR_CUDA;
}

}  // extern "C"
