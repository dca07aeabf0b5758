// Internal interface between the runtime (runtime.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <utility>

#include "common.cuh"

namespace lq8 {

// Device-resident step state. The decode step reads pos and token from here,
// so one captured CUDA graph serves every decode position; the lm_head
// epilogue writes the greedy token back and advances pos.
struct DevState {
    int32_t pos;    // position of the token being processed (decode)
    int32_t token;  // token the next decode step embeds
    int32_t n_out;  // tokens written to out_ids so far
    int32_t err;    // 0, or a llama_q8_status raised on the device
};

enum Epi : int {
    EPI_STORE = 0,     // y[t][n] = acc
    EPI_RESIDUAL = 1,  // y[t][n] += acc            (O-proj, down-proj)
    EPI_QKV = 2,       // rope_i on q/k rows, q -> q_out, k/v -> KV cache at pos
    EPI_SILU = 3,      // rows interleaved gate/up: a[t][n/2] = silu(g) * u
    EPI_ARGMAX = 4     // logits[n] = acc; greedy token -> state / out_ids
};

struct EpiArgs {
    float* y = nullptr;  // STORE / RESIDUAL output, row stride ldy
    int ldy = 0;
    const float* res = nullptr;  // RESIDUAL (matrix-vector only): y = res + acc instead of y += acc
    // QKV
    float* q_out = nullptr;  // [m][q_rows]
    float* k_cache = nullptr;  // layer base, [n_head_kv][max_seq][head_dim]
    float* v_cache = nullptr;
    int q_rows = 0, kv_rows = 0, head_dim = 0, max_seq = 0;
    const float* rope_cos = nullptr;  // [max_seq][head_dim/2]
    const float* rope_sin = nullptr;
    int pos0 = 0;                     // position of the first token (when state == nullptr)
    const DevState* state = nullptr;  // decode: position read from the device
    // SILU
    float* a_out = nullptr;
    int lda = 0;
    // ARGMAX
    float* logits = nullptr;
    unsigned long long* best_key = nullptr;  // zero between launches
    unsigned int* done_count = nullptr;      // zero between launches
    DevState* st = nullptr;
    int32_t* out_ids = nullptr;
    int pos_after = -1;  // >= 0: state->pos := pos_after; < 0: state->pos += 1
    // matrix-vector kernel: timeline stamps of this launch (instrumented decode graph), or null
    unsigned long long* stamp = nullptr;
};

// Launch with an optional programmatic-dependent-launch attribute (the kernel
// may start before its predecessor finishes and waits for it with
// griddepcontrol.wait). Used inside the model's own launch sequences only;
// device-level entry points launch plainly because a caller's preceding
// kernel may have written any of their inputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_ex(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                      Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// quant.cu
cudaError_t launch_quantize(const float* w, int64_t rows, int64_t k, uint8_t* out, cudaStream_t s);
cudaError_t launch_pack(const uint8_t* q8, int64_t rows, int64_t k, uint8_t* packed_base,
                        int64_t dst_rows, int64_t row_offset, int64_t row_stride, cudaStream_t s);
cudaError_t launch_embed(const PackedQ8& E, const int32_t* ids, int T, const DevState* st_token,
                         DevState* st_err, float* x, int n_vocab, bool pdl, cudaStream_t s,
                         unsigned long long* stamp = nullptr);
// One 32-thread CTA that stamps its entry and the return of its grid dependency
// wait: placed after the last kernel of the instrumented decode graph, its wait
// returns when that kernel has completed.
cudaError_t launch_stamp(unsigned long long* stamp, cudaStream_t s);
// The operand of a tensor-core product of m token rows of k activations (the
// row scaling and hi / lo split of common.cuh): rowmax[m] holds each row's
// largest |x| (the product's epilogue undoes the row's scale from it), hl[m][2k]
// the split rows.
struct SplitRows {
    float* rowmax = nullptr;
    __half* hl = nullptr;
};
// y = RMSNorm rows of x (written when y is non-null); with split, also the
// tensor-core operand of y (split->rowmax and split->hl)
cudaError_t launch_rmsnorm(const float* x, const float* g, float eps, int m, int k, float* y, bool pdl,
                           cudaStream_t s, const SplitRows* split = nullptr);
cudaError_t launch_set_state(DevState* st, int pos, int token, int n_out, cudaStream_t s);
cudaError_t launch_wait_timeout(int* err, int code, cudaStream_t s);  // bounded-wait self-test

// gemv.cu (m == 1)
// With the fused RMSNorm, the input may first be the sum x + part[0] + ... +
// part[n_part - 1] (partials of the preceding kernel, each k floats, stride
// part_stride), taken in that order; the first CTA stores that sum to
// x_sum_out for the residual of a later kernel.
struct GemvPreSum {
    const float* part = nullptr;
    int n_part = 0;
    int part_stride = 0;
    float* x_sum_out = nullptr;
};
// force_splits: 0 = automatic (persistent row-parallel CTAs when the row tiles
// fill the GPU, else the block range of each tile split over a cluster);
// 2..8 = split every tile's block range over a cluster of that many CTAs.
cudaError_t launch_gemv(const PackedQ8& W, const float* x, const float* norm_g, float eps, int epi,
                        const EpiArgs& e, bool pdl, int* err, cudaStream_t s, const GemvPreSum* pre = nullptr,
                        int force_splits = 0);
size_t gemv_max_k();
// gemv_formats.cu: the matrix-vector product for other GGUF block formats
// (GGUF type ids), on the library's repacked layout of each.
constexpr int kGgufQ5_0 = 6, kGgufQ8_0 = 8, kGgufQ4_K = 12, kGgufQ6_K = 14;
bool fmt_supported(int type);                        // Q5_0, Q4_K, Q6_K
int fmt_block_weights(int type);                     // 32 or 256
int64_t fmt_packed_bytes(int type, int64_t rows, int64_t k);
int64_t fmt_max_k(int type);
cudaError_t launch_pack_fmt(int type, const uint8_t* src, int64_t rows, int64_t k, uint8_t* dst, cudaStream_t s);
cudaError_t launch_gemv_fmt(int type, const uint8_t* packed, int rows, int k, const float* x, float* y, bool pdl,
                            int* err, cudaStream_t s);
cudaError_t init_gemv_fmt_attributes();
// gemv.cu, m >= 2 token rows on the CUDA cores, in chunks of 16: each weight
// tile streamed once per chunk for all of its rows
cudaError_t launch_gemv_rows(const PackedQ8& W, const float* X, int m, int ldx, int epi, const EpiArgs& e, bool pdl,
                             int* err, cudaStream_t s);
bool gemv_rows_fits(int64_t m, int64_t k);  // a chunk's x slices fit beside the ring (at most 8 splits)
// gemm_tc.cu: tcgen05 kernel for many rows (f16 products of the codes and of
// each token's activations scaled by a power of two and split into hi and lo).
// split: device memory for the operand of X (m floats, m x 2k halves): filled
// from X by a pass launched just before the product, or (split_ready) already
// written by the kernel that produced X, in which case X is not read.
cudaError_t launch_gemm_tc(const PackedQ8& W, const float* X, int m, int ldx, int epi, const EpiArgs& e, bool pdl,
                           int* err, cudaStream_t s, const SplitRows& split, bool split_ready = false);
cudaError_t init_gemm_tc_attributes();
// Every kernel's attributes on the current device, once per device (runtime.cu).
cudaError_t ensure_kernel_attributes();
// Which kernel takes a product of m > 1 token rows: the tensor cores above 16
// rows, the CUDA-core rows kernel up to 16 (either can be forced). Measured on
// the 135M prefill shapes at 203 rows, the tensor cores win even there, where
// their start-up dominates: 14.5-20.6 us against 33-88 us for the rows kernel
// in 16-row chunks.
constexpr int kTensorCoreMinRows = 16;
enum MatmulPath : int { MATMUL_AUTO = 0, MATMUL_TENSOR_CORES = 1, MATMUL_CUDA_CORES = 2 };
inline bool matmul_on_tensor_cores(int m, int rows, int k, int path) {
    (void)rows;
    (void)k;
    if (path == MATMUL_TENSOR_CORES) return true;
    if (path == MATMUL_CUDA_CORES) return false;
    return m > kTensorCoreMinRows;
}
// split / split_ready: the tensor-core operand (launch_gemm_tc); the CUDA-core
// kernel reads X and ignores them
inline cudaError_t launch_matmul_rows(const PackedQ8& W, const float* X, int m, int ldx, int epi, const EpiArgs& e,
                                      bool pdl, int* err, cudaStream_t s, const SplitRows& split,
                                      int path = MATMUL_AUTO, bool split_ready = false) {
    return matmul_on_tensor_cores(m, W.rows, W.k, path)
               ? launch_gemm_tc(W, X, m, ldx, epi, e, pdl, err, s, split, split_ready)
               : launch_gemv_rows(W, X, m, ldx, epi, e, pdl, err, s);
}

// attention.cu
size_t attn_workspace_bytes(int n_head, int n_head_kv, int head_dim, int max_seq);
cudaError_t launch_attn_decode(const float* q, const float* k_cache, const float* v_cache,
                               int n_head, int n_head_kv, int head_dim, int cache_stride,
                               int kv_len, const DevState* st, float* out, void* workspace,
                               bool pdl, cudaStream_t s);
cudaError_t launch_attn_decode_cluster(const float* q, const float* k_cache, const float* v_cache, int n_head,
                                       int n_head_kv, int head_dim, int cache_stride, int kv_len,
                                       const DevState* st, float* out, bool pdl, int* err, cudaStream_t s,
                                       unsigned long long* stamp = nullptr);
// Decode attention whose clusters also apply the O projection: cluster kh
// writes part[kh][0..rows) = W_o[:, columns of its query heads] o, the n_kv
// partials summing to W_o o (added to the residual by the next kernel).
// supported() is false when the model's W_o does not fit the kernel.
bool attn_oproj_fused_supported(int n_head, int n_kv, int head_dim, const PackedQ8& Wo);
// The front half of a decode layer (RMSNorm, the Q/K/V rows of each KV head,
// rope_i, KV append, attention, W_o column slice -> part) as one kernel with a
// cluster per KV head, for models whose per-head projections are small.
struct FrontArgs {
    const float* x;        // [h] residual stream base (written by the preceding kernel)
    const float* xparts;   // [n_xparts][h] partials added to x in order (the MLP's clusters), or null
    int n_xparts;
    float* x_store;        // [h] where the first CTA keeps x + partials (the MLP's input), or null
    const float* g;        // [h] attention RMSNorm weight
    float eps;
    PackedQ8 wqkv;         // [Wq;Wk;Wv]
    PackedQ8 wo;
    float* kc;             // layer K cache [n_kv][stride][hd]
    float* vc;
    const float* rope_cos; // [stride][hd/2]
    const float* rope_sin;
    int n_head, n_kv, stride;
    const DevState* st;
    float scale;
    float* part;           // [n_kv][part_stride] partials of W_o o
    int part_stride;
    int* err;
    unsigned long long* stamp;  // timeline stamps (instrumented decode graph), or null
};
int layer_front_cluster_size(const FrontArgs& fa, int head_dim);  // 0: not supported

// mlp.cu: the MLP half of a decode layer as one kernel (clusters of 8 CTAs).
struct MlpArgs {
    const float* x;          // [h] residual stream before the attention output is added
    const float* attn_part;  // [n_attn_part][h] partials of W_o o (added in order)
    int n_attn_part;
    const float* g;          // [h] FFN RMSNorm weight
    float eps;
    PackedQ8 wgu;            // row-interleaved [W_g;W_u]
    PackedQ8 wdown;
    float* xr_out;           // [h] x + W_o o (written by the first CTA): the next residual base
    float* mlp_part;         // [clusters][h] partials of W_down a, one per cluster
    int* err;
    unsigned long long* stamp;  // timeline stamps (instrumented decode graph), or null
};
int decode_mlp_clusters(int h, int ff, int gu_rows);  // 0: not supported
cudaError_t launch_decode_mlp(const MlpArgs& ma, bool pdl, cudaStream_t s);
cudaError_t launch_layer_front(const FrontArgs& fa, int head_dim, int cl, bool pdl, cudaStream_t s);
cudaError_t launch_attn_oproj(const float* q, const float* k_cache, const float* v_cache, int n_head, int n_head_kv,
                              int head_dim, int cache_stride, const DevState* st, const PackedQ8& Wo, float* part,
                              int part_stride, bool pdl, int* err, cudaStream_t s,
                              unsigned long long* stamp = nullptr);
cudaError_t launch_attn_prefill(const float* q, const float* k_cache, const float* v_cache,
                                int T, int index_pos, int n_head, int n_head_kv, int head_dim,
                                int cache_stride, float* out, bool pdl, cudaStream_t s);

PackedQ8 packed_view(const uint8_t* base, int64_t rows, int64_t k);

}  // namespace lq8
