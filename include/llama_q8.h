/*
 * llama_q8.h — C ABI of the GB300 (sm_103a) Q8_0 Llama forward.
 *
 * One forward pass of a Q8_0-quantised Llama, as described on the candle
 * 0.11.0 documentation pages "量化 llama 的一次前向" (quantized-llama),
 * "生成一个 token" (one-token) and "速度" (speed):
 *   - ModelWeights::from_gguf keeps the projections in Q8_0, dequantises the
 *     embedding, and uses the embedding as the output head when the file has
 *     no output.weight ("生成一个 token", section 建模型：按名字取张量);
 *   - forward(ids, index_pos) returns logits for the last position only,
 *     builds a causal mask only when T > 1, drops the KV cache when
 *     index_pos == 0 and appends to it otherwise ("量化 llama 的一次前向",
 *     sections forward：mask 什么时候建 and forward_attn：自己拼 KV);
 *   - the rotary table holds 4096 positions and index_pos + T > 4096 is an
 *     error (same page, section from_gguf：键名写死了 llama.);
 *   - clear_kv_cache drops the cache (same page, section 换 prompt 要不要
 *     clear_kv_cache).
 *
 * Conventions for every call:
 *   - Every call returns a llama_q8_status. On any error nothing is launched
 *     and the context state (cached length, KV cache) is unchanged, except
 *     LQ8_ERR_CUDA, after which the context only accepts llama_q8_free.
 *   - "host" pointers are ordinary or pinned CPU memory; "device" pointers
 *     are CUDA device memory on the context's device. The caller owns every
 *     pointer it passes; the library copies what it needs and keeps no
 *     caller pointer after a call returns.
 *   - Model calls run on the context's own CUDA stream and are synchronous
 *     unless the name ends in _async (those enqueue and return).
 *   - Batch size is 1 (the pages' forward ignores the batch dimension).
 *   - Activations, the KV cache and logits are f32; weights are Q8_0.
 *   - All kernels are written for sm_103a; there is no CPU fallback. A call
 *     on a machine without such a GPU returns LQ8_ERR_CUDA.
 */
#ifndef LLAMA_Q8_H
#define LLAMA_Q8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum llama_q8_status {
    LQ8_OK = 0,
    LQ8_ERR_ARG = 1,         /* NULL pointer, non-positive size, inconsistent config */
    LQ8_ERR_POS = 2,         /* index_pos is neither 0 nor the number of cached positions */
    LQ8_ERR_CTX = 3,         /* index_pos + T exceeds max_seq (4096 on the pages) */
    LQ8_ERR_TOKEN = 4,       /* a token id outside [0, n_vocab) */
    LQ8_ERR_CUDA = 5,        /* a CUDA runtime call or a kernel launch failed */
    LQ8_ERR_OOM = 6,         /* device or pinned-host allocation failed */
    LQ8_ERR_STATE = 7,       /* context already failed, or call order violated */
    LQ8_ERR_UNSUPPORTED = 8, /* shape outside what the kernels implement */
    LQ8_ERR_FORMAT = 9       /* GGUF file unreadable, not GGUF, or missing a key or tensor */
} llama_q8_status;

/* Q8_0 block: 32 consecutive weights of one row along the input dimension,
 * stored as an IEEE fp16 scale d (little-endian) followed by 32 int8 codes,
 * 34 bytes; w = d * q. A [rows, k] matrix is rows * (k / 32) blocks, row-major.
 * The pages fix the 34-bytes-per-32-weights size through the GGUF byte counts
 * ("生成一个 token", 实验程序 and 读 GGUF; "速度", CPU GGUF). */
#define LLAMA_Q8_BLOCK 32
#define LLAMA_Q8_BLOCK_BYTES 34

typedef struct llama_q8_config {
    int32_t n_layer;      /* llama.block_count, 30 for the 135M model */
    int32_t n_embd;       /* llama.embedding_length (hidden), multiple of 32 */
    int32_t n_head;       /* llama.attention.head_count */
    int32_t n_head_kv;    /* llama.attention.head_count_kv; n_head % n_head_kv == 0, ratio <= 8 */
    int32_t head_dim;     /* 64 or 128 */
    int32_t n_ff;         /* llama.feed_forward_length, multiple of 32 */
    int32_t n_vocab;
    int32_t max_seq;      /* rotary table rows and KV capacity; the pages use 4096 */
    float rms_eps;        /* 1e-5 */
    float rope_theta;     /* 10000 */
    int32_t tied_output;  /* 1: the head is token_embd (no output.weight) */
    int32_t decode_kernel; /* decode step: 0 = automatic (two kernels per layer when each KV
                              head's Q/K/V rows and W_o slice fit a cluster and the MLP fits
                              16-CTA clusters, else three, four or five), 1 = five per-layer
                              kernels, 3 = four per layer (attention applying W_o), 4 = three
                              per layer (norm, Q/K/V, attention and W_o fused; gate/up; down);
                              3-4 give LQ8_ERR_UNSUPPORTED at load when the model does not
                              fit; 2 and 5 (one cluster kernel for the whole step / per layer)
                              are not built (measured slower): LQ8_ERR_UNSUPPORTED */
    int32_t rope_style;   /* 0: rope_i, dims 2i and 2i+1 form a pair (the Llama convention);
                             1: NEOX, dim i pairs with dim i + head_dim/2; both at angle
                             p * theta^(-2i/head_dim) ("量化 llama 的一次前向", RoPE：两种约定，
                             按架构名选). Other values -> LQ8_ERR_ARG */
    int32_t head_splits;  /* lm_head matrix-vector product of the decode step and of the
                             prefill's last row: 0 = row-parallel (persistent CTAs, each
                             taking whole 32-row tiles over the full n_embd); 2..8 = split-K,
                             each tile's n_embd range split over a cluster of that many CTAs
                             whose partial sums meet in distributed shared memory. Other
                             values, or more splits than n_embd / 32, -> LQ8_ERR_ARG */
} llama_q8_config;

/* The rotary convention the pages' loader picks from general.architecture:
 * 1 (NEOX) for the architectures it lists, 0 (rope_i) for any other name, -1
 * for NULL. The pages print five names of that list (qwen, qwen2, falcon,
 * phi3, stablelm) and say it has about twenty; this function knows the five
 * printed ones, and a file of another listed architecture sets rope_style
 * itself. */
int32_t llama_q8_rope_style_for_arch(const char* general_architecture);

typedef struct llama_q8_layer_weights {
    const float* attn_norm;   /* [n_embd] f32 */
    const float* ffn_norm;    /* [n_embd] f32 */
    const void* attn_q;       /* Q8_0 [n_head*head_dim, n_embd] */
    const void* attn_k;       /* Q8_0 [n_head_kv*head_dim, n_embd] */
    const void* attn_v;       /* Q8_0 [n_head_kv*head_dim, n_embd] */
    const void* attn_output;  /* Q8_0 [n_embd, n_head*head_dim] */
    const void* ffn_gate;     /* Q8_0 [n_ff, n_embd] */
    const void* ffn_up;       /* Q8_0 [n_ff, n_embd] */
    const void* ffn_down;     /* Q8_0 [n_embd, n_ff] */
} llama_q8_layer_weights;

typedef struct llama_q8_weights {
    const void* token_embd;    /* Q8_0 [n_vocab, n_embd] */
    const float* output_norm;  /* [n_embd] f32 */
    const void* output;        /* Q8_0 [n_vocab, n_embd]; NULL when tied_output */
    const llama_q8_layer_weights* layers;  /* host array of n_layer entries */
    int32_t on_device;         /* 0: tensor pointers are host memory; 1: device memory */
} llama_q8_weights;

typedef struct llama_q8_ctx llama_q8_ctx;

/* Build a context on CUDA device `device`: copy and repack every tensor into
 * the library's device layout (with rope_style 1, each head's Q and K rows
 * are stored interleaved — row i and row i + head_dim/2 side by side — so the
 * NEOX pairs become adjacent and the same fused rotation serves both
 * conventions; attention scores are unchanged because q and k share the
 * permutation, and llama_q8_read_kv returns K in the natural order), build
 * the rotary cos/sin table
 * [max_seq, head_dim/2] (angle p * theta^(-2i/head_dim), computed in double,
 * stored f32), allocate the KV cache [n_layer][n_head_kv][max_seq][head_dim]
 * for K and for V, and create the context's stream. `*out` receives the
 * context, owned by the caller until llama_q8_free. Errors: LQ8_ERR_ARG,
 * LQ8_ERR_UNSUPPORTED, LQ8_ERR_OOM, LQ8_ERR_CUDA ("量化 llama 的一次前向",
 * from_gguf). */
llama_q8_status llama_q8_load(const llama_q8_config* cfg, const llama_q8_weights* w,
                              int32_t device, llama_q8_ctx** out);

/* from_gguf: read a GGUF file's header ("生成一个 token", 读 GGUF: magic,
 * version, metadata key/values, tensor directory; the weights are not read)
 * and fill *cfg the way the pages' loader does ("量化 llama 的一次前向",
 * from_gguf：键名写死了 llama.): n_layer = llama.block_count, n_embd =
 * llama.embedding_length, n_head = llama.attention.head_count, n_head_kv =
 * llama.attention.head_count_kv (head_count when absent), head_dim = n_embd /
 * n_head, n_ff = llama.feed_forward_length, n_vocab = token_embd.weight's row
 * count, max_seq = 4096, rms_eps = llama.attention.layer_norm_rms_epsilon
 * (1e-5 when absent), rope_theta = llama.rope.freq_base (10000 when absent),
 * tied_output = no output.weight in the file, rope_style from
 * general.architecture (llama_q8_rope_style_for_arch), decode_kernel 0. Every
 * tensor the model needs is checked: present under its GGUF name
 * (token_embd.weight, output_norm.weight, output.weight optional,
 * blk.{i}.attn_norm / ffn_norm / attn_q / attn_k / attn_v / attn_output /
 * ffn_gate / ffn_up / ffn_down .weight), Q8_0 for matrices and F32 for norms
 * (LQ8_ERR_UNSUPPORTED otherwise), with the extents the hyperparameters give
 * and inside the file. n_tensors and data_offset (either may be NULL) receive
 * the directory's size and where the data region starts. No GPU is used.
 * Errors: LQ8_ERR_ARG (NULL path or cfg), LQ8_ERR_FORMAT (unreadable, not
 * GGUF v2/v3, a missing llama.* key, a missing or malformed tensor),
 * LQ8_ERR_UNSUPPORTED. */
llama_q8_status llama_q8_gguf_config(const char* path, llama_q8_config* cfg, int64_t* n_tensors,
                                     int64_t* data_offset);

/* llama_q8_gguf_config, then llama_q8_load of the file's tensors (mapped
 * read-only, copied to device `device` and unmapped before returning) with
 * the given decode_kernel. */
llama_q8_status llama_q8_load_gguf(const char* path, int32_t device, int32_t decode_kernel,
                                   llama_q8_ctx** out);

/* forward(ids, index_pos): run T tokens (host ids[T]) starting at position
 * index_pos and write the f32 logits of the LAST position to host
 * logits[n_vocab]. index_pos == 0 drops the cache first; otherwise index_pos
 * must equal the number of cached positions (LQ8_ERR_POS) — a deliberate
 * tightening of the pages, where a wrong index_pos is silent when T == 1
 * ("量化 llama 的一次前向", index_pos 传错). index_pos + T > max_seq gives
 * LQ8_ERR_CTX; T <= 0 gives LQ8_ERR_ARG; an id outside [0, n_vocab) gives
 * LQ8_ERR_TOKEN. Checked in that order: ARG, TOKEN, CTX, POS. T == 1 runs
 * the captured CUDA-graph decode step; T > 1 runs the prefill kernels with
 * the causal mask. */
llama_q8_status llama_q8_forward(llama_q8_ctx* ctx, const int32_t* ids, int32_t T,
                                 int32_t index_pos, float* logits);

/* As llama_q8_forward, but returns only the greedy next token (argmax of the
 * last position's logits, lowest index on ties) in host *next. */
llama_q8_status llama_q8_forward_argmax(llama_q8_ctx* ctx, const int32_t* ids, int32_t T,
                                        int32_t index_pos, int32_t* next);

/* The generation loop of "生成一个 token" (实验程序): prefill the host
 * prompt[T] at position 0, then n_decode greedy decode steps, each feeding
 * back the previous token. out_ids (host, n_decode + 1 entries) receives the
 * token chosen by the prefill followed by one token per decode step. The
 * decode steps replay the captured decode graphs back to back (one of eight
 * steps while they fit, whose launches chain across the steps, then single
 * steps) with the token fed back on
 * the device; the host reads the tokens once at the end. Requires
 * T + n_decode <= max_seq (LQ8_ERR_CTX). */
llama_q8_status llama_q8_generate(llama_q8_ctx* ctx, const int32_t* prompt, int32_t T,
                                  int32_t n_decode, int32_t* out_ids);

/* Device-resident variants for callers that keep ids on the GPU. They enqueue
 * on the context's stream and return at once; llama_q8_sync waits.
 * prefill_async: device d_ids[T] at index_pos (same position rules as
 * llama_q8_forward, checked on the host); writes the greedy token to device
 * *d_next and keeps it as the token the next decode step consumes.
 * decode_async: n_steps decode steps starting from that token; device
 * d_out[n_steps] receives one token per step. Ids in device memory are not
 * seen by the host: an out-of-range id is clamped to 0 by the embedding
 * kernel and reported as LQ8_ERR_TOKEN by the next llama_q8_sync. */
llama_q8_status llama_q8_prefill_async(llama_q8_ctx* ctx, const int32_t* d_ids, int32_t T,
                                       int32_t index_pos, int32_t* d_next);
llama_q8_status llama_q8_decode_async(llama_q8_ctx* ctx, int32_t n_steps, int32_t* d_out);
llama_q8_status llama_q8_sync(llama_q8_ctx* ctx);

/* clear_kv_cache: cached length := 0. Frees nothing (the cache is
 * preallocated); the next forward must use index_pos 0. */
llama_q8_status llama_q8_reset(llama_q8_ctx* ctx);

/* Release every device and host resource of ctx. NULL is accepted. */
llama_q8_status llama_q8_free(llama_q8_ctx* ctx);

/* Number of cached positions (the value index_pos must take next). */
llama_q8_status llama_q8_cache_len(const llama_q8_ctx* ctx, int32_t* len);

/* Copy cached K and V rows [pos0, pos0 + n) of one layer to host buffers
 * k_out, v_out, each [n_head_kv][n][head_dim] f32 (K is stored after RoPE).
 * Requires pos0 + n <= cached length. */
llama_q8_status llama_q8_read_kv(llama_q8_ctx* ctx, int32_t layer, int32_t pos0, int32_t n,
                                 float* k_out, float* v_out);

/* The context's CUDA stream (a cudaStream_t), for recording events around
 * the _async calls. */
void* llama_q8_stream(llama_q8_ctx* ctx);

/* Number of kernel launches one decode step makes (the CUDA-graph nodes):
 * n_layer * {5, 4, 3, 2} + 2 (embedding, per-layer kernels, lm_head + argmax;
 * see decode_kernel). */
int32_t llama_q8_decode_kernel_count(const llama_q8_ctx* ctx);

/* Cumulative number of kernel launches this context has issued; a CUDA-graph
 * decode step counts as its llama_q8_decode_kernel_count() kernels. */
int64_t llama_q8_launch_count(const llama_q8_ctx* ctx);

/* Per-kernel timeline of the decode step, in the spirit of the per-span self
 * times on "量化 llama 的一次前向" (一个 decode 步里时间去了哪). Replays an
 * instrumented copy of the CUDA-graph decode step n_steps times (greedy
 * decode, continuing from the current cached length and advancing it like
 * llama_q8_decode_async): the same kernels, launch order and programmatic
 * dependent launches as the step llama_q8_decode_async replays, each launch
 * also recording on the GPU's global nanosecond timer when its first CTA
 * started and when its grid dependency wait first returned (that is, when the
 * previous launch had completed); a one-CTA stamp kernel after the lm_head
 * closes the step. Per kernel family: launches; ms = summed exclusive time
 * (from the return of the launch's dependency wait to that of the next
 * launch: these add up to the step); span_ms = summed time from the launch's
 * first CTA entry to the next launch's wait return (includes the part that
 * overlapped the previous kernel); bytes = summed algorithmic bytes (weights
 * read once, activations, the K/V rows read at the step's cache length,
 * outputs written). stats: host array of max_stats (>= 10) entries; *n_stats
 * receives the number of families. Requires a non-empty cache and cached
 * length + n_steps <= max_seq. Allocates a small device and pinned host
 * buffer for the stamps. */
typedef struct llama_q8_kernel_stat {
    char name[32];
    int32_t launches;
    double ms;
    double span_ms;
    double bytes;
} llama_q8_kernel_stat;
llama_q8_status llama_q8_profile_decode(llama_q8_ctx* ctx, int32_t n_steps, llama_q8_kernel_stat* stats,
                                        int32_t max_stats, int32_t* n_stats);

const char* llama_q8_status_str(llama_q8_status s);

/* Self-test of the kernels' bounded waits: launches one CTA that waits on a
 * shared-memory barrier nothing completes, with the same ~1 s limit every
 * kernel of the library uses; the kernel gives up, records the wait's code
 * in device memory and returns. On return *code holds that code (the library
 * uses nonzero codes only for such timeouts) and the device is still usable.
 * Synchronous; about one second. LQ8_ERR_ARG for a NULL code. */
llama_q8_status llama_q8_selftest_wait_timeout(int32_t* code);

/* ---------------------------------------------------------------------------
 * Device-level entry points (kernel workloads). All data pointers are device
 * memory; `stream` is a cudaStream_t (NULL = legacy default stream). They
 * enqueue and return.
 * ------------------------------------------------------------------------- */

/* Quantise f32 w[rows][k] (k % 32 == 0) to Q8_0 blocks out[rows][k/32][34]
 * with the rule d = max|w|/127 (f32), q = round(w/d) (f32 IEEE division,
 * ties away from zero, clamp +-127, d == 0 -> 0), d stored as fp16 (round to
 * nearest even). The pages only fix the block size through byte counts;
 * this rule is the block format's definition the build follows. */
llama_q8_status llama_q8_quantize(const float* w, int64_t rows, int64_t k, void* out,
                                  void* stream);

/* Bytes of the library's device layout for a [rows, k] Q8_0 matrix
 * (rows padded to a multiple of 32; same 34 bytes per block otherwise). */
size_t llama_q8_packed_bytes(int64_t rows, int64_t k);

/* Repack Q8_0 blocks q8[rows][k/32][34] into the device layout used by
 * llama_q8_matmul: packed must hold llama_q8_packed_bytes(rows, k) bytes. */
llama_q8_status llama_q8_pack(const void* q8, int64_t rows, int64_t k, void* packed,
                              void* stream);

/* QMatMul forward: y[m][rows] = x[m][k] . W[rows][k]^T with W the packed Q8_0
 * matrix, f32 x and y. m == 1 runs the matrix-vector kernel, m > 1 a
 * matrix-matrix kernel (the dispatch "生成一个 token" describes for
 * kernel_mul_mv_q8_0_f32 / kernel_mul_mm_q8_0_f32): up to 16 rows on the CUDA
 * cores with f32 accumulation (each 32-row weight tile streamed once and
 * multiplied with every row of x), more rows on the tcgen05 tensor cores: per
 * Q8_0 block the int8 codes (exact in f16) times x, each token row scaled by
 * a power of two (its largest |x| into [2^14, 2^15)) and split into f16 hi
 * and lo parts by a short pass before the product (two f16 products per
 * step, f32 accumulation in tensor memory), the block sums scaled by d and
 * added in f32, the row scale undone exactly; at most 2^-22 relative error per
 * product, plus 2^-39 of the row's largest |x| times the weight. The tensor-core
 * path takes stream-ordered scratch of 4 m + 4 m k bytes (cudaMallocAsync on
 * `stream`, freed after the product; LQ8_ERR_OOM if it fails). packed and x
 * must be 16-byte aligned (LQ8_ERR_ARG otherwise). */
llama_q8_status llama_q8_matmul(const void* packed, int64_t rows, int64_t k, const float* x,
                                int64_t m, float* y, void* stream);

/* llama_q8_matmul with flags. LQ8_MATMUL_EARLY_WEIGHTS: the kernel may start
 * streaming W before the kernel enqueued just before it on `stream` has
 * finished (programmatic dependent launch; x is still read, and y written,
 * only after that kernel has completed). Set it only when no kernel in flight
 * on the stream writes W; it is how the decode step chains its projections.
 * Unknown flag bits -> LQ8_ERR_ARG. */
#define LQ8_MATMUL_EARLY_WEIGHTS 1
/* Kernel for m > 1 token rows (m == 1 always takes the matrix-vector kernel).
 * Neither flag: the tensor cores when m > 16, else the CUDA-core rows kernel,
 * which streams each 32-row weight tile once per chunk of 16 token rows.
 * LQ8_MATMUL_TENSOR_CORES / LQ8_MATMUL_CUDA_CORES force one kernel for any m
 * > 1 (both -> LQ8_ERR_ARG; the CUDA-core kernel with more than 16 rows
 * and k > 16896, or fewer rows and a k whose x slices do not fit its shared
 * memory -> LQ8_ERR_UNSUPPORTED). Both compute the same product within the
 * bounds stated above. */
#define LQ8_MATMUL_TENSOR_CORES 2
#define LQ8_MATMUL_CUDA_CORES 4
llama_q8_status llama_q8_matmul_ex(const void* packed, int64_t rows, int64_t k, const float* x,
                                   int64_t m, float* y, int32_t flags, void* stream);

/* Other GGUF block formats in the matrix-vector product ("速度", CPU GGUF：
 * decode 快，prefill 慢: the pages time QMatMul in Q5_0, Q4K and Q6K and find a
 * 135M Q4_K_M file mostly Q5_0, with Q4K / Q6K for the down projections whose
 * rows of 1536 are a multiple of the 256-weight K-quant block). gguf_type is
 * the GGUF tensor type id: 6 = Q5_0 (32 weights in 22 bytes: fp16 d, 32 bits
 * of fifth bits, 16 bytes of low nibbles; w = d (q - 16)), 12 = Q4_K (256
 * weights in 144 bytes: fp16 d and dmin, 12 bytes of 6-bit scales and mins for
 * eight sub-blocks of 32, 128 bytes of 4-bit codes; w = d sc q - dmin m),
 * 14 = Q6_K (256 weights in 210 bytes: 128 bytes of low nibbles, 64 of top
 * two bits, 16 int8 scales per 16 weights, fp16 d; w = d sc (q - 32)); 8 =
 * Q8_0 routes to the calls above. Layouts inside the blocks are the
 * published GGUF definitions. A [rows, k] matrix is rows * (k / block)
 * blocks, row-major, as in the file; k must be a multiple of the block size
 * (LQ8_ERR_ARG). Other types: LQ8_ERR_UNSUPPORTED. */
#define LLAMA_Q8_GGUF_Q5_0 6
#define LLAMA_Q8_GGUF_Q8_0 8
#define LLAMA_Q8_GGUF_Q4_K 12
#define LLAMA_Q8_GGUF_Q6_K 14

/* Bytes of the library's device layout of a [rows, k] matrix of gguf_type
 * (rows padded to a multiple of 32; the same bytes per block otherwise); 0
 * for an unsupported type or a k that is not a multiple of the block. */
size_t llama_q8_packed_bytes_fmt(int32_t gguf_type, int64_t rows, int64_t k);

/* Repack device blocks[rows][k / block][block bytes] into the device layout
 * (packed: llama_q8_packed_bytes_fmt bytes, device memory, caller-owned; the
 * padding rows are zeroed). Each (32-row tile, block) becomes one contiguous
 * record whose fields are regrouped by row. Enqueues on `stream`. */
llama_q8_status llama_q8_pack_fmt(int32_t gguf_type, const void* blocks, int64_t rows, int64_t k, void* packed,
                                  void* stream);

/* y[rows] = W x for one token (the decode product): x[k] and y[rows] f32
 * device memory, W packed by llama_q8_pack_fmt. Codes are converted to f32
 * exactly and multiplied in f32 with f32 accumulation; Q4_K subtracts
 * dmin * m * (sum of x over the sub-block). packed and x must be 16-byte
 * aligned (LQ8_ERR_ARG); k above the shared-memory limit of the kernel
 * (>= 32768 for every type) gives LQ8_ERR_UNSUPPORTED. flags: as
 * llama_q8_matmul_ex (LQ8_MATMUL_EARLY_WEIGHTS). Enqueues on `stream`. */
llama_q8_status llama_q8_matvec_fmt(int32_t gguf_type, const void* packed, int64_t rows, int64_t k, const float* x,
                                    float* y, int32_t flags, void* stream);

/* Grouped-query attention over a KV cache: for each of T queries at
 * positions index_pos + t, out = softmax(q k^T / sqrt(head_dim) + mask) v,
 * query head h reading KV head h / (n_head / n_head_kv). q[T][n_head][head_dim];
 * k_cache, v_cache [n_head_kv][cache_stride][head_dim] with positions
 * [0, index_pos + T) filled; out[T][n_head][head_dim]. T == 1: the split-KV
 * decode kernel, no mask; T > 1: the causal prefill kernel, query t sees
 * positions <= index_pos + t ("量化 llama 的一次前向", forward：mask 什么时候建).
 * workspace: device scratch of llama_q8_attention_workspace_bytes(...) bytes
 * (split-KV partial results and completion counters); its counters must be
 * zero before the first call and are left zero by every call; calls sharing a
 * workspace must not overlap on the GPU. q, k_cache, v_cache and out must be
 * 16-byte aligned (LQ8_ERR_ARG otherwise). */
size_t llama_q8_attention_workspace_bytes(int32_t n_head, int32_t n_head_kv, int32_t head_dim,
                                          int32_t cache_stride);
llama_q8_status llama_q8_attention(const float* q, const float* k_cache, const float* v_cache,
                                   int32_t T, int32_t index_pos, int32_t n_head,
                                   int32_t n_head_kv, int32_t head_dim, int32_t cache_stride,
                                   float* out, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Single-token grouped-query attention as the decode step runs it: out =
 * softmax(q k^T / sqrt(head_dim)) v over cache positions [0, kv_len), query
 * head h reading KV head h / (n_head / n_head_kv) ("生成一个 token", prefill
 * 和 decode: the fused single-token kernel, query heads of a group sharing their
 * KV head). q[n_head][head_dim]; k_cache, v_cache [n_head_kv][cache_stride]
 * [head_dim]; out[n_head][head_dim]. One cluster of 16 CTAs per KV head (8
 * when the clusters of all KV heads cannot be resident together) splits the
 * positions, streams K/V rows with bulk async copies and merges its partial
 * results through distributed shared memory, so no scratch memory is needed. q, k_cache,
 * v_cache and out must be 16-byte aligned (LQ8_ERR_ARG otherwise); other
 * errors as llama_q8_attention. Enqueues on `stream` and returns. */
llama_q8_status llama_q8_attention_decode(const float* q, const float* k_cache, const float* v_cache,
                                          int32_t kv_len, int32_t n_head, int32_t n_head_kv,
                                          int32_t head_dim, int32_t cache_stride, float* out,
                                          void* stream);

/* Allocation-free single-token attention. No counterpart on the pages: it is
 * a service to callers that cannot allocate device memory — a host that
 * hands all GPU memory to its own pool and accepts only the buffers it
 * passes in, a real-time loop that cannot afford cudaMalloc's implicit
 * device synchronisation, or a plugin that must not create allocations it
 * cannot account for. Same computation as llama_q8_attention with T == 1
 * (q[n_head][head_dim] against cache positions [0, kv_len), out
 * [n_head][head_dim]), but the split-KV partial results and completion
 * counters live in a fixed 2 MiB device array inside this library, which
 * every GPU that loads the library holds until the process exits. The call
 * makes no allocation of any kind; it clears the counters at the start of
 * every call (the array keeps the previous call's contents). Shapes whose
 * scratch need exceeds 2 MiB (n_head_kv * ceil(cache_stride/64) * group *
 * (head_dim + 2) floats, plus counters) return LQ8_ERR_UNSUPPORTED, as do
 * head_dim other than 64/128 and groups above 8; kv_len > cache_stride is
 * LQ8_ERR_CTX. q, k_cache, v_cache and out must be 16-byte aligned (the
 * kernel moves them in 16-byte pieces): LQ8_ERR_ARG otherwise, before any
 * launch. The first call on each device looks up the array's device
 * address (and sets the kernel's shared-memory limit): make that first call
 * before any stream capture. All calls share the one array, so calls that
 * overlap on the GPU (other streams, other threads) race and give wrong
 * results; serialise them. Enqueues on `stream` and returns. */
llama_q8_status llama_q8_attention_decode_noalloc(const float* q, const float* k_cache,
                                                  const float* v_cache, int32_t kv_len, int32_t n_head,
                                                  int32_t n_head_kv, int32_t head_dim,
                                                  int32_t cache_stride, float* out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LLAMA_Q8_H */
