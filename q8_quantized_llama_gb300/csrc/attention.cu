// Grouped-query attention over the preallocated KV cache.
//
// Decode (T = 1): the fused single-token kernel the pages describe for the
// Metal path ("生成一个 token", prefill 和 decode：同一个 forward，不同的路:
// q k^T, scale, softmax and the product with v in one kernel, the query heads
// of a group sharing their KV head inside it). Here the cache is split into
// 64-position chunks, one CTA per (KV head, chunk), all query heads of the
// group handled by that CTA so each K/V row is read from HBM once; the last
// CTA of a KV head (completion counter) merges the chunk results with the
// usual max/sum rescaling. No repeat_kv copy and no cat.
//
// Prefill (T > 1): a causal flash-style kernel, one CTA per (query head,
// 32-query tile), streaming 32-position K/V tiles through shared memory with
// an online softmax; query t sees positions <= index_pos + t ("量化 llama 的一次
// 前向", forward：mask 什么时候建 — the mask is a predicate here, never built).
#include <mutex>

#include "kernels.cuh"
#include "llama_q8.h"
#include "ptx.cuh"

namespace lq8 {

constexpr int kChunk = 64;       // positions per decode CTA
constexpr int kDecThreads = 128;
constexpr int kMaxGroup = 8;

static inline int max_splits_for(int cache_stride) { return (cache_stride + kChunk - 1) / kChunk; }

size_t attn_workspace_bytes(int n_head, int n_head_kv, int head_dim, int cache_stride) {
    const int G = n_head / n_head_kv;
    const size_t ms = (size_t)max_splits_for(cache_stride);
    size_t counters = ((size_t)n_head_kv * 4 + 255) / 256 * 256;
    size_t ml = ((size_t)n_head_kv * ms * G * 2 * 4 + 255) / 256 * 256;
    size_t o = (size_t)n_head_kv * ms * G * head_dim * 4;
    return counters + ml + o;
}

template <int HD>
__global__ void __launch_bounds__(kDecThreads) attn_decode_kernel(
    const float* __restrict__ q, const float* __restrict__ kc, const float* __restrict__ vc, int n_head,
    int n_kv, int cache_stride, int kv_len_host, const DevState* st, float scale, float* __restrict__ out,
    unsigned int* counters, float* part_ml, float* part_o, int max_splits) {
    extern __shared__ float4 sm4[];
    float* Ks = reinterpret_cast<float*>(sm4);      // [kChunk][HD + 4]
    float* Vs = Ks + kChunk * (HD + 4);             // [kChunk][HD]
    float* Qs = Vs + kChunk * HD;                   // [G][HD]
    float* Ps = Qs + kMaxGroup * HD;                // [G][kChunk]
    __shared__ float s_m[kMaxGroup], s_l[kMaxGroup];
    __shared__ int s_last;

    const int kh = blockIdx.x, split = blockIdx.y;
    const int G = n_head / n_kv;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kv_len = st ? st->pos + 1 : kv_len_host;
    const int n_splits = (kv_len + kChunk - 1) / kChunk;
    if (split >= n_splits) return;
    const int j0 = split * kChunk;
    const int n = min(kChunk, kv_len - j0);

    // Rows cached by earlier steps are read before waiting on the preceding
    // kernel; the newest row (position kv_len - 1) is written by that kernel
    // (the QKV epilogue) and is read after the wait, together with q.
    const int n_old = (st && j0 + n == kv_len) ? n - 1 : n;
    const float4* kb = reinterpret_cast<const float4*>(kc + ((int64_t)kh * cache_stride + j0) * HD);
    const float4* vb = reinterpret_cast<const float4*>(vc + ((int64_t)kh * cache_stride + j0) * HD);
    for (int f = tid; f < n_old * (HD / 4); f += kDecThreads) {
        const int row = f / (HD / 4), c = f % (HD / 4);
        *reinterpret_cast<float4*>(Ks + row * (HD + 4) + c * 4) = kb[f];
        reinterpret_cast<float4*>(Vs)[f] = vb[f];
    }
    pdl_wait();
    if (tid == 0) pdl_launch_dependents();
    for (int f = n_old * (HD / 4) + tid; f < n * (HD / 4); f += kDecThreads) {
        const int row = f / (HD / 4), c = f % (HD / 4);
        *reinterpret_cast<float4*>(Ks + row * (HD + 4) + c * 4) = kb[f];
        reinterpret_cast<float4*>(Vs)[f] = vb[f];
    }
    for (int i = tid; i < G * HD; i += kDecThreads) Qs[i] = q[(int64_t)kh * G * HD + i];
    __syncthreads();

    if (tid < n) {
        const float* kr = Ks + tid * (HD + 4);
        for (int g = 0; g < G; ++g) {
            const float* qg = Qs + g * HD;
            float s = 0.0f;
#pragma unroll
            for (int d = 0; d < HD; d += 4) {
                const float4 kk = *reinterpret_cast<const float4*>(kr + d);
                const float4 qq = *reinterpret_cast<const float4*>(qg + d);
                s = fmaf(qq.x, kk.x, s); s = fmaf(qq.y, kk.y, s);
                s = fmaf(qq.z, kk.z, s); s = fmaf(qq.w, kk.w, s);
            }
            Ps[g * kChunk + tid] = s * scale;
        }
    }
    __syncthreads();

    for (int g = warp; g < G; g += kDecThreads / 32) {
        const float a = lane < n ? Ps[g * kChunk + lane] : -INFINITY;
        const float b = lane + 32 < n ? Ps[g * kChunk + lane + 32] : -INFINITY;
        const float mx = warp_max(fmaxf(a, b));
        const float ea = lane < n ? expf(a - mx) : 0.0f;
        const float eb = lane + 32 < n ? expf(b - mx) : 0.0f;
        Ps[g * kChunk + lane] = ea;
        Ps[g * kChunk + lane + 32] = eb;
        const float l = warp_sum(ea + eb);
        if (lane == 0) { s_m[g] = mx; s_l[g] = l; }
    }
    __syncthreads();

    const int64_t pbase = ((int64_t)kh * max_splits + split) * G;
    for (int o = tid; o < G * HD; o += kDecThreads) {
        const int g = o / HD, d = o % HD;
        const float* pg = Ps + g * kChunk;
        float acc = 0.0f;
        for (int j = 0; j < n; ++j) acc = fmaf(pg[j], Vs[j * HD + d], acc);
        if (n_splits == 1) {
            out[((int64_t)kh * G + g) * HD + d] = acc / s_l[g];
        } else {
            part_o[(pbase + g) * HD + d] = acc;
        }
    }
    if (n_splits == 1) return;
    if (tid < G) {
        part_ml[(pbase + tid) * 2 + 0] = s_m[tid];
        part_ml[(pbase + tid) * 2 + 1] = s_l[tid];
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned int ticket = atomicAdd(&counters[kh], 1u);
        s_last = (ticket == (unsigned)(n_splits - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int o = tid; o < G * HD; o += kDecThreads) {
        const int g = o / HD, d = o % HD;
        float M = -INFINITY;
        for (int s = 0; s < n_splits; ++s)
            M = fmaxf(M, __ldcg(part_ml + (((int64_t)kh * max_splits + s) * G + g) * 2));
        float L = 0.0f, acc = 0.0f;
        for (int s = 0; s < n_splits; ++s) {
            const int64_t pb = ((int64_t)kh * max_splits + s) * G + g;
            const float w = expf(__ldcg(part_ml + pb * 2) - M);
            L = fmaf(w, __ldcg(part_ml + pb * 2 + 1), L);
            acc = fmaf(w, __ldcg(part_o + pb * HD + d), acc);
        }
        out[((int64_t)kh * G + g) * HD + d] = acc / L;
    }
    if (tid == 0) atomicExch(&counters[kh], 0u);
}

static constexpr size_t decode_smem_bytes(int hd) {
    return (size_t)(kChunk * (hd + 4) + kChunk * hd + kMaxGroup * hd + kMaxGroup * kChunk) * 4;
}



template <int HD>
static cudaError_t attn_decode_launch(const float* q, const float* kc, const float* vc, int n_head,
                                      int n_kv, int cache_stride, int kv_len, const DevState* st,
                                      float* out, void* ws, bool pdl, cudaStream_t s) {
    const int ms = max_splits_for(cache_stride);
    const int G = n_head / n_kv;
    uint8_t* w = reinterpret_cast<uint8_t*>(ws);
    unsigned int* counters = reinterpret_cast<unsigned int*>(w);
    size_t off = ((size_t)n_kv * 4 + 255) / 256 * 256;
    float* part_ml = reinterpret_cast<float*>(w + off);
    off += ((size_t)n_kv * ms * G * 2 * 4 + 255) / 256 * 256;
    float* part_o = reinterpret_cast<float*>(w + off);
    const size_t smem = decode_smem_bytes(HD);
    const int grid_y = st ? ms : (kv_len + kChunk - 1) / kChunk;
    const float scale = 1.0f / sqrtf((float)HD);
    return launch_ex(attn_decode_kernel<HD>, dim3(n_kv, grid_y), dim3(kDecThreads), smem, s, pdl, q, kc, vc,
                     n_head, n_kv, cache_stride, kv_len, st, scale, out, counters, part_ml, part_o, ms);
}

cudaError_t launch_attn_decode(const float* q, const float* k_cache, const float* v_cache, int n_head,
                               int n_head_kv, int head_dim, int cache_stride, int kv_len,
                               const DevState* st, float* out, void* workspace, bool pdl, cudaStream_t s) {
    if (head_dim == 64)
        return attn_decode_launch<64>(q, k_cache, v_cache, n_head, n_head_kv, cache_stride, kv_len, st, out,
                                      workspace, pdl, s);
    if (head_dim == 128)
        return attn_decode_launch<128>(q, k_cache, v_cache, n_head, n_head_kv, cache_stride, kv_len, st, out,
                                       workspace, pdl, s);
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Decode, cluster form (the decode step's kernel): one cluster of kClusterCtas
// CTAs per KV head; CTA r takes an equal share of the cached positions and
// walks it in 64-position sub-chunks (K/V rows by cp.async, two buffers,
// online softmax across sub-chunks). The group's query heads are handled
// together, so each K/V row is read once. Each CTA stores its (max, sum,
// weighted values) straight into the first CTA's shared memory through the
// cluster's distributed shared memory; one cluster barrier later the first
// CTA merges them: no global scratch, no atomics.
// ---------------------------------------------------------------------------
constexpr int kClusterCtas = 8;
constexpr int kSub = 64;

template <int HD>
struct ClusterSmem {
    float K[2][kSub * HD];
    float V[2][kSub * HD];
    float Q[kMaxGroup * HD];
    float P[kMaxGroup * kSub];
    float O[kMaxGroup * HD];                   // this CTA's running unnormalised output
    float M[kMaxGroup];
    float L[kMaxGroup];
    float corr[kMaxGroup];
    float PO[kClusterCtas][kMaxGroup * HD];    // rank 0: the cluster's partial outputs
    float PM[kClusterCtas][kMaxGroup];
    float PL[kClusterCtas][kMaxGroup];
};

__device__ __forceinline__ void cp_async16_attn(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit_attn() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all_but_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void st_dsmem_f32(float* local_ptr, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_ptr)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

template <int HD>
__global__ void __launch_bounds__(kDecThreads) attn_decode_cluster_kernel(
    const float* __restrict__ q, const float* __restrict__ kc, const float* __restrict__ vc, int n_head, int n_kv,
    int cache_stride, int kv_len_host, const DevState* st, float scale, float* __restrict__ out, int* err) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    ClusterSmem<HD>& S = *reinterpret_cast<ClusterSmem<HD>*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kh = blockIdx.x / kClusterCtas, rank = blockIdx.x % kClusterCtas;
    const int G = n_head / n_kv;
    const int kv_len = st ? st->pos + 1 : kv_len_host;
    const int per = (kv_len + kClusterCtas - 1) / kClusterCtas;
    const int j_begin = min(kv_len, rank * per), j_end = min(kv_len, j_begin + per);
    const int n_rows = j_end - j_begin;
    const int n_sub = (n_rows + kSub - 1) / kSub;
    // The newest position is written by the preceding kernel (QKV epilogue):
    // everything older may be read before the grid dependency wait.
    const int j_new = st ? kv_len - 1 : kv_len;
    const float* kb = kc + (int64_t)kh * cache_stride * HD;
    const float* vb = vc + (int64_t)kh * cache_stride * HD;
    constexpr int C4 = HD / 4;  // float4 chunks per row

    // copy rows [a, b) of sub-chunk i into buffer i&1 (one commit group)
    auto copy_rows = [&](int i, int a, int b) {
        const int base = j_begin + i * kSub;
        for (int f = tid; f < (b - a) * C4; f += kDecThreads) {
            const int row = a - base + f / C4, c = f % C4;
            cp_async16_attn(S.K[i & 1] + row * HD + c * 4, kb + (int64_t)(base + row) * HD + c * 4);
            cp_async16_attn(S.V[i & 1] + row * HD + c * 4, vb + (int64_t)(base + row) * HD + c * 4);
        }
    };
    int split0 = j_begin;
    if (n_sub > 0) {
        const int b = min(j_end, j_begin + kSub);
        split0 = min(b, j_new);
        if (split0 < j_begin) split0 = j_begin;
        copy_rows(0, j_begin, split0);  // cached rows, before the wait
    }
    pdl_wait();
    if (tid == 0) pdl_launch_dependents();
    if (n_sub > 0) copy_rows(0, split0, min(j_end, j_begin + kSub));  // the newest row, if it is here
    cp_async_commit_attn();
    if (n_sub > 1) copy_rows(1, j_begin + kSub, min(j_end, j_begin + 2 * kSub));
    cp_async_commit_attn();
    for (int i = tid; i < G * HD; i += kDecThreads) {
        S.Q[i] = q[(int64_t)kh * G * HD + i];
        S.O[i] = 0.0f;
    }
    if (tid < kMaxGroup) {
        S.M[tid] = -INFINITY;
        S.L[tid] = 0.0f;
    }

    for (int i = 0; i < n_sub; ++i) {
        const int buf = i & 1;
        const int n = min(kSub, n_rows - i * kSub);
        cp_async_wait_all_but_one();
        __syncthreads();
        // scores: 4 threads per position, each a quarter of the head dimension
        {
            const int row = tid >> 2, part = tid & 3;
            const float* kr = S.K[buf] + row * HD + part * (HD / 4);
            for (int g = 0; g < G; ++g) {
                const float* qg = S.Q + g * HD + part * (HD / 4);
                float a0 = 0.0f, a1 = 0.0f;
                if (row < n) {
#pragma unroll
                    for (int d = 0; d < HD / 4; d += 8) {
                        const float4 k0 = *reinterpret_cast<const float4*>(kr + d);
                        const float4 k1 = *reinterpret_cast<const float4*>(kr + d + 4);
                        const float4 q0 = *reinterpret_cast<const float4*>(qg + d);
                        const float4 q1 = *reinterpret_cast<const float4*>(qg + d + 4);
                        a0 = fmaf(q0.x, k0.x, a0); a0 = fmaf(q0.y, k0.y, a0);
                        a0 = fmaf(q0.z, k0.z, a0); a0 = fmaf(q0.w, k0.w, a0);
                        a1 = fmaf(q1.x, k1.x, a1); a1 = fmaf(q1.y, k1.y, a1);
                        a1 = fmaf(q1.z, k1.z, a1); a1 = fmaf(q1.w, k1.w, a1);
                    }
                }
                float sc = a0 + a1;
                sc += __shfl_xor_sync(0xffffffffu, sc, 1);
                sc += __shfl_xor_sync(0xffffffffu, sc, 2);
                if (part == 0 && row < kSub) S.P[g * kSub + row] = sc * scale;
            }
            // rows 32..63 of the sub-chunk
            if (kSub > kDecThreads / 4) {
                const int row2 = row + kDecThreads / 4;
                const float* kr2 = S.K[buf] + row2 * HD + part * (HD / 4);
                for (int g = 0; g < G; ++g) {
                    const float* qg = S.Q + g * HD + part * (HD / 4);
                    float a0 = 0.0f, a1 = 0.0f;
                    if (row2 < n) {
#pragma unroll
                        for (int d = 0; d < HD / 4; d += 8) {
                            const float4 k0 = *reinterpret_cast<const float4*>(kr2 + d);
                            const float4 k1 = *reinterpret_cast<const float4*>(kr2 + d + 4);
                            const float4 q0 = *reinterpret_cast<const float4*>(qg + d);
                            const float4 q1 = *reinterpret_cast<const float4*>(qg + d + 4);
                            a0 = fmaf(q0.x, k0.x, a0); a0 = fmaf(q0.y, k0.y, a0);
                            a0 = fmaf(q0.z, k0.z, a0); a0 = fmaf(q0.w, k0.w, a0);
                            a1 = fmaf(q1.x, k1.x, a1); a1 = fmaf(q1.y, k1.y, a1);
                            a1 = fmaf(q1.z, k1.z, a1); a1 = fmaf(q1.w, k1.w, a1);
                        }
                    }
                    float sc = a0 + a1;
                    sc += __shfl_xor_sync(0xffffffffu, sc, 1);
                    sc += __shfl_xor_sync(0xffffffffu, sc, 2);
                    if (part == 0 && row2 < kSub) S.P[g * kSub + row2] = sc * scale;
                }
            }
        }
        __syncthreads();
        // online softmax statistics per head (one warp per head)
        for (int g = warp; g < G; g += kDecThreads / 32) {
            const float a = lane < n ? S.P[g * kSub + lane] : -INFINITY;
            const float b = lane + 32 < n ? S.P[g * kSub + lane + 32] : -INFINITY;
            const float m_old = S.M[g];
            const float m_new = fmaxf(m_old, warp_max(fmaxf(a, b)));
            const float ea = lane < n ? expf(a - m_new) : 0.0f;
            const float eb = lane + 32 < n ? expf(b - m_new) : 0.0f;
            S.P[g * kSub + lane] = ea;
            S.P[g * kSub + lane + 32] = eb;
            const float sum = warp_sum(ea + eb);
            if (lane == 0) {
                const float corr = expf(m_old - m_new);  // 0 on the first sub-chunk
                S.corr[g] = corr;
                S.L[g] = S.L[g] * corr + sum;
                S.M[g] = m_new;
            }
        }
        __syncthreads();
        for (int o = tid; o < G * HD; o += kDecThreads) {
            const int g = o / HD, d = o % HD;
            const float* pg = S.P + g * kSub;
            const float* vcol = S.V[buf] + d;
            float a0 = 0.0f, a1 = 0.0f;
            int j = 0;
            for (; j + 1 < n; j += 2) {
                a0 = fmaf(pg[j], vcol[j * HD], a0);
                a1 = fmaf(pg[j + 1], vcol[(j + 1) * HD], a1);
            }
            if (j < n) a0 = fmaf(pg[j], vcol[j * HD], a0);
            S.O[o] = fmaf(S.O[o], S.corr[g], a0 + a1);
        }
        __syncthreads();  // buffer buf is free again
        if (i + 2 < n_sub) copy_rows(i + 2, j_begin + (i + 2) * kSub, min(j_end, j_begin + (i + 3) * kSub));
        cp_async_commit_attn();
    }

    // ---- push this CTA's partial result into rank 0, then merge there --------
    if (rank == 0) {
        for (int o = tid; o < G * HD; o += kDecThreads) S.PO[0][o] = S.O[o];
        if (tid < G) {
            S.PM[0][tid] = S.M[tid];
            S.PL[0][tid] = S.L[tid];
        }
    } else {
        for (int o = tid; o < G * HD; o += kDecThreads) st_dsmem_f32(&S.PO[rank][o], 0, S.O[o]);
        if (tid < G) {
            st_dsmem_f32(&S.PM[rank][tid], 0, S.M[tid]);
            st_dsmem_f32(&S.PL[rank][tid], 0, S.L[tid]);
        }
    }
    cluster_sync();
    if (rank == 0) {
        for (int o = tid; o < G * HD; o += kDecThreads) {
            const int g = o / HD;
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < kClusterCtas; ++r) M = fmaxf(M, S.PM[r][g]);
            float Lsum = 0.0f, acc = 0.0f;
#pragma unroll
            for (int r = 0; r < kClusterCtas; ++r) {
                const float m_r = S.PM[r][g];
                const float w = m_r == -INFINITY ? 0.0f : expf(m_r - M);
                Lsum = fmaf(w, S.PL[r][g], Lsum);
                acc = fmaf(w, S.PO[r][o], acc);
            }
            out[(int64_t)kh * G * HD + o] = acc / Lsum;
        }
    }
    (void)err;
}

template <int HD>
static cudaError_t attn_cluster_launch(const float* q, const float* kc, const float* vc, int n_head, int n_kv,
                                       int cache_stride, int kv_len, const DevState* st, float* out, bool pdl,
                                       int* err, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_kv * kClusterCtas);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = sizeof(ClusterSmem<HD>);
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = kClusterCtas;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    int n = 1;
    if (pdl) {
        attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[1].val.programmaticStreamSerializationAllowed = 1;
        n = 2;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    const float scale = 1.0f / sqrtf((float)HD);
    return cudaLaunchKernelEx(&cfg, attn_decode_cluster_kernel<HD>, q, kc, vc, n_head, n_kv, cache_stride, kv_len, st,
                              scale, out, err);
}

cudaError_t launch_attn_decode_cluster(const float* q, const float* k_cache, const float* v_cache, int n_head,
                                       int n_head_kv, int head_dim, int cache_stride, int kv_len,
                                       const DevState* st, float* out, bool pdl, int* err, cudaStream_t s) {
    if (head_dim == 64)
        return attn_cluster_launch<64>(q, k_cache, v_cache, n_head, n_head_kv, cache_stride, kv_len, st, out, pdl,
                                       err, s);
    if (head_dim == 128)
        return attn_cluster_launch<128>(q, k_cache, v_cache, n_head, n_head_kv, cache_stride, kv_len, st, out, pdl,
                                        err, s);
    return cudaErrorInvalidValue;
}

cudaError_t init_attention_attributes() {
    cudaError_t err = cudaFuncSetAttribute(attn_decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)decode_smem_bytes(64));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(attn_decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)decode_smem_bytes(128));
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(attn_decode_cluster_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)sizeof(ClusterSmem<64>));
    if (err != cudaSuccess) return err;
    return cudaFuncSetAttribute(attn_decode_cluster_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(ClusterSmem<128>));
}

// ---------------------------------------------------------------------------
// Prefill
// ---------------------------------------------------------------------------
constexpr int kQTile = 32;
constexpr int kKTile = 32;

template <int HD>
__global__ void __launch_bounds__(128) attn_prefill_kernel(const float* __restrict__ q, const float* __restrict__ kc,
                                                           const float* __restrict__ vc, int T, int index_pos,
                                                           int n_head, int n_kv, int cache_stride, float scale,
                                                           float* __restrict__ out) {
    constexpr int DS = HD / 4;  // dims per thread
    __shared__ __align__(16) float Ks[kKTile][HD + 4];
    __shared__ __align__(16) float Vs[kKTile][HD + 4];
    pdl_wait();
    pdl_launch_dependents();
    const int h = blockIdx.x, qt = blockIdx.y;
    const int G = n_head / n_kv, kh = h / G;
    const int tid = threadIdx.x, r = tid >> 2, c = tid & 3;
    const int i = qt * kQTile + r;
    float qv[DS], o[DS];
#pragma unroll
    for (int d = 0; d < DS; ++d) {
        qv[d] = i < T ? q[((int64_t)i * n_head + h) * HD + c * DS + d] : 0.0f;
        o[d] = 0.0f;
    }
    float m = -INFINITY, l = 0.0f;
    const int kv_end = index_pos + min(T, (qt + 1) * kQTile);
    const float* kbase = kc + (int64_t)kh * cache_stride * HD;
    const float* vbase = vc + (int64_t)kh * cache_stride * HD;
    for (int j0 = 0; j0 < kv_end; j0 += kKTile) {
        const int nt = min(kKTile, kv_end - j0);
        for (int f = tid; f < kKTile * (HD / 4); f += 128) {
            const int row = f / (HD / 4), cc = f % (HD / 4);
            float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
            if (row < nt) {
                kv = *reinterpret_cast<const float4*>(kbase + (int64_t)(j0 + row) * HD + cc * 4);
                vv = *reinterpret_cast<const float4*>(vbase + (int64_t)(j0 + row) * HD + cc * 4);
            }
            *reinterpret_cast<float4*>(&Ks[row][cc * 4]) = kv;
            *reinterpret_cast<float4*>(&Vs[row][cc * 4]) = vv;
        }
        __syncthreads();
        float s[kKTile];
        float mt = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kKTile; ++jj) {
            float p = 0.0f;
#pragma unroll
            for (int d = 0; d < DS; d += 4) {
                const float4 kk = *reinterpret_cast<const float4*>(&Ks[jj][c * DS + d]);
                p = fmaf(qv[d], kk.x, p); p = fmaf(qv[d + 1], kk.y, p);
                p = fmaf(qv[d + 2], kk.z, p); p = fmaf(qv[d + 3], kk.w, p);
            }
            p += __shfl_xor_sync(0xffffffffu, p, 1);
            p += __shfl_xor_sync(0xffffffffu, p, 2);
            const int j = j0 + jj;
            const bool vis = (jj < nt) && (j <= index_pos + i) && (i < T);
            s[jj] = vis ? p * scale : -INFINITY;
            mt = fmaxf(mt, s[jj]);
        }
        const float m_new = fmaxf(m, mt);
        if (m_new != -INFINITY) {
            const float corr = expf(m - m_new);
            l *= corr;
#pragma unroll
            for (int d = 0; d < DS; ++d) o[d] *= corr;
#pragma unroll
            for (int jj = 0; jj < kKTile; ++jj) {
                const float p = expf(s[jj] - m_new);
                l += p;
#pragma unroll
                for (int d = 0; d < DS; d += 4) {
                    const float4 vv = *reinterpret_cast<const float4*>(&Vs[jj][c * DS + d]);
                    o[d] = fmaf(p, vv.x, o[d]); o[d + 1] = fmaf(p, vv.y, o[d + 1]);
                    o[d + 2] = fmaf(p, vv.z, o[d + 2]); o[d + 3] = fmaf(p, vv.w, o[d + 3]);
                }
            }
            m = m_new;
        }
        __syncthreads();
    }
    if (i < T) {
        const float inv = 1.0f / l;
#pragma unroll
        for (int d = 0; d < DS; ++d) out[((int64_t)i * n_head + h) * HD + c * DS + d] = o[d] * inv;
    }
}

cudaError_t launch_attn_prefill(const float* q, const float* k_cache, const float* v_cache, int T,
                                int index_pos, int n_head, int n_head_kv, int head_dim, int cache_stride,
                                float* out, bool pdl, cudaStream_t s) {
    dim3 grid(n_head, (T + kQTile - 1) / kQTile);
    const float scale = 1.0f / sqrtf((float)head_dim);
    if (head_dim == 64)
        return launch_ex(attn_prefill_kernel<64>, grid, dim3(128), 0, s, pdl, q, k_cache, v_cache, T, index_pos,
                         n_head, n_head_kv, cache_stride, scale, out);
    if (head_dim == 128)
        return launch_ex(attn_prefill_kernel<128>, grid, dim3(128), 0, s, pdl, q, k_cache, v_cache, T, index_pos,
                         n_head, n_head_kv, cache_stride, scale, out);
    return cudaErrorInvalidValue;
}

}  // namespace lq8

// ---------------------------------------------------------------------------
// Allocation-free decode attention: the split-KV decode kernel above, with its
// partial results and completion counters in a fixed device array of this
// library instead of caller-provided or allocated memory.
// ---------------------------------------------------------------------------
namespace lq8 {
namespace {

constexpr size_t kNoAllocScratchBytes = 2u << 20;  // 2 MiB, held by every GPU that loads the library
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the host-side name of the array is not a device address).
cudaError_t noalloc_scratch(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        err = init_attention_attributes();
        if (err != cudaSuccess) return err;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace lq8

extern "C" llama_q8_status llama_q8_attention_decode_noalloc(const float* q, const float* k_cache,
                                                             const float* v_cache, int32_t kv_len, int32_t n_head,
                                                             int32_t n_head_kv, int32_t head_dim,
                                                             int32_t cache_stride, float* out, void* stream) {
    using namespace lq8;
    if (!q || !k_cache || !v_cache || !out || kv_len <= 0 || n_head <= 0 || n_head_kv <= 0 ||
        n_head % n_head_kv || cache_stride <= 0)
        return LQ8_ERR_ARG;
    if (kv_len > cache_stride) return LQ8_ERR_CTX;
    if (head_dim != 64 && head_dim != 128) return LQ8_ERR_UNSUPPORTED;
    if (n_head / n_head_kv > kMaxGroup) return LQ8_ERR_UNSUPPORTED;
    if (attn_workspace_bytes(n_head, n_head_kv, head_dim, cache_stride) > kNoAllocScratchBytes)
        return LQ8_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (noalloc_scratch(&scratch) != cudaSuccess) return LQ8_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    // The completion counters must start at zero; the array keeps whatever the
    // previous call left, so clear them on every call.
    const size_t counter_bytes = ((size_t)n_head_kv * 4 + 255) / 256 * 256;
    if (cudaMemsetAsync(scratch, 0, counter_bytes, s) != cudaSuccess) return LQ8_ERR_CUDA;
    if (launch_attn_decode(q, k_cache, v_cache, n_head, n_head_kv, head_dim, cache_stride, kv_len, nullptr, out,
                           scratch, false, s) != cudaSuccess)
        return LQ8_ERR_CUDA;
    return LQ8_OK;
}
