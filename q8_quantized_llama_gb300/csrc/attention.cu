// Grouped-query attention over the preallocated KV cache.
//
// Decode (T = 1): the fused single-token kernel the pages describe for the
// Metal path ("生成一个 token", prefill 和 decode：同一个 forward，不同的路:
// q k^T, scale, softmax and the product with v in one kernel, the query heads
// of a group sharing their KV head inside it). Two forms, neither with a
// repeat_kv copy or a cat:
//  - attn_decode_kernel (split-KV with a workspace): the cache is split into
//    64-position chunks, one CTA per (KV head, chunk), all query heads of the
//    group handled by that CTA so each K/V row is read from HBM once; the last
//    CTA of a KV head (completion counter) merges the chunk results with the
//    usual max/sum rescaling;
//  - attn_decode_cluster_kernel (the decode step's form, no scratch): one
//    thread-block cluster per KV head splits the positions, streams K/V rows
//    with bulk async copies and merges its partials through distributed
//    shared memory (optionally applying the head's W_o column slice).
//
// Prefill (T > 1): attn_prefill_kernel<HD, RT, KS>, a causal flash-style
// kernel, one CTA per (query head, 16*RT query rows) with 256 threads as a
// 16 x 16 grid (or a cluster of KS CTAs splitting the keys: for short
// prompts, and for 64-row tiles when the grid is at most two waves, where the
// causal mask would leave the last row tiles' CTAs alone setting the time;
// the row tiles with the most visible keys are scheduled first),
// register-blocked scores, K/V tiles of 64 positions (head_dim 64)
// or 32 (head_dim 128) double-buffered in shared memory, online softmax; query
// t sees positions <= index_pos + t ("量化 llama 的一次前向", forward：mask
// 什么时候建 — the mask is a predicate here, never built).
#include <mutex>

#include "attn_core.cuh"
#include "kernels.cuh"
#include "llama_q8.h"
#include "ptx.cuh"

namespace lq8 {

constexpr int kChunk = 64;       // positions per decode CTA
constexpr int kDecThreads = 128;

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
// Decode, cluster form (the decode step's kernel): one cluster of CL CTAs per
// KV head (CL = 16 when all the heads' clusters can be resident at once, else
// 8); CTA r takes an equal share of the positions. The share is walked in
// windows of up to 256 positions, each in two passes over 64-position stages
// that a producer warp streams (one bulk copy per stage) through a 4-deep
// ring of shared-memory stages:
//   K pass  lane c of a warp holds float4 chunk c of every query head of the
//           group in registers and multiplies it into chunk c of the warp's
//           rows (one conflict-free 128-bit load per row); a butterfly
//           reduce-scatter over the lanes of a row then leaves one finished
//           (row, head) score in each lane;
//   softmax warp g updates head g's running max and sum over the window and
//           turns its scores into weights in place;
//   V pass  thread (d4, slice) accumulates the float4 of output dims d4 for
//           every head over its slice of positions (the group's weights of a
//           position in one broadcast load).
// The V rows of a window are requested as soon as a stage is free, so they
// overlap the K pass and the softmax. K/V rows cached by earlier steps are
// requested before the grid dependency wait, the newest row after it. The
// slices are summed in shared memory and every CTA stores its (max, sum,
// weighted values) into the first CTA's shared memory through distributed
// shared memory; one cluster barrier later the first CTA merges them. All the
// group's query heads share each K/V row read ("生成一个 token": the KV heads
// are shared inside the kernel, no repeat_kv copy). GP is the group size
// rounded up to 4 or 8; the padding heads have q = 0 and are never stored.
// ---------------------------------------------------------------------------
template <int HD, int CL, int GP, bool FO>
__global__ void __launch_bounds__(kCaThreads, 1) attn_decode_cluster_kernel(
    const float* __restrict__ q, const float* __restrict__ kc, const float* __restrict__ vc, int n_head, int n_kv,
    int cache_stride, int kv_len_host, const DevState* st, float scale, float* __restrict__ out, AttnOproj fo,
    int* err) {
    using Geo = CaGeom<HD>;
    constexpr int D4 = HD / 4;
    extern __shared__ __align__(128) float smf[];
    __shared__ __align__(8) uint64_t full[kCaStages];
    __shared__ __align__(8) uint64_t empty[kCaStages];
    __shared__ __align__(8) uint64_t wo_bar;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) stamp_at(fo.stamp, 0);
    const int kh = blockIdx.x / CL, rank = blockIdx.x % CL;
    const int G = n_head / n_kv;
    const int nbk = G * HD / 32;                       // W_o column blocks of this group
    const int tiles = FO ? fo.wo.rows_pad >> 5 : 0;
    const CaPlan pl = ca_plan<HD>(G, GP, CL, FO ? fo_wo_bytes(fo.wo.rows_pad, G, HD, CL) : 0);
    float* S = smf + pl.s;
    float* Q = smf + pl.q;
    float* CORR = smf + pl.corr;
    float* PO = smf + pl.po;
    float* PM = smf + pl.pm;
    float* PLs = smf + pl.pl;
    float* OM = smf + pl.om;
    float* RED2 = smf + pl.red2;
    uint8_t* WO = reinterpret_cast<uint8_t*>(smf + pl.wo);

    const int kv_len = st ? st->pos + 1 : kv_len_host;
    const int per = (kv_len + CL - 1) / CL;
    const int j_begin = min(kv_len, rank * per), j_end = min(kv_len, j_begin + per);
    // The newest position is written by the preceding kernel (the QKV
    // epilogue) in the decode step; every older row may be read before the
    // grid dependency wait.
    const int j_new = st ? kv_len - 1 : kv_len;
    const float* kb = kc + (int64_t)kh * cache_stride * HD;
    const float* vb = vc + (int64_t)kh * cache_stride * HD;

    if (tid == 0) {
        for (int s = 0; s < kCaStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCaWarps);
        }
        mbar_init(&wo_bar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCaWarps) {
        if (lane == 0) {
            if (FO) {
                // this CTA's W_o tiles, the group's column blocks: constant weights, requested first
                int n_t = 0;
                for (int t = rank; t < tiles; t += CL) ++n_t;
                mbar_arrive_expect_tx(&wo_bar, (uint32_t)(n_t * nbk * 1088));
                const int nb = fo.wo.k >> 5, b0 = kh * nbk;
                int i = 0;
                for (int t = rank; t < tiles; t += CL, ++i) {
                    uint8_t* dst = WO + (size_t)i * nbk * 1088;
                    bulk_g2s(dst, reinterpret_cast<const uint8_t*>(fo.wo.qs) + (size_t)t * fo.wo.k * 32 + b0 * 1024,
                             (uint32_t)(nbk * 1024), &wo_bar);
                    bulk_g2s(dst + nbk * 1024,
                             reinterpret_cast<const uint8_t*>(fo.wo.d) + ((size_t)t * nb + b0) * 64,
                             (uint32_t)(nbk * 64), &wo_bar);
                }
            }
            bool waited = false;
            int j = 0;
            ca_produce_head<HD>(smf, full, empty, kb, vb, j_begin, j_end, j_new, false, waited, j, err);
        }
        __syncwarp();
        cluster_sync();  // pairs with the consumers' cluster barriers below
        if (FO) cluster_sync();
        return;
    }

    // ---- consumers ---------------------------------------------------------------------
    pdl_wait();
    if (tid == 0) {
        pdl_launch_dependents();
        stamp_at(fo.stamp, 1);
    }
    for (int i = tid; i < GP * HD; i += kCaCT) Q[i] = i < G * HD ? q[(int64_t)kh * G * HD + i] : 0.0f;
    named_bar_sync(1, kCaCT);
    float4 qr[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) qr[g] = *reinterpret_cast<const float4*>(Q + g * HD + (lane % D4) * 4);
    float4 o[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) o[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    float m_run = -INFINITY, l_run = 0.0f;
    int j = 0;
    bool first = true;
    ca_consume_head<HD, GP>(smf, full, empty, S, CORR, qr, G, j_begin, j_end, scale, j, first, o, m_run, l_run, err);

    // ---- sum the position slices, push the CTA's partial result to rank 0 ----------------
    const int d4 = tid % D4, slice = tid / D4;
    named_bar_sync(1, kCaCT);  // the ring is free: reuse it for the slice sums
    float* RED = smf;          // [kSlices][G][HD]
#pragma unroll
    for (int g = 0; g < GP; ++g)
        if (g < G) *reinterpret_cast<float4*>(RED + (slice * G + g) * HD + d4 * 4) = o[g];
    named_bar_sync(1, kCaCT);
    for (int e = tid; e < G * HD; e += kCaCT) {
        float acc = 0.0f;
        for (int s = 0; s < Geo::kSlices; ++s) acc += RED[s * G * HD + e];
        st_dsmem_f32(&PO[rank * G * HD + e], 0, acc);
    }
    if (warp < G && lane == 0) {
        st_dsmem_f32(&PM[rank * G + warp], 0, m_run);
        st_dsmem_f32(&PLs[rank * G + warp], 0, l_run);
    }
    cluster_sync();
    if (rank == 0) {
        for (int e = tid; e < G * HD; e += kCaCT) {
            const int g = e / HD;
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < CL; ++r) M = fmaxf(M, PM[r * G + g]);
            float Lsum = 0.0f, acc = 0.0f;
#pragma unroll
            for (int r = 0; r < CL; ++r) {
                const float m_r = PM[r * G + g];
                const float wgt = m_r == -INFINITY ? 0.0f : expf(m_r - M);
                Lsum = fmaf(wgt, PLs[r * G + g], Lsum);
                acc = fmaf(wgt, PO[r * G * HD + e], acc);
            }
            const float val = acc / Lsum;
            if (FO) {
#pragma unroll
                for (int r = 0; r < CL; ++r) st_dsmem_f32(&OM[e], (uint32_t)r, val);
            } else {
                out[(int64_t)kh * G * HD + e] = val;
            }
        }
    }
    if (!FO) return;

    // ---- O projection of the group: part[kh] = W_o[:, group columns] o ---------------------
    cluster_sync();  // the merged output is in every CTA
    mbar_wait_bounded(&wo_bar, 0, err, 24);
    int i = 0;
    for (int t = rank; t < tiles; t += CL, ++i) {
        const uint8_t* tw = WO + (size_t)i * nbk * 1088;
        float acc = 0.0f;
        for (int b = warp; b < nbk; b += kCaWarps) {
            const uint4 q0 = *reinterpret_cast<const uint4*>(tw + b * 1024 + lane * 16);
            const uint4 q1 = *reinterpret_cast<const uint4*>(tw + b * 1024 + 512 + lane * 16);
            const float d = __half2float(reinterpret_cast<const __half*>(tw + nbk * 1024)[b * 32 + lane]);
            const float4* x4 = reinterpret_cast<const float4*>(OM + b * 32);
            uint64_t a0 = 0, a1 = 0;
            a0 = dot4_acc(q0.x, x4[0], a0); a1 = dot4_acc(q1.x, x4[4], a1);
            a0 = dot4_acc(q0.y, x4[1], a0); a1 = dot4_acc(q1.y, x4[5], a1);
            a0 = dot4_acc(q0.z, x4[2], a0); a1 = dot4_acc(q1.z, x4[6], a1);
            a0 = dot4_acc(q0.w, x4[3], a0); a1 = dot4_acc(q1.w, x4[7], a1);
            acc = fmaf(d, (f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1)), acc);
        }
        RED2[warp * 33 + lane] = acc;
        named_bar_sync(1, kCaCT);
        if (warp == 0) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kCaWarps; ++w) v += RED2[w * 33 + lane];
            const int r = t * 32 + lane;
            if (r < fo.wo.rows) fo.part[(int64_t)kh * fo.part_stride + r] = v;
        }
        named_bar_sync(1, kCaCT);
    }
}

// ---------------------------------------------------------------------------
// Front half of a decode layer for models whose per-KV-head projections are
// small: ONE kernel per layer does RMSNorm -> the Q/K/V rows of KV head kh ->
// rope_i -> KV append -> attention -> the group's W_o column slice, in one
// cluster of CL CTAs per KV head ("量化 llama 的一次前向", forward: the same
// steps as the separate kernels, fused). Cluster kh owns the q rows of its G
// query heads and the k and v rows of head kh (G*hd/32 + 2*hd/32 tiles of
// [Wq;Wk;Wv]); CTA r computes tiles r, r + CL, ... of that list against the
// normalised x and broadcasts the finished (rotated) rows into every CTA of
// the cluster through distributed shared memory, writing k and v to the
// cache as well. After a cluster barrier each CTA runs the attention passes
// over its position share with the newest K/V row taken from shared memory,
// then the merge and the W_o slice as the attention kernel does. The
// exchanges between CTAs are asynchronous stores (st.async) that complete
// transaction counts on the receiving CTA's mbarriers, so no cluster-wide
// barrier waits on the producer warp while it waits for free ring stages.
// Weights (both projections' tiles) and the cached K/V rows are requested
// before the grid dependency wait; only x waits for the preceding kernel.
// ---------------------------------------------------------------------------

__host__ __device__ inline int front_qkv_tiles(int G, int hd) { return (G * hd + 2 * hd) / 32; }
__host__ __device__ inline int front_wq_bytes(int G, int hd, int h, int cl) {
    return (front_qkv_tiles(G, hd) + cl - 1) / cl * (h / 32) * 1088;
}
struct FrontPlan {
    CaPlan ca;
    int wq, xn, knew, vnew, floats;
};
template <int HD>
__host__ __device__ inline FrontPlan front_plan(int G, int GP, int cl, int h, int wo_bytes) {
    FrontPlan p;
    p.ca = ca_plan<HD>(G, GP, cl, wo_bytes);
    int o = p.ca.floats;
    auto take = [&](int n) { const int r = o; o += ca_round(n); return r; };
    p.wq = take(front_wq_bytes(G, HD, h, cl) / 4);
    p.xn = take(h);
    p.knew = take(HD);
    p.vnew = take(HD);
    p.floats = o;
    return p;
}

template <int HD, int CL, int GP>
__global__ void __launch_bounds__(kCaThreads, 1) layer_front_cluster_kernel(FrontArgs fa) {
    constexpr int D4 = HD / 4;
    extern __shared__ __align__(128) float smf[];
    __shared__ __align__(8) uint64_t full[kCaStages];
    __shared__ __align__(8) uint64_t empty[kCaStages];
    __shared__ __align__(8) uint64_t wo_bar, wq_bar;
    __shared__ __align__(8) uint64_t rows_bar, part_bar;  // completed by st.async bytes

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) stamp_at(fa.stamp, 0);
    const int kh = blockIdx.x / CL, rank = blockIdx.x % CL;
    const int n_head = fa.n_head, n_kv = fa.n_kv, G = n_head / n_kv;
    const int h = fa.wqkv.k, nbx = h >> 5;
    const int qd = n_head * HD, kvd = n_kv * HD;
    const int nbk = G * HD / 32;                        // W_o column blocks of this group
    const int o_tiles = fa.wo.rows_pad >> 5;
    const int nq = G * HD / 32, nkt = HD / 32, n_qkv = nq + 2 * nkt;
    const FrontPlan pl = front_plan<HD>(G, GP, CL, h, fo_wo_bytes(fa.wo.rows_pad, G, HD, CL));
    float* S = smf + pl.ca.s;
    float* Q = smf + pl.ca.q;
    float* CORR = smf + pl.ca.corr;
    float* PO = smf + pl.ca.po;
    float* PM = smf + pl.ca.pm;
    float* PLs = smf + pl.ca.pl;
    float* OM = smf + pl.ca.om;
    float* RED2 = smf + pl.ca.red2;
    uint8_t* WO = reinterpret_cast<uint8_t*>(smf + pl.ca.wo);
    uint8_t* WQ = reinterpret_cast<uint8_t*>(smf + pl.wq);
    float* XN = smf + pl.xn;
    float* KNEW = smf + pl.knew;
    float* VNEW = smf + pl.vnew;

    const int pos = fa.st->pos;  // written two or more launches back
    const int kv_len = pos + 1;
    const int per = (kv_len + CL - 1) / CL;
    const int j_begin = min(kv_len, rank * per), j_end = min(kv_len, j_begin + per);
    const int j_new = kv_len - 1;
    const float* kb = fa.kc + (int64_t)kh * fa.stride * HD;
    const float* vb = fa.vc + (int64_t)kh * fa.stride * HD;

    // first row (in [Wq;Wk;Wv]) of entry i of this cluster's tile list
    auto qkv_tile_row0 = [&](int i) -> int {
        if (i < nq) return kh * G * HD + i * 32;
        if (i < nq + nkt) return qd + kh * HD + (i - nq) * 32;
        return qd + kvd + kh * HD + (i - nq - nkt) * 32;
    };

    if (tid == 0) {
        for (int s = 0; s < kCaStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCaWarps);
        }
        mbar_init(&wo_bar, 1);
        mbar_init(&wq_bar, 1);
        mbar_init(&rows_bar, 1);
        mbar_init(&part_bar, 1);
        fence_mbar_init();
        // the bytes each exchange brings into this CTA
        mbar_arrive_expect_tx(&rows_bar, (uint32_t)((G + 2) * HD * 4));
        mbar_arrive_expect_tx(&part_bar, (uint32_t)(CL * (G * HD + 2 * G) * 4));
    }
    __syncthreads();
    // Every CTA's barriers exist (and expect their bytes) before any peer
    // stores into it. This is the only cluster-wide barrier: the exchanges
    // below are asynchronous stores that complete transaction counts on the
    // receiver's mbarriers, so the producer warp never has to join a barrier
    // while it waits for free ring stages.
    cluster_sync();

    if (warp == kCaWarps) {
        if (lane == 0) {
            // projection tiles: constant weights, requested first
            int n_t = 0;
            for (int i = rank; i < n_qkv; i += CL) ++n_t;
            mbar_arrive_expect_tx(&wq_bar, (uint32_t)(n_t * nbx * 1088));
            int u = 0;
            for (int i = rank; i < n_qkv; i += CL, ++u) {
                const int t = qkv_tile_row0(i) >> 5;
                uint8_t* dst = WQ + (size_t)u * nbx * 1088;
                bulk_g2s(dst, reinterpret_cast<const uint8_t*>(fa.wqkv.qs) + (size_t)t * h * 32,
                         (uint32_t)(nbx * 1024), &wq_bar);
                bulk_g2s(dst + nbx * 1024, reinterpret_cast<const uint8_t*>(fa.wqkv.d) + (size_t)t * nbx * 64,
                         (uint32_t)(nbx * 64), &wq_bar);
            }
            n_t = 0;
            for (int t = rank; t < o_tiles; t += CL) ++n_t;
            mbar_arrive_expect_tx(&wo_bar, (uint32_t)(n_t * nbk * 1088));
            const int nbo = fa.wo.k >> 5, b0 = kh * nbk;
            u = 0;
            for (int t = rank; t < o_tiles; t += CL, ++u) {
                uint8_t* dst = WO + (size_t)u * nbk * 1088;
                bulk_g2s(dst, reinterpret_cast<const uint8_t*>(fa.wo.qs) + (size_t)t * fa.wo.k * 32 + b0 * 1024,
                         (uint32_t)(nbk * 1024), &wo_bar);
                bulk_g2s(dst + nbk * 1024, reinterpret_cast<const uint8_t*>(fa.wo.d) + ((size_t)t * nbo + b0) * 64,
                         (uint32_t)(nbk * 64), &wo_bar);
            }
            // cached K/V rows of this CTA's share; the newest row comes from the projection
            bool waited = false;
            int j = 0;
            ca_produce_head<HD>(smf, full, empty, kb, vb, j_begin, j_end, j_new, true, waited, j, fa.err);
        }
        return;
    }

    // ---- consumers: RMSNorm of x ----------------------------------------------------------
    // the norm weight is constant: loaded before the dependency wait (h <= 1024)
    constexpr int kGPre = 4;
    float gpre[kGPre];
#pragma unroll
    for (int u = 0; u < kGPre; ++u) {
        const int i = tid + u * kCaCT;
        gpre[u] = i < h ? fa.g[i] : 0.0f;
    }
    // the rotary row of this position (the table is constant and pos was written
    // two or more launches back): into shared memory before the wait, so the
    // rotation after the projections reads no global memory
    __shared__ float rope_cs[2][HD / 2];
    if (tid < HD / 2) {
        rope_cs[0][tid] = fa.rope_cos[(int64_t)pos * (HD / 2) + tid];
        rope_cs[1][tid] = fa.rope_sin[(int64_t)pos * (HD / 2) + tid];
    }
    pdl_wait();
    if (tid == 0) {
        pdl_launch_dependents();
        stamp_at(fa.stamp, 1);
    }
    // x * g into XN and the sum of squares; the scale 1/rms multiplies the finished
    // projection rows, so no barrier waits on the reduction before the products.
    float r_norm;
    {
        float ss = 0.0f;
        const bool keep = fa.x_store && kh == 0 && rank == 0;
        // x and every partial of each element are requested before any is used,
        // so the whole input costs one memory round trip
        constexpr int kMaxParts = 8;
        float xin[kGPre], xp[kGPre][kMaxParts];
#pragma unroll
        for (int u = 0; u < kGPre; ++u) {
            const int i = tid + u * kCaCT;
            xin[u] = i < h ? fa.x[i] : 0.0f;
#pragma unroll
            for (int p = 0; p < kMaxParts; ++p)
                xp[u][p] = (i < h && p < fa.n_xparts) ? fa.xparts[(size_t)p * h + i] : 0.0f;
        }
        for (int i = tid, u = 0; i < h; i += kCaCT, ++u) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kGPre; ++w)
                if (w == u) {
                    v = xin[w];
#pragma unroll
                    for (int p = 0; p < kMaxParts; ++p)
                        if (p < fa.n_xparts) v += xp[w][p];
                }
            if (keep) fa.x_store[i] = v;
            ss = fmaf(v, v, ss);
            float gg = 0.0f;
#pragma unroll
            for (int w = 0; w < kGPre; ++w)
                if (w == u) gg = gpre[w];
            if (u >= kGPre) gg = fa.g[i];
            XN[i] = v * gg;
        }
        ss = warp_sum(ss);
        if (lane == 0) RED2[warp * 33 + 32] = ss;
        for (int i = tid; i < GP * HD; i += kCaCT)
            if (i >= G * HD) Q[i] = 0.0f;  // padding heads
        named_bar_sync(1, kCaCT);
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < kCaWarps; ++w) t += RED2[w * 33 + 32];
        r_norm = 1.0f / sqrtf(t / (float)h + fa.eps);
    }

    // ---- this CTA's projection tiles; rotated rows to every CTA of the cluster ----------
    mbar_wait_bounded(&wq_bar, 0, fa.err, 25);
    {
        const float* cosr = rope_cs[0];
        const float* sinr = rope_cs[1];
        int u = 0;
        for (int i = rank; i < n_qkv; i += CL, ++u) {
            const uint8_t* tw = WQ + (size_t)u * nbx * 1088;
            const float acc = tile_blocks_dot(tw, nbx, warp, kCaWarps, nbx, lane, XN);
            RED2[warp * 33 + lane] = acc;
            named_bar_sync(1, kCaCT);
            // every warp sums the eight partials (same order, same result) and
            // sends the rows to its share of the cluster's CTAs: ranks warp,
            // warp + 8; warp 0 also writes the cache
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kCaWarps; ++w) v += RED2[w * 33 + lane];
            v *= r_norm;
            const float other = __shfl_xor_sync(0xffffffffu, v, 1);
            const int row = qkv_tile_row0(i) + lane;  // row of [Wq;Wk;Wv]
            const int d = row % HD;
            float val = v;
            float* dst = &VNEW[d];
            if (i < nq + nkt) {
                // q or k row: rotate the pair (2m, 2m+1) of its head
                const float cs = cosr[d >> 1], sn = sinr[d >> 1];
                val = (lane & 1) ? other * sn + v * cs : v * cs - other * sn;
                dst = i < nq ? &Q[row - kh * G * HD] : &KNEW[d];
                if (i >= nq && warp == 0) fa.kc[((int64_t)kh * fa.stride + pos) * HD + d] = val;
            } else if (warp == 0) {
                fa.vc[((int64_t)kh * fa.stride + pos) * HD + d] = v;
            }
            for (int r = warp; r < CL; r += kCaWarps) st_async_f32(dst, (uint32_t)r, val, &rows_bar);
            if (i + CL < n_qkv) named_bar_sync(1, kCaCT);  // RED2 is refilled by the next tile
        }
    }
    mbar_wait_bounded(&rows_bar, 0, fa.err, 26);  // q, k and v of the new position are here

    // ---- attention over this CTA's positions, newest row from shared memory -------------
    float4 qr[GP], o[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
        qr[g] = *reinterpret_cast<const float4*>(Q + g * HD + (lane % D4) * 4);
        o[g] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m_run = -INFINITY, l_run = 0.0f;
    int j = 0;
    bool first = true;
    ca_consume_head<HD, GP>(smf, full, empty, S, CORR, qr, G, j_begin, j_end, fa.scale, j, first, o, m_run, l_run,
                            fa.err, j_new, KNEW, VNEW);
    const int d4 = tid % D4, slice = tid / D4;
    named_bar_sync(1, kCaCT);  // the ring is free: reuse it for the slice sums
    float* RED = smf;          // [kSlices][G][HD]
#pragma unroll
    for (int g = 0; g < GP; ++g)
        if (g < G) *reinterpret_cast<float4*>(RED + (slice * G + g) * HD + d4 * 4) = o[g];
    named_bar_sync(1, kCaCT);
    // every CTA gets every CTA's partial result and merges all of them itself
    for (int e4 = tid; e4 < G * HD / 4; e4 += kCaCT) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s2 = 0; s2 < CaGeom<HD>::kSlices; ++s2) {
            const float4 v = *reinterpret_cast<const float4*>(RED + s2 * G * HD + e4 * 4);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
#pragma unroll 4
        for (int r = 0; r < CL; ++r) st_async_f32x4(&PO[rank * G * HD + e4 * 4], (uint32_t)r, acc, &part_bar);
    }
    if (warp < G && lane < CL) {
        st_async_f32(&PM[rank * G + warp], (uint32_t)lane, m_run, &part_bar);
        st_async_f32(&PLs[rank * G + warp], (uint32_t)lane, l_run, &part_bar);
    }
    // every CTA's partial result is here; these are the last stores any peer
    // makes into this CTA, so after this wait the CTA may run to its end
    mbar_wait_bounded(&part_bar, 0, fa.err, 27);
    {
        // merge weights once per (head, source CTA): w = exp(m_r - M) / sum_r' exp(m_r' - M) l_r'
        float* WGT = RED2;  // [G][CL], G * CL <= 8 * 16 of the 8 x 33 floats
        if (warp < G) {
            const float m_r = lane < CL ? PM[lane * G + warp] : -INFINITY;
            const float M = warp_max(m_r);
            const float w = (lane < CL && m_r != -INFINITY) ? expf(m_r - M) : 0.0f;
            const float L = warp_sum(lane < CL ? w * PLs[lane * G + warp] : 0.0f);
            if (lane < CL) WGT[warp * CL + lane] = w / L;
        }
        named_bar_sync(1, kCaCT);
        for (int e = tid; e < G * HD; e += kCaCT) {
            const float* wg = WGT + (e / HD) * CL;
            float acc = 0.0f;
#pragma unroll
            for (int r = 0; r < CL; ++r) acc = fmaf(wg[r], PO[r * G * HD + e], acc);
            OM[e] = acc;
        }
    }
    named_bar_sync(1, kCaCT);

    // ---- W_o column slice of the group: part[kh] ------------------------------------------
    mbar_wait_bounded(&wo_bar, 0, fa.err, 24);
    int u = 0;
    for (int t = rank; t < o_tiles; t += CL, ++u) {
        const uint8_t* tw = WO + (size_t)u * nbk * 1088;
        float acc = 0.0f;
        for (int b = warp; b < nbk; b += kCaWarps) {
            const uint4 q0 = *reinterpret_cast<const uint4*>(tw + b * 1024 + lane * 16);
            const uint4 q1 = *reinterpret_cast<const uint4*>(tw + b * 1024 + 512 + lane * 16);
            const float d = __half2float(reinterpret_cast<const __half*>(tw + nbk * 1024)[b * 32 + lane]);
            const float4* x4 = reinterpret_cast<const float4*>(OM + b * 32);
            uint64_t a0 = 0, a1 = 0;
            a0 = dot4_acc(q0.x, x4[0], a0); a1 = dot4_acc(q1.x, x4[4], a1);
            a0 = dot4_acc(q0.y, x4[1], a0); a1 = dot4_acc(q1.y, x4[5], a1);
            a0 = dot4_acc(q0.z, x4[2], a0); a1 = dot4_acc(q1.z, x4[6], a1);
            a0 = dot4_acc(q0.w, x4[3], a0); a1 = dot4_acc(q1.w, x4[7], a1);
            acc = fmaf(d, (f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1)), acc);
        }
        RED2[warp * 33 + lane] = acc;
        named_bar_sync(1, kCaCT);
        if (warp == 0) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < kCaWarps; ++w) v += RED2[w * 33 + lane];
            const int r = t * 32 + lane;
            if (r < fa.wo.rows) fa.part[(int64_t)kh * fa.part_stride + r] = v;
        }
        if (t + CL < o_tiles) named_bar_sync(1, kCaCT);  // RED2 is refilled by the next tile
    }
}

template <int HD, int CL, int GP, bool FO>
static cudaLaunchConfig_t ca_config(int n_kv, int G, int wo_bytes, cudaStream_t s, cudaLaunchAttribute* attrs,
                                    bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_kv * CL);
    cfg.blockDim = dim3(kCaThreads);
    cfg.dynamicSmemBytes = (size_t)ca_plan<HD>(G, GP, CL, wo_bytes).floats * 4;
    cfg.stream = s;
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = CL;
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
    return cfg;
}

static constexpr int kCaSmemLimit = 227 * 1024 - 1024;

template <int HD, int CL, int GP, bool FO>
static cudaError_t ca_set_attrs() {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_cluster_kernel<HD, CL, GP, FO>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kCaSmemLimit);
    if (e == cudaSuccess && CL > 8)
        e = cudaFuncSetAttribute(attn_decode_cluster_kernel<HD, CL, GP, FO>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

// How many 16-CTA clusters of a configuration can be resident at once, cached
// per (head dim, group, O-projection bytes). A launch uses 16-CTA clusters
// only when every KV head's cluster fits at the same time.
struct CaOcc {
    int hd, G, wo_bytes, max16;
};
static CaOcc g_ca_occ[32];
static int g_ca_n_occ = 0;
static std::mutex g_ca_mu;
static bool g_ca16_ok = false;

template <int HD, int GP, bool FO>
static int ca_max16(int G, int wo_bytes) {
    std::lock_guard<std::mutex> lock(g_ca_mu);
    for (int i = 0; i < g_ca_n_occ; ++i)
        if (g_ca_occ[i].hd == HD && g_ca_occ[i].G == G && g_ca_occ[i].wo_bytes == wo_bytes) return g_ca_occ[i].max16;
    int n = -1;
    if (g_ca16_ok && (size_t)ca_plan<HD>(G, GP, 16, wo_bytes).floats * 4 <= (size_t)kCaSmemLimit) {
        cudaLaunchAttribute attrs[2];
        cudaLaunchConfig_t cfg = ca_config<HD, 16, GP, FO>(1, G, wo_bytes, 0, attrs, false);
        if (cudaOccupancyMaxActiveClusters(&n, attn_decode_cluster_kernel<HD, 16, GP, FO>, &cfg) != cudaSuccess ||
            n < 1) {
            cudaGetLastError();
            n = -1;
        }
    }
    if (g_ca_n_occ < 32) g_ca_occ[g_ca_n_occ++] = CaOcc{HD, G, wo_bytes, n};
    return n;
}

template <int HD, int GP, bool FO>
static int ca_cluster_size(int n_kv, int G, const AttnOproj* fo) {
    const int wo16 = FO ? fo_wo_bytes(fo->wo.rows_pad, G, HD, 16) : 0;
    return ca_max16<HD, GP, FO>(G, wo16) >= n_kv ? 16 : 8;
}

template <int HD, int GP, bool FO>
static cudaError_t ca_launch(const float* q, const float* kc, const float* vc, int n_head, int n_kv, int cache_stride,
                             int kv_len, const DevState* st, float* out, const AttnOproj* fo, bool pdl, int* err,
                             cudaStream_t s, unsigned long long* stamp) {
    const int G = n_head / n_kv;
    const float scale = 1.0f / sqrtf((float)HD);
    AttnOproj f = FO ? *fo : AttnOproj{};
    f.stamp = stamp;
    cudaLaunchAttribute attrs[2];
    if (ca_cluster_size<HD, GP, FO>(n_kv, G, fo) == 16) {
        const int wo = FO ? fo_wo_bytes(f.wo.rows_pad, G, HD, 16) : 0;
        cudaLaunchConfig_t cfg = ca_config<HD, 16, GP, FO>(n_kv, G, wo, s, attrs, pdl);
        return cudaLaunchKernelEx(&cfg, attn_decode_cluster_kernel<HD, 16, GP, FO>, q, kc, vc, n_head, n_kv,
                                  cache_stride, kv_len, st, scale, out, f, err);
    }
    const int wo = FO ? fo_wo_bytes(f.wo.rows_pad, G, HD, 8) : 0;
    cudaLaunchConfig_t cfg = ca_config<HD, 8, GP, FO>(n_kv, G, wo, s, attrs, pdl);
    return cudaLaunchKernelEx(&cfg, attn_decode_cluster_kernel<HD, 8, GP, FO>, q, kc, vc, n_head, n_kv, cache_stride,
                              kv_len, st, scale, out, f, err);
}

template <bool FO>
static cudaError_t ca_dispatch(const float* q, const float* k_cache, const float* v_cache, int n_head, int n_head_kv,
                               int head_dim, int cache_stride, int kv_len, const DevState* st, float* out,
                               const AttnOproj* fo, bool pdl, int* err, cudaStream_t s,
                               unsigned long long* stamp) {
    if (n_head_kv <= 0 || n_head % n_head_kv || n_head / n_head_kv > kMaxGroup) return cudaErrorInvalidValue;
    const bool wide = n_head / n_head_kv > 4;
    if (head_dim == 64)
        return wide ? ca_launch<64, 8, FO>(q, k_cache, v_cache, n_head, n_head_kv, cache_stride, kv_len, st, out, fo,
                                           pdl, err, s, stamp)
                    : ca_launch<64, 4, FO>(q, k_cache, v_cache, n_head, n_head_kv, cache_stride, kv_len, st, out, fo,
                                           pdl, err, s, stamp);
    if (head_dim == 128)
        return wide ? ca_launch<128, 8, FO>(q, k_cache, v_cache, n_head, n_head_kv, cache_stride, kv_len, st, out,
                                            fo, pdl, err, s, stamp)
                    : ca_launch<128, 4, FO>(q, k_cache, v_cache, n_head, n_head_kv, cache_stride, kv_len, st, out,
                                            fo, pdl, err, s, stamp);
    return cudaErrorInvalidValue;
}

cudaError_t launch_attn_decode_cluster(const float* q, const float* k_cache, const float* v_cache, int n_head,
                                       int n_head_kv, int head_dim, int cache_stride, int kv_len,
                                       const DevState* st, float* out, bool pdl, int* err, cudaStream_t s,
                                       unsigned long long* stamp) {
    return ca_dispatch<false>(q, k_cache, v_cache, n_head, n_head_kv, head_dim, cache_stride, kv_len, st, out,
                              nullptr, pdl, err, s, stamp);
}

// The O projection fits the decode attention kernel when every CTA's W_o
// slice (its 32-row tiles x the group's column blocks) is at most 32 KB and
// the shared-memory plan fits.
bool attn_oproj_fused_supported(int n_head, int n_kv, int head_dim, const PackedQ8& Wo) {
    if (n_kv <= 0 || n_head % n_kv || n_head / n_kv > kMaxGroup) return false;
    if (head_dim != 64 && head_dim != 128) return false;
    if (Wo.k != n_head * head_dim) return false;
    const int G = n_head / n_kv, GP = ca_group_pad(G);
    for (int cl : {16, 8}) {
        const int wo = fo_wo_bytes(Wo.rows_pad, G, head_dim, cl);
        if (wo > kFoMaxWoBytes) return false;
        const int floats = head_dim == 64 ? ca_plan<64>(G, GP, cl, wo).floats : ca_plan<128>(G, GP, cl, wo).floats;
        if ((size_t)floats * 4 > (size_t)kCaSmemLimit) return false;
    }
    return true;
}

cudaError_t launch_attn_oproj(const float* q, const float* k_cache, const float* v_cache, int n_head, int n_head_kv,
                              int head_dim, int cache_stride, const DevState* st, const PackedQ8& Wo, float* part,
                              int part_stride, bool pdl, int* err, cudaStream_t s, unsigned long long* stamp) {
    if (!st) return cudaErrorInvalidValue;
    const AttnOproj fo{Wo, part, part_stride, nullptr};
    return ca_dispatch<true>(q, k_cache, v_cache, n_head, n_head_kv, head_dim, cache_stride, 0, st, nullptr, &fo,
                             pdl, err, s, stamp);
}

// ---- fused layer front: host side --------------------------------------------------------
template <int HD, int CL, int GP>
static cudaLaunchConfig_t front_config(const FrontArgs& fa, cudaStream_t s, cudaLaunchAttribute* attrs, bool pdl) {
    const int G = fa.n_head / fa.n_kv;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(fa.n_kv * CL);
    cfg.blockDim = dim3(kCaThreads);
    cfg.dynamicSmemBytes =
        (size_t)front_plan<HD>(G, GP, CL, fa.wqkv.k, fo_wo_bytes(fa.wo.rows_pad, G, HD, CL)).floats * 4;
    cfg.stream = s;
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = CL;
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
    return cfg;
}

template <int HD, int CL, int GP>
static cudaError_t front_set_attrs() {
    cudaError_t e = cudaFuncSetAttribute(layer_front_cluster_kernel<HD, CL, GP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kCaSmemLimit);
    if (e == cudaSuccess && CL > 8)
        e = cudaFuncSetAttribute(layer_front_cluster_kernel<HD, CL, GP>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}
static bool g_front_ok = false;

// Cluster size for the fused front (16 when all KV heads' clusters fit at
// once), or 0 when the model does not fit the kernel.
template <int HD, int GP>
static int front_cluster_t(const FrontArgs& fa) {
    if (!g_front_ok) return 0;
    const int G = fa.n_head / fa.n_kv, h = fa.wqkv.k;
    for (int cl : {16, 8}) {
        if (cl == 16 && !g_ca16_ok) continue;
        if (front_wq_bytes(G, HD, h, cl) > 48 * 1024 || fo_wo_bytes(fa.wo.rows_pad, G, HD, cl) > kFoMaxWoBytes)
            continue;
        const size_t smem = (size_t)front_plan<HD>(G, GP, cl, h, fo_wo_bytes(fa.wo.rows_pad, G, HD, cl)).floats * 4;
        if (smem > (size_t)kCaSmemLimit) continue;
        cudaLaunchAttribute attrs[2];
        int n = 0;
        cudaError_t e;
        if (cl == 16) {
            cudaLaunchConfig_t cfg = front_config<HD, 16, GP>(fa, 0, attrs, false);
            e = cudaOccupancyMaxActiveClusters(&n, layer_front_cluster_kernel<HD, 16, GP>, &cfg);
        } else {
            cudaLaunchConfig_t cfg = front_config<HD, 8, GP>(fa, 0, attrs, false);
            e = cudaOccupancyMaxActiveClusters(&n, layer_front_cluster_kernel<HD, 8, GP>, &cfg);
        }
        if (e != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (n >= fa.n_kv) return cl;
    }
    return 0;
}

int layer_front_cluster_size(const FrontArgs& fa, int head_dim) {
    if (fa.n_kv <= 0 || fa.n_head % fa.n_kv || fa.n_head / fa.n_kv > kMaxGroup) return 0;
    if (fa.wo.k != fa.n_head * head_dim || (fa.n_head / fa.n_kv) * head_dim % 32) return 0;
    const bool wide = fa.n_head / fa.n_kv > 4;
    if (head_dim == 64) return wide ? front_cluster_t<64, 8>(fa) : front_cluster_t<64, 4>(fa);
    if (head_dim == 128) return wide ? front_cluster_t<128, 8>(fa) : front_cluster_t<128, 4>(fa);
    return 0;
}

template <int HD, int GP>
static cudaError_t front_launch_t(const FrontArgs& fa, int cl, bool pdl, cudaStream_t s) {
    cudaLaunchAttribute attrs[2];
    if (cl == 16) {
        cudaLaunchConfig_t cfg = front_config<HD, 16, GP>(fa, s, attrs, pdl);
        return cudaLaunchKernelEx(&cfg, layer_front_cluster_kernel<HD, 16, GP>, fa);
    }
    cudaLaunchConfig_t cfg = front_config<HD, 8, GP>(fa, s, attrs, pdl);
    return cudaLaunchKernelEx(&cfg, layer_front_cluster_kernel<HD, 8, GP>, fa);
}

cudaError_t launch_layer_front(const FrontArgs& fa, int head_dim, int cl, bool pdl, cudaStream_t s) {
    if (!fa.st || (cl != 16 && cl != 8)) return cudaErrorInvalidValue;
    const bool wide = fa.n_head / fa.n_kv > 4;
    if (head_dim == 64) return wide ? front_launch_t<64, 8>(fa, cl, pdl, s) : front_launch_t<64, 4>(fa, cl, pdl, s);
    if (head_dim == 128) return wide ? front_launch_t<128, 8>(fa, cl, pdl, s) : front_launch_t<128, 4>(fa, cl, pdl, s);
    return cudaErrorInvalidValue;
}

cudaError_t init_attn_prefill_attributes();

cudaError_t init_attention_attributes() {
    cudaError_t err = cudaFuncSetAttribute(attn_decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)decode_smem_bytes(64));
    if (err != cudaSuccess) return err;
    if ((err = init_attn_prefill_attributes()) != cudaSuccess) return err;
    err = cudaFuncSetAttribute(attn_decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)decode_smem_bytes(128));
    if (err != cudaSuccess) return err;
    if ((err = ca_set_attrs<64, 8, 4, false>()) != cudaSuccess) return err;
    if ((err = ca_set_attrs<64, 8, 8, false>()) != cudaSuccess) return err;
    if ((err = ca_set_attrs<128, 8, 4, false>()) != cudaSuccess) return err;
    if ((err = ca_set_attrs<128, 8, 8, false>()) != cudaSuccess) return err;
    if ((err = ca_set_attrs<64, 8, 4, true>()) != cudaSuccess) return err;
    if ((err = ca_set_attrs<64, 8, 8, true>()) != cudaSuccess) return err;
    if ((err = ca_set_attrs<128, 8, 4, true>()) != cudaSuccess) return err;
    if ((err = ca_set_attrs<128, 8, 8, true>()) != cudaSuccess) return err;
    g_ca16_ok = ca_set_attrs<64, 16, 4, false>() == cudaSuccess && ca_set_attrs<64, 16, 8, false>() == cudaSuccess &&
                ca_set_attrs<128, 16, 4, false>() == cudaSuccess && ca_set_attrs<128, 16, 8, false>() == cudaSuccess &&
                ca_set_attrs<64, 16, 4, true>() == cudaSuccess && ca_set_attrs<64, 16, 8, true>() == cudaSuccess &&
                ca_set_attrs<128, 16, 4, true>() == cudaSuccess && ca_set_attrs<128, 16, 8, true>() == cudaSuccess;
    cudaGetLastError();
    g_front_ok = front_set_attrs<64, 8, 4>() == cudaSuccess && front_set_attrs<64, 8, 8>() == cudaSuccess &&
                 front_set_attrs<128, 8, 4>() == cudaSuccess && front_set_attrs<128, 8, 8>() == cudaSuccess &&
                 front_set_attrs<64, 16, 4>() == cudaSuccess && front_set_attrs<64, 16, 8>() == cudaSuccess &&
                 front_set_attrs<128, 16, 4>() == cudaSuccess && front_set_attrs<128, 16, 8>() == cudaSuccess;
    cudaGetLastError();
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// Prefill
// ---------------------------------------------------------------------------
// Causal attention for T > 1 rows ("量化 llama 的一次前向", forward：mask 什么时候建):
// query t (position index_pos + t) sees cache positions j <= index_pos + t.
// CTA = one query head x R = 16 * RT query rows, 256 threads as a 16 x 16 grid
// (ty = tid / 16, tx = tid % 16). Per KV tile of KT positions:
//  - scores: thread (ty, tx) computes rows RT * ty + i (i < RT) against keys
//    tx + 16 k (k < KT / 16), q and k read as float4 from shared rows padded
//    by 4 floats (lanes tx = 0..7 hit distinct 16-byte bank groups);
//  - online softmax: a row's maximum is reduced over its 16 tx lanes (one
//    half-warp) with shuffles; the row sums stay per thread until the end;
//  - P = e^(s - m) goes to shared memory, read back only by the same half-warp
//    (the rows it owns), so a warp barrier suffices;
//  - output: thread (ty, tx) accumulates its RT rows x HD / 16 dims (float4
//    groups tx and tx + 16) over the tile's keys.
// K/V tiles are double-buffered with cp.async across the whole CTA.
// Key split (KS > 1, short prompts whose row tiles cannot fill the GPU): a
// cluster of KS CTAs shares one (head, row tile), rank z taking key tiles z,
// z + KS, ...; each keeps its unnormalised output, row maxima and row sums in
// shared memory, and rank 0 reads the peers' through distributed shared
// memory and merges them (weights e^(m_z - M)) before the division.
template <int HD, int RT>
struct PfCfg {
    static constexpr int R = 16 * RT;              // query rows per CTA
    static constexpr int KT = HD == 64 ? 64 : 32;  // positions per tile
    static constexpr int KPT = KT / 16;            // keys per thread (scores)
    static constexpr int DG = HD / 64;             // float4 dim groups per thread (output)
    static constexpr int LD = HD + 4;              // floats per q / k / v row in shared memory
    static constexpr int LDP = KT + 4;             // floats per P row
    static constexpr int kQ = 0, kK = R * LD, kV = kK + 2 * KT * LD, kP = kV + 2 * KT * LD;
    static constexpr size_t kSmem = (size_t)(kP + R * LDP) * sizeof(float);
    // key split: this CTA's unnormalised output rows, row maxima and row sums,
    // in the K/V stages (free once the last key tile has been used)
    static constexpr int kMO = kK, kMM = kMO + R * HD, kML = kMM + R;
    static_assert(kML + R <= kP, "the merge buffers fit in the K/V stages");
    static constexpr size_t kSmemSplit = kSmem;
};
constexpr int kPfThreads = 256;

template <int HD, int RT, int KS>
__global__ void __launch_bounds__(kPfThreads, 2) attn_prefill_kernel(const float* __restrict__ q,
                                                                     const float* __restrict__ kc,
                                                                     const float* __restrict__ vc, int T,
                                                                     int index_pos, int n_head, int n_kv,
                                                                     int cache_stride, float scale,
                                                                     float* __restrict__ out) {
    using C = PfCfg<HD, RT>;
    constexpr int R = C::R, KT = C::KT, KPT = C::KPT, DG = C::DG, LD = C::LD, LDP = C::LDP;
    extern __shared__ __align__(16) float pf_smem[];
    float* Qs = pf_smem + C::kQ;
    float* Ps = pf_smem + C::kP;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    // z: rank in the key split; the last row tiles (the most visible keys) first
    const int h = blockIdx.x / KS, z = blockIdx.x % KS, t0 = (gridDim.y - 1 - blockIdx.y) * R;
    const int kh = h / (n_head / n_kv);
    const float* kbase = kc + (int64_t)kh * cache_stride * HD;
    const float* vbase = vc + (int64_t)kh * cache_stride * HD;
    const int kv_end = index_pos + min(T, t0 + R);
    const int n_tiles = (kv_end + KT - 1) / KT;
    const int n_mine = n_tiles > z ? (n_tiles - z + KS - 1) / KS : 0;  // key tiles z, z + KS, ...

    pdl_wait();
    pdl_launch_dependents();

    // copy this CTA's key tile number `it` (tile z + it * KS) of K and V into
    // stage `st` (positions past kv_end zero-filled)
    auto issue = [&](int it, int st) {
        if (it < n_mine) {
            const int t = z + it * KS;
            float* ks = pf_smem + C::kK + st * KT * LD;
            float* vs = pf_smem + C::kV + st * KT * LD;
            for (int f = tid; f < KT * (HD / 4); f += kPfThreads) {
                const int row = f / (HD / 4), cc = f % (HD / 4);
                const int j = t * KT + row;
                const bool ok = j < kv_end;
                const int64_t off = (int64_t)(ok ? j : 0) * HD + cc * 4;
                cp_async16(ks + row * LD + cc * 4, kbase + off, ok ? 16u : 0u);
                cp_async16(vs + row * LD + cc * 4, vbase + off, ok ? 16u : 0u);
            }
        }
        cp_async_commit();
    };
    issue(0, 0);
    // q rows of this CTA, pre-scaled by 1/sqrt(head_dim); rows past T are zero
    for (int f = tid; f < R * (HD / 4); f += kPfThreads) {
        const int row = f / (HD / 4), cc = f % (HD / 4);
        const int t = t0 + row;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < T) v = *reinterpret_cast<const float4*>(q + ((int64_t)t * n_head + h) * HD + cc * 4);
        v.x *= scale; v.y *= scale; v.z *= scale; v.w *= scale;
        *reinterpret_cast<float4*>(Qs + row * LD + cc * 4) = v;
    }

    float o[RT][DG][4], m[RT], l[RT];
#pragma unroll
    for (int i = 0; i < RT; ++i) {
        m[i] = -INFINITY;
        l[i] = 0.0f;
#pragma unroll
        for (int g = 0; g < DG; ++g) o[i][g][0] = o[i][g][1] = o[i][g][2] = o[i][g][3] = 0.0f;
    }

    for (int it = 0; it < n_mine; ++it) {
        const int t = z + it * KS;
        issue(it + 1, (it + 1) & 1);
        cp_async_wait<1>();
        __syncthreads();  // tile t (and, at the first tile, the q rows) visible to every thread
        const float* ks = pf_smem + C::kK + (it & 1) * KT * LD;
        const float* vs = pf_smem + C::kV + (it & 1) * KT * LD;
        float sc[RT][KPT];
#pragma unroll
        for (int i = 0; i < RT; ++i)
#pragma unroll
            for (int k = 0; k < KPT; ++k) sc[i][k] = 0.0f;
#pragma unroll 4
        for (int d = 0; d < HD; d += 4) {
            float4 qv[RT], kv[KPT];
#pragma unroll
            for (int i = 0; i < RT; ++i) qv[i] = *reinterpret_cast<const float4*>(Qs + (ty * RT + i) * LD + d);
#pragma unroll
            for (int k = 0; k < KPT; ++k) kv[k] = *reinterpret_cast<const float4*>(ks + (tx + 16 * k) * LD + d);
#pragma unroll
            for (int i = 0; i < RT; ++i)
#pragma unroll
                for (int k = 0; k < KPT; ++k) {
                    sc[i][k] = fmaf(qv[i].x, kv[k].x, sc[i][k]);
                    sc[i][k] = fmaf(qv[i].y, kv[k].y, sc[i][k]);
                    sc[i][k] = fmaf(qv[i].z, kv[k].z, sc[i][k]);
                    sc[i][k] = fmaf(qv[i].w, kv[k].w, sc[i][k]);
                }
        }
        // mask, row maxima over the half-warp, P into shared memory
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            const int row = ty * RT + i;
            const int last = index_pos + t0 + row;  // last visible position of this row
            const bool row_ok = t0 + row < T;
            float mt = -INFINITY;
#pragma unroll
            for (int k = 0; k < KPT; ++k) {
                const int j = t * KT + tx + 16 * k;
                if (!(row_ok && j <= last && j < kv_end)) sc[i][k] = -INFINITY;
                mt = fmaxf(mt, sc[i][k]);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, off));
            const float m_new = fmaxf(m[i], mt);
            const float corr = m_new == -INFINITY ? 1.0f : expf(m[i] - m_new);
            float ps = 0.0f;
#pragma unroll
            for (int k = 0; k < KPT; ++k) {
                const float pk = m_new == -INFINITY ? 0.0f : expf(sc[i][k] - m_new);
                ps += pk;
                Ps[row * LDP + tx + 16 * k] = pk;
            }
            l[i] = l[i] * corr + ps;
            m[i] = m_new;
#pragma unroll
            for (int g = 0; g < DG; ++g) {
                o[i][g][0] *= corr; o[i][g][1] *= corr; o[i][g][2] *= corr; o[i][g][3] *= corr;
            }
        }
        __syncwarp();  // a half-warp reads back only the P rows it wrote
#pragma unroll 2
        for (int j = 0; j < KT; j += 4) {
            float4 pv[RT];
#pragma unroll
            for (int i = 0; i < RT; ++i) pv[i] = *reinterpret_cast<const float4*>(Ps + (ty * RT + i) * LDP + j);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                for (int g = 0; g < DG; ++g) {
                    const float4 vv = *reinterpret_cast<const float4*>(vs + (j + jj) * LD + (tx + 16 * g) * 4);
#pragma unroll
                    for (int i = 0; i < RT; ++i) {
                        const float pj = jj == 0 ? pv[i].x : (jj == 1 ? pv[i].y : (jj == 2 ? pv[i].z : pv[i].w));
                        o[i][g][0] = fmaf(pj, vv.x, o[i][g][0]);
                        o[i][g][1] = fmaf(pj, vv.y, o[i][g][1]);
                        o[i][g][2] = fmaf(pj, vv.z, o[i][g][2]);
                        o[i][g][3] = fmaf(pj, vv.w, o[i][g][3]);
                    }
                }
            }
        }
        __syncthreads();  // the stage and P are read before they are refilled
    }
    cp_async_wait<0>();
    // row sums over the half-warp
#pragma unroll
    for (int i = 0; i < RT; ++i) {
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) l[i] += __shfl_xor_sync(0xffffffffu, l[i], off);
    }
    if (KS > 1) {
        // key split: every rank leaves (o, m, l) in its shared memory; rank 0
        // merges the peers' into its registers, the others are done after the
        // second cluster barrier (which keeps their shared memory until rank 0
        // has read it)
        float* MO = pf_smem + C::kMO;
        float* MM = pf_smem + C::kMM;
        float* ML = pf_smem + C::kML;
        __syncthreads();  // every thread is done with the stages the buffers reuse
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            const int row = ty * RT + i;
#pragma unroll
            for (int g = 0; g < DG; ++g)
                *reinterpret_cast<float4*>(MO + row * HD + (tx + 16 * g) * 4) =
                    make_float4(o[i][g][0], o[i][g][1], o[i][g][2], o[i][g][3]);
            if (tx == 0) {
                MM[row] = m[i];
                ML[row] = l[i];
            }
        }
        cluster_sync();
        if (z == 0) {
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                const int row = ty * RT + i;
                float mz[KS];
                mz[0] = m[i];
                float mx = m[i];
#pragma unroll
                for (int r = 1; r < KS; ++r) {
                    mz[r] = ld_dsmem_f32(MM + row, (uint32_t)r);
                    mx = fmaxf(mx, mz[r]);
                }
                // weights e^(m_r - M); a rank that saw no visible key has m = -inf
                const float w0 = m[i] == -INFINITY ? 0.0f : expf(m[i] - mx);
                l[i] *= w0;
#pragma unroll
                for (int g = 0; g < DG; ++g) {
                    o[i][g][0] *= w0; o[i][g][1] *= w0; o[i][g][2] *= w0; o[i][g][3] *= w0;
                }
#pragma unroll
                for (int r = 1; r < KS; ++r) {
                    const float wr = mz[r] == -INFINITY ? 0.0f : expf(mz[r] - mx);
                    l[i] = fmaf(wr, ld_dsmem_f32(ML + row, (uint32_t)r), l[i]);
#pragma unroll
                    for (int g = 0; g < DG; ++g) {
                        const float4 v = ld_dsmem_f32x4(MO + row * HD + (tx + 16 * g) * 4, (uint32_t)r);
                        o[i][g][0] = fmaf(wr, v.x, o[i][g][0]);
                        o[i][g][1] = fmaf(wr, v.y, o[i][g][1]);
                        o[i][g][2] = fmaf(wr, v.z, o[i][g][2]);
                        o[i][g][3] = fmaf(wr, v.w, o[i][g][3]);
                    }
                }
            }
        }
        cluster_sync();
        if (z != 0) return;
    }
    // o / l
#pragma unroll
    for (int i = 0; i < RT; ++i) {
        const int t = t0 + ty * RT + i;
        if (t < T) {
            const float inv = 1.0f / l[i];
#pragma unroll
            for (int g = 0; g < DG; ++g)
                *reinterpret_cast<float4*>(out + ((int64_t)t * n_head + h) * HD + (tx + 16 * g) * 4) =
                    make_float4(o[i][g][0] * inv, o[i][g][1] * inv, o[i][g][2] * inv, o[i][g][3] * inv);
        }
    }
}

template <int HD, int RT, int KS>
static cudaError_t pf_attr() {
    return cudaFuncSetAttribute(attn_prefill_kernel<HD, RT, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(KS > 1 ? PfCfg<HD, RT>::kSmemSplit : PfCfg<HD, RT>::kSmem));
}

template <int HD>
static cudaError_t pf_attr_hd() {
    cudaError_t err = pf_attr<HD, 4, 1>();
    if (err == cudaSuccess) err = pf_attr<HD, 4, 2>();
    if (err == cudaSuccess) err = pf_attr<HD, 1, 1>();
    if (err == cudaSuccess) err = pf_attr<HD, 1, 2>();
    if (err == cudaSuccess) err = pf_attr<HD, 1, 4>();
    if (err == cudaSuccess) err = pf_attr<HD, 1, 8>();
    return err;
}

cudaError_t init_attn_prefill_attributes() {
    cudaError_t err = pf_attr_hd<64>();
    if (err == cudaSuccess) err = pf_attr_hd<128>();
    return err;
}

template <int HD, int RT, int KS>
static cudaError_t pf_launch(const float* q, const float* k_cache, const float* v_cache, int T, int index_pos,
                             int n_head, int n_head_kv, int cache_stride, float* out, bool pdl, cudaStream_t s) {
    constexpr int R = PfCfg<HD, RT>::R;
    const float scale = 1.0f / sqrtf((float)HD);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n_head * KS, (T + R - 1) / R);
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = KS > 1 ? PfCfg<HD, RT>::kSmemSplit : PfCfg<HD, RT>::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int n = 0;
    if (KS > 1) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = KS;
        attrs[n].val.clusterDim.y = 1;
        attrs[n].val.clusterDim.z = 1;
        ++n;
    }
    if (pdl) {
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<HD, RT, KS>, q, k_cache, v_cache, T, index_pos, n_head,
                              n_head_kv, cache_stride, scale, out);
}

template <int HD>
static cudaError_t pf_dispatch(const float* q, const float* k_cache, const float* v_cache, int T, int index_pos,
                               int n_head, int n_head_kv, int cache_stride, float* out, bool pdl, cudaStream_t s,
                               int sms) {
    // 64 rows per CTA when that still gives every SM a CTA; their keys split
    // over a cluster of 2 when the doubled grid stays within two waves of two
    // resident CTAs per SM (under a causal mask the last row tiles see the
    // most keys: in one wave they alone would set the time). Else 16 rows,
    // and when even those leave SMs idle, each row tile's keys split over a
    // cluster of 2, 4 or 8 CTAs (two resident per SM, at least one key tile
    // each)
    const int64_t ctas64 = (int64_t)n_head * ((T + 63) / 64);
    if (ctas64 >= sms) {
        const int tiles64 = (index_pos + T + PfCfg<HD, 4>::KT - 1) / PfCfg<HD, 4>::KT;
        if (ctas64 * 2 <= 4 * (int64_t)sms && tiles64 >= 4)
            return pf_launch<HD, 4, 2>(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, cache_stride, out, pdl, s);
        return pf_launch<HD, 4, 1>(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, cache_stride, out, pdl, s);
    }
    const int64_t ctas = (int64_t)n_head * ((T + 15) / 16);
    const int tiles = (index_pos + T + PfCfg<HD, 1>::KT - 1) / PfCfg<HD, 1>::KT;
    int ks = 1;
    while (ks < 8 && ctas * ks * 2 <= 2 * (int64_t)sms && tiles >= ks * 2) ks *= 2;
    switch (ks) {
        case 2: return pf_launch<HD, 1, 2>(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, cache_stride, out, pdl, s);
        case 4: return pf_launch<HD, 1, 4>(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, cache_stride, out, pdl, s);
        case 8: return pf_launch<HD, 1, 8>(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, cache_stride, out, pdl, s);
    }
    return pf_launch<HD, 1, 1>(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, cache_stride, out, pdl, s);
}

cudaError_t launch_attn_prefill(const float* q, const float* k_cache, const float* v_cache, int T,
                                int index_pos, int n_head, int n_head_kv, int head_dim, int cache_stride,
                                float* out, bool pdl, cudaStream_t s) {
    static int sms = 0;
    if (sms <= 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 148;
    }
    if (head_dim == 64)
        return pf_dispatch<64>(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, cache_stride, out, pdl, s, sms);
    if (head_dim == 128)
        return pf_dispatch<128>(q, k_cache, v_cache, T, index_pos, n_head, n_head_kv, cache_stride, out, pdl, s, sms);
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
        err = ensure_kernel_attributes();
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
    // the kernel reads q, K and V and writes out as 16-byte vectors
    if (((uintptr_t)q | (uintptr_t)k_cache | (uintptr_t)v_cache | (uintptr_t)out) & 15) return LQ8_ERR_ARG;
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
