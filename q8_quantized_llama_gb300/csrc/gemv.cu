// Q8_0 matrix-vector product for one token (decode, and the lm_head of every
// forward): the counterpart of the quantised mat-vec kernel the pages name on
// "生成一个 token" (prefill 和 decode：同一个 forward，不同的路), written for
// sm_103a.
//
// Work unit: one tile of 32 output rows x a contiguous range of 32-weight
// blocks. In the packed layout that range is one contiguous run of codes
// (1 KiB per block) and one of scales (64 B per block), so a producer warp
// streams it into a ring of shared-memory stages with bulk async copies
// (8 blocks per stage, completion counted on an mbarrier). Eight consumer
// warps take one block each per stage: lane l owns row tile*32 + l and reads
// its 2 x 16 codes with conflict-free 128-bit shared loads. Codes become f32
// exactly (byte-permute into 2^23 + u, one packed subtraction per pair) and
// are multiplied into f32x2 accumulators against the activation vector
// staged in shared memory (normalised there when RMSNorm is fused). When the
// tile count alone cannot fill the GPU, the block range is split over a
// cluster of CTAs and the leader adds its peers' partial sums through
// distributed shared memory, in rank order (deterministic).
//
// Programmatic dependent launch: the producer starts streaming weights (which
// no kernel writes) before the grid waits on its predecessor, so the weight
// reads of a decode step overlap the tail of the previous kernel.
#include <algorithm>
#include <map>
#include <mutex>

#include "epilogue.cuh"
#include "ptx.cuh"

namespace lq8 {

constexpr int kCWarps = 8;                        // consumer warps
constexpr int kGemvThreads = (kCWarps + 1) * 32;  // + one producer warp
// Ring shape: stages x blocks per stage (a multiple of kCWarps). Matrices
// with many row tiles stream best through 3 stages of 16 blocks (three CTAs
// per SM); those split over clusters (few tiles) through 2 stages of 32.
template <int STAGES, int SBLK>
struct Ring {
    static constexpr int kStages = STAGES;
    static constexpr int kStageBlocks = SBLK;
    static constexpr int kStageCodeBytes = SBLK * 1024;
    static constexpr int kStageBytes = kStageCodeBytes + SBLK * 64;
    static constexpr int kCtasPerSm = (227 * 1024) / (STAGES * kStageBytes + 16 * 1024 + 2048);
};
using RingWide = Ring<3, 16>;
using RingDeep = Ring<2, 32>;
constexpr int kGemvMaxSmem = 227 * 1024 - 4096;

struct GemvArgs {
    PackedQ8 W;
    const float* x;
    const float* g;  // RMSNorm weight when the norm is fused, else unused
    float eps;
    EpiArgs e;
    int splits;      // CTAs (one cluster) per tile
    int* err;        // set on a bounded-wait timeout
    GemvPreSum pre;  // fused norm only: partials added to x first
};

__device__ __forceinline__ float block_dot32(const uint4& q0, const uint4& q1, const float* xs) {
    const float4* x4 = reinterpret_cast<const float4*>(xs);
    uint64_t a0 = 0, a1 = 0;
    a0 = dot4_acc(q0.x, x4[0], a0);
    a1 = dot4_acc(q1.x, x4[4], a1);
    a0 = dot4_acc(q0.y, x4[1], a0);
    a1 = dot4_acc(q1.y, x4[5], a1);
    a0 = dot4_acc(q0.z, x4[2], a0);
    a1 = dot4_acc(q1.z, x4[6], a1);
    a0 = dot4_acc(q0.w, x4[3], a0);
    a1 = dot4_acc(q1.w, x4[7], a1);
    return (f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1));
}

// Epilogue on the 32 rows of a tile (warp-wide; lane = row within the tile).
// pre: for EPI_RESIDUAL, the residual value of this lane's row, read before
// the tile's products so that its latency overlaps them. For EPI_ARGMAX the
// logits are stored and the tile's best packed key (value, lowest index) is
// folded into *best (warp-uniform); the CTA publishes it once at the end.
template <int EPI>
__device__ __forceinline__ void gemv_epilogue(const EpiArgs& e, int rows, int tile, int lane, float v, float pre,
                                              unsigned long long* best, float2 cs) {
    const int r = tile * 32 + lane;
    const bool valid = r < rows;
    if (EPI == EPI_STORE) {
        if (valid) e.y[r] = v;
    } else if (EPI == EPI_RESIDUAL) {
        if (valid) e.y[r] = pre + v;
    } else if (EPI == EPI_QKV) {
        const float other = __shfl_xor_sync(0xffffffffu, v, 1);
        const int pos = e.state ? e.state->pos : e.pos0;
        if (!(lane & 1) && valid) epi_qkv_pair_cs(e, 0, pos, r, v, other, cs);
    } else if (EPI == EPI_SILU) {
        const float up = __shfl_xor_sync(0xffffffffu, v, 1);
        if (!(lane & 1) && valid) e.a_out[r >> 1] = silu_f32(v) * up;
    } else if (EPI == EPI_ARGMAX) {
        if (valid) e.logits[r] = v;
        unsigned long long key = valid ? argmax_key(v, r) : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
            key = other > key ? other : key;
        }
        *best = key > *best ? key : *best;
    }
}

// Greedy token: every publishing CTA raises the shared maximum key, then takes
// a ticket with release semantics (ordering its maximum before the ticket, no
// separate fence); the CTA holding the last ticket (acquire: it sees every
// maximum) reads the key, resets both accumulators for the next launch with
// plain stores (the kernel boundary orders them before it) and writes the
// token and position to the step state. One thread.
__device__ __forceinline__ void argmax_publish(const EpiArgs& e, unsigned long long best, unsigned int n_pub) {
    atomicMax(e.best_key, best);
    unsigned int ticket;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(ticket) : "l"(e.done_count) : "memory");
    if (ticket == n_pub - 1) {
        unsigned long long key;
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(key) : "l"(e.best_key) : "memory");
        *e.best_key = 0ull;
        *e.done_count = 0u;
        const int tok = argmax_key_index(key);
        DevState* st = e.st;
        st->token = tok;
        if (e.out_ids) e.out_ids[st->n_out] = tok;
        st->n_out += 1;
        st->pos = e.pos_after >= 0 ? e.pos_after : st->pos + 1;
    }
}

// Grid: with S == 1 a persistent set of CTAs (at most what is resident at
// once), each taking row tiles blockIdx.x, blockIdx.x + gridDim.x, ... and
// streaming their weights through one continuous ring; with S > 1 one cluster
// of S CTAs per tile, rank r taking the r-th part of the block range.
template <int EPI, bool NORM, typename RG>
__global__ void __launch_bounds__(kGemvThreads) q8_gemv_kernel(GemvArgs a) {
    constexpr int kStages = RG::kStages, kStageBlocks = RG::kStageBlocks;
    constexpr int kStageCodeBytes = RG::kStageCodeBytes, kStageBytes = RG::kStageBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    float* xs = reinterpret_cast<float*>(smem + kStages * kStageBytes);
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ __align__(8) uint64_t empty[kStages];
    __shared__ __align__(8) uint64_t xbar;
    __shared__ float red[2][kCWarps][32];  // per-warp tile sums, by tile parity
    __shared__ float ssq[kCWarps];          // per-warp sums of squares (fused norm)
    __shared__ float part[32];

    const PackedQ8& W = a.W;
    const int k = W.k, nb = k >> 5;
    const int S = a.splits;
    const int tiles = W.rows_pad >> 5;
    const int cl_id = blockIdx.x / S, split = blockIdx.x % S, n_cl = gridDim.x / S;
    const int my_tiles = cl_id < tiles ? (tiles - cl_id + n_cl - 1) / n_cl : 0;
    const int b0 = (split * nb) / S, b1 = ((split + 1) * nb) / S;
    const int nblk = b1 - b0;
    const int n_stage = (nblk + kStageBlocks - 1) / kStageBlocks;  // per tile
    const int total = my_tiles * n_stage;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) stamp_at(a.e.stamp, 0);

    // The activation vector goes to shared memory by one bulk copy issued after
    // the grid dependency wait: the whole vector when the fused RMSNorm needs
    // all of it on a split unit, else only this unit's slice.
    const bool x_full = NORM && S > 1;
    const int x0 = b0 * 32, xn = nblk * 32;
    float* xslice = x_full ? xs + x0 : xs;
    const int np = NORM ? a.pre.n_part : 0;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCWarps);
        }
        mbar_init(&xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCWarps) {
        // ---- producer: stream the codes and scales of every tile of this CTA ----
        if (lane == 0) {
            const uint8_t* qs = reinterpret_cast<const uint8_t*>(W.qs);
            const uint8_t* ds = reinterpret_cast<const uint8_t*>(W.d);
            auto issue_stage = [&](int g) {
                const int slot = g % kStages;
                if (g >= kStages) mbar_wait_bounded(&empty[slot], ((g / kStages) - 1) & 1, a.err, 9);
                const int tile = cl_id + (g / n_stage) * n_cl, j = g % n_stage;
                const int bs = b0 + j * kStageBlocks;
                const int nbs = min(kStageBlocks, b1 - bs);
                uint8_t* dst = stages + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(nbs * 1024 + nbs * 64));
                bulk_g2s(dst, qs + (size_t)tile * k * 32 + (size_t)bs * 1024, nbs * 1024, &full[slot]);
                bulk_g2s(dst + kStageCodeBytes, ds + (size_t)tile * nb * 64 + (size_t)bs * 64, nbs * 64,
                         &full[slot]);
            };
            const int first = min(kStages, total);
            for (int g = 0; g < first; ++g) issue_stage(g);  // weights: no kernel writes them
            pdl_wait();                                      // x: written by the preceding kernel
            const int xoff = x_full ? 0 : x0, xcnt = x_full ? k : xn;
            mbar_arrive_expect_tx(&xbar, (uint32_t)(xcnt * 4 * (1 + np)));
            bulk_g2s(xs, a.x + xoff, (uint32_t)(xcnt * 4), &xbar);
            for (int p = 0; p < np; ++p)
                bulk_g2s(xs + (size_t)(p + 1) * k, a.pre.part + (size_t)p * a.pre.part_stride, (uint32_t)(k * 4),
                         &xbar);
            for (int g = first; g < total; ++g) issue_stage(g);
        }
    } else {
        // ---- consumers --------------------------------------------------------
        // The norm weight is constant: each thread loads its float4s of the
        // slice before the dependency wait (up to 4 per thread; k <= 4096).
        constexpr int kGPre = 4;
        float4 gpre[kGPre];
        if (NORM) {
#pragma unroll
            for (int u = 0; u < kGPre; ++u) {
                const int i = threadIdx.x * 4 + u * kCWarps * 32 * 4;
                gpre[u] = i < xn ? *reinterpret_cast<const float4*>(a.g + x0 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        // QKV: the rotary (cos, sin) of the first tile's row pairs, before the wait
        // (the table is constant and the position was written two or more launches back)
        float2 cs = make_float2(1.0f, 0.0f);
        const int qkv_pos = (EPI == EPI_QKV) ? (a.e.state ? a.e.state->pos : a.e.pos0) : 0;
        if (EPI == EPI_QKV && warp == 0 && split == 0 && my_tiles > 0 && cl_id * 32 + lane < W.rows)
            cs = rope_cs_for_row(a.e, qkv_pos, (cl_id * 32 + lane) & ~1);
        pdl_wait();
        if (tid == 0) {
            pdl_launch_dependents();
            stamp_at(a.e.stamp, 1);
        }
        constexpr int kCT = kCWarps * 32;
        mbar_wait_bounded(&xbar, 0, a.err, 13);
        float rscale = 1.0f;
        if (NORM) {
            // x (+ the partials, in order) -> sum of squares for the scale, and x * g in
            // place; the scale 1/rms multiplies the finished dot products in the epilogue,
            // so no barrier waits on the reduction before the products start.
            const int nx = x_full ? k : xn;  // == k when unsplit
            const bool keep = blockIdx.x == 0 && a.pre.x_sum_out != nullptr;
            float ss = 0.0f;
            for (int i = tid * 4, u = 0; i < nx; i += kCT * 4, ++u) {
                float4 v = *reinterpret_cast<const float4*>(xs + i);
                for (int p = 0; p < np; ++p) {
                    const float4 w = *reinterpret_cast<const float4*>(xs + (size_t)(p + 1) * k + i);
                    v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
                }
                if (keep) *reinterpret_cast<float4*>(a.pre.x_sum_out + i) = v;
                ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
                if (!x_full) {  // unsplit: this thread's elements are the ones it scales
                    float4 gg;
#pragma unroll
                    for (int w = 0; w < kGPre; ++w)
                        if (w == u) gg = gpre[w];
                    if (u >= kGPre) gg = *reinterpret_cast<const float4*>(a.g + i);
                    v.x *= gg.x; v.y *= gg.y; v.z *= gg.z; v.w *= gg.w;
                }
                *reinterpret_cast<float4*>(xs + i) = v;
            }
            ss = warp_sum(ss);
            if (lane == 0) ssq[warp] = ss;
            named_bar_sync(1, kCT);
            if (x_full) {  // split unit: scale this unit's slice after every sum has landed
                for (int i = tid * 4, u = 0; i < xn; i += kCT * 4, ++u) {
                    float4 v = *reinterpret_cast<float4*>(xslice + i);
                    float4 gg;
#pragma unroll
                    for (int w = 0; w < kGPre; ++w)
                        if (w == u) gg = gpre[w];
                    if (u >= kGPre) gg = *reinterpret_cast<const float4*>(a.g + x0 + i);
                    v.x *= gg.x; v.y *= gg.y; v.z *= gg.z; v.w *= gg.w;
                    *reinterpret_cast<float4*>(xslice + i) = v;
                }
                named_bar_sync(1, kCT);
            }
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < kCWarps; ++w) t += ssq[w];
            rscale = 1.0f / sqrtf(t / (float)k + a.eps);
        }

        unsigned long long best = 0ull;  // EPI_ARGMAX, warp 0
        float res_pre = 0.0f;            // EPI_RESIDUAL: residual of the row this lane finishes
        for (int ti = 0; ti < my_tiles; ++ti) {
            const int tile = cl_id + ti * n_cl;
            if (EPI == EPI_RESIDUAL && split == 0 && warp == 0) {
                const int r = tile * 32 + lane;
                if (r < W.rows) res_pre = a.e.res ? a.e.res[r] : a.e.y[r];
            }
            if (EPI == EPI_QKV && ti > 0 && split == 0 && warp == 0 && tile * 32 + lane < W.rows)
                cs = rope_cs_for_row(a.e, qkv_pos, (tile * 32 + lane) & ~1);  // used after the tile's products
            float acc = 0.0f;
            for (int j = 0; j < n_stage; ++j) {
                const int g = ti * n_stage + j;
                const int slot = g % kStages;
                mbar_wait_bounded(&full[slot], (g / kStages) & 1, a.err, 10);
                const int bs = j * kStageBlocks;  // relative to b0
                const int nbs = min(kStageBlocks, nblk - bs);
                const uint8_t* st = stages + slot * kStageBytes;
#pragma unroll
                for (int bi = warp; bi < kStageBlocks; bi += kCWarps) {
                    if (bi < nbs) {
                        const uint4 q0 = *reinterpret_cast<const uint4*>(st + bi * 1024 + lane * 16);
                        const uint4 q1 = *reinterpret_cast<const uint4*>(st + bi * 1024 + 512 + lane * 16);
                        const float d =
                            __half2float(reinterpret_cast<const __half*>(st + kStageCodeBytes)[bi * 32 + lane]);
                        acc = fmaf(d, block_dot32(q0, q1, xslice + (bs + bi) * 32), acc);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[slot]);
            }
            red[ti & 1][warp][lane] = acc;
            named_bar_sync(1, kCT);
            if (warp == 0) {
                float v = 0.0f;
#pragma unroll
                for (int w = 0; w < kCWarps; ++w) v += red[ti & 1][w][lane];
                if (S == 1)
                    gemv_epilogue<EPI>(a.e, W.rows, tile, lane, NORM ? v * rscale : v, res_pre, &best, cs);
                else
                    part[lane] = v;  // one tile per cluster: reduced below
            }
        }
        if (S > 1) {
            // ---- cluster reduction and epilogue (one tile per cluster) -------------
            __syncwarp();
            cluster_sync();
            if (split == 0 && warp == 0 && my_tiles > 0) {
                float v = part[lane];
                for (int rnk = 1; rnk < S; ++rnk) v += ld_dsmem_f32(&part[lane], (uint32_t)rnk);
                gemv_epilogue<EPI>(a.e, W.rows, cl_id, lane, NORM ? v * rscale : v, res_pre, &best, cs);
            }
            cluster_sync();  // peers keep their shared memory until the leader has read it
        }
        if (EPI == EPI_ARGMAX && split == 0 && tid == 0) argmax_publish(a.e, best, (unsigned)n_cl);
        return;
    }
    // the producer warp joins the cluster barriers of a split launch
    if (S > 1) {
        __syncwarp();
        cluster_sync();
        cluster_sync();
    }
}

// Splits per tile: enough CTAs to cover the GPU in one wave, at least 16
// blocks per split, at most 8 (a portable cluster).
static int gemv_splits(int tiles, int nb, int sm_count, int ctas_per_sm) {
    const int capacity = sm_count * ctas_per_sm;
    int s = 1;
    while (s < 8 && tiles * (s + 1) <= capacity && nb / (s + 1) >= 16) ++s;
    return s;
}

static int g_sm_count[64] = {};

static int sm_count_current() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!g_sm_count[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = n > 0 ? n : 148;
    }
    return g_sm_count[dev];
}

// ---------------------------------------------------------------------------
// Token rows on the CUDA cores (prefill chunks of 2..16 tokens, and small
// products of more rows in chunks of 16): the same weight stream, each 32-row
// tile read once per chunk and multiplied with every token row of the chunk.
// Lane = weight row; per 32-weight block the lane turns its codes into f32
// once and takes the dot product with each token's x block (broadcast
// shared-memory reads). Grid: x = (tile, split), y = 16-token chunk; the block
// range of a tile split over a cluster when the CTAs cannot fill the GPU or the
// chunk's slices of x would not fit in shared memory; the leader adds the
// peers' partial sums in rank order.
// ---------------------------------------------------------------------------
constexpr int kRowsMax = 16;
// dynamic shared memory of the few-rows kernel, beside its ~19 KB of static arrays
constexpr int kRowsMaxSmem = 200 * 1024;

struct GemvRowsArgs {
    PackedQ8 W;
    const float* X;  // [m][ldx]
    int m, ldx;
    EpiArgs e;
    int splits;
    int* err;
};

template <int EPI>
__device__ __forceinline__ void rows_epilogue(const EpiArgs& e, int rows, int tile, int lane, int t, float v) {
    const int r = tile * 32 + lane;
    const bool valid = r < rows;
    if (EPI == EPI_STORE) {
        if (valid) e.y[(int64_t)t * e.ldy + r] = v;
    } else if (EPI == EPI_RESIDUAL) {
        if (valid) e.y[(int64_t)t * e.ldy + r] += v;
    } else if (EPI == EPI_QKV) {
        const float other = __shfl_xor_sync(0xffffffffu, v, 1);
        if (!(lane & 1) && valid) epi_qkv_pair(e, t, e.pos0 + t, r, v, other);
    } else if (EPI == EPI_SILU) {
        const float up = __shfl_xor_sync(0xffffffffu, v, 1);
        if (!(lane & 1) && valid) e.a_out[(int64_t)t * e.lda + (r >> 1)] = silu_f32(v) * up;
    }
}

template <int EPI, typename RG>
__global__ void __launch_bounds__(kGemvThreads) q8_gemv_rows_kernel(GemvRowsArgs a) {
    constexpr int kStages = RG::kStages, kStageBlocks = RG::kStageBlocks;
    constexpr int kStageCodeBytes = RG::kStageCodeBytes, kStageBytes = RG::kStageBytes;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    float* xs = reinterpret_cast<float*>(smem + kStages * kStageBytes);  // [m][xn]
    __shared__ __align__(8) uint64_t full[kStages];
    __shared__ __align__(8) uint64_t empty[kStages];
    __shared__ __align__(8) uint64_t xbar;
    __shared__ float red[kCWarps][kRowsMax][32];
    __shared__ float part[kRowsMax][32];

    const PackedQ8& W = a.W;
    const int k = W.k, nb = k >> 5;
    const int t0 = blockIdx.y * kRowsMax, m = min(kRowsMax, a.m - t0);  // this CTA's token rows
    const float* X = a.X + (size_t)t0 * a.ldx;
    const int S = a.splits;
    const int tile = blockIdx.x / S, split = blockIdx.x % S;
    const int b0 = (split * nb) / S, b1 = ((split + 1) * nb) / S;
    const int nblk = b1 - b0, xn = nblk * 32;
    const int n_stage = (nblk + kStageBlocks - 1) / kStageBlocks;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCWarps);
        }
        mbar_init(&xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kCWarps) {
        if (lane == 0) {
            const uint8_t* gcodes = reinterpret_cast<const uint8_t*>(W.qs) + (size_t)tile * k * 32;
            const uint8_t* gscales = reinterpret_cast<const uint8_t*>(W.d) + (size_t)tile * nb * 64;
            auto issue_stage = [&](int j) {
                const int slot = j % kStages;
                if (j >= kStages) mbar_wait_bounded(&empty[slot], ((j / kStages) - 1) & 1, a.err, 14);
                const int bs = b0 + j * kStageBlocks;
                const int nbs = min(kStageBlocks, b1 - bs);
                uint8_t* dst = stages + slot * kStageBytes;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(nbs * 1024 + nbs * 64));
                bulk_g2s(dst, gcodes + (size_t)bs * 1024, nbs * 1024, &full[slot]);
                bulk_g2s(dst + kStageCodeBytes, gscales + (size_t)bs * 64, nbs * 64, &full[slot]);
            };
            const int first = min(kStages, n_stage);
            for (int j = 0; j < first; ++j) issue_stage(j);  // weights: no kernel writes them
            pdl_wait();                                      // x: written by the preceding kernel
            mbar_arrive_expect_tx(&xbar, (uint32_t)(m * xn * 4));
            for (int t = 0; t < m; ++t)
                bulk_g2s(xs + (size_t)t * xn, X + (size_t)t * a.ldx + b0 * 32, (uint32_t)(xn * 4), &xbar);
            for (int j = first; j < n_stage; ++j) issue_stage(j);
        }
    } else {
        pdl_wait();
        if (tid == 0) pdl_launch_dependents();
        mbar_wait_bounded(&xbar, 0, a.err, 15);
        float acc[kRowsMax];
#pragma unroll
        for (int t = 0; t < kRowsMax; ++t) acc[t] = 0.0f;
        for (int j = 0; j < n_stage; ++j) {
            const int slot = j % kStages;
            mbar_wait_bounded(&full[slot], (j / kStages) & 1, a.err, 16);
            const int bs = j * kStageBlocks;  // relative to b0
            const int nbs = min(kStageBlocks, nblk - bs);
            const uint8_t* st = stages + slot * kStageBytes;
            for (int bi = warp; bi < nbs; bi += kCWarps) {
                const uint4 q0 = *reinterpret_cast<const uint4*>(st + bi * 1024 + lane * 16);
                const uint4 q1 = *reinterpret_cast<const uint4*>(st + bi * 1024 + 512 + lane * 16);
                const float d = __half2float(reinterpret_cast<const __half*>(st + kStageCodeBytes)[bi * 32 + lane]);
                // the 32 codes as 16 exact f32 pairs, once for every token row
                uint64_t w[16];
                const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t u = qw[i] ^ 0x80808080u;
                    w[2 * i] = codes2_f2<0>(u);
                    w[2 * i + 1] = codes2_f2<2>(u);
                }
                const float* xb = xs + (bs + bi) * 32;
#pragma unroll
                for (int t = 0; t < kRowsMax; ++t) {
                    if (t < m) {
                        const float4* x4 = reinterpret_cast<const float4*>(xb + (size_t)t * xn);
                        uint64_t s0 = 0, s1 = 0;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float4 xv = x4[i];
                            s0 = fma_f2(w[2 * i], pack_f2(xv.x, xv.y), s0);
                            s1 = fma_f2(w[2 * i + 1], pack_f2(xv.z, xv.w), s1);
                        }
                        acc[t] = fmaf(d, (f2_lo(s0) + f2_hi(s0)) + (f2_lo(s1) + f2_hi(s1)), acc[t]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
#pragma unroll
        for (int t = 0; t < kRowsMax; ++t)
            if (t < m) red[warp][t][lane] = acc[t];
        named_bar_sync(1, kCWarps * 32);
        // warp w finishes token rows w, w + 8: the sum over the eight warps
        for (int t = warp; t < m; t += kCWarps) {
            float v = 0.0f;
#pragma unroll
            for (int w2 = 0; w2 < kCWarps; ++w2) v += red[w2][t][lane];
            if (S == 1)
                rows_epilogue<EPI>(a.e, W.rows, tile, lane, t0 + t, v);
            else
                part[t][lane] = v;
        }
        if (S > 1) {
            cluster_sync();
            if (split == 0) {
                for (int t = warp; t < m; t += kCWarps) {
                    float v = part[t][lane];
                    for (int rnk = 1; rnk < S; ++rnk) v += ld_dsmem_f32(&part[t][lane], (uint32_t)rnk);
                    rows_epilogue<EPI>(a.e, W.rows, tile, lane, t0 + t, v);
                }
            }
            cluster_sync();  // peers keep their shared memory until the leader has read it
        }
        return;
    }
    if (S > 1) {
        __syncwarp();
        cluster_sync();
        cluster_sync();
    }
}

template <int EPI>
static cudaError_t gemv_rows_launch(const PackedQ8& W, const float* X, int m, int ldx, const EpiArgs& e, bool pdl,
                                    int* err, cudaStream_t s) {
    using RG = RingDeep;
    constexpr size_t ring = (size_t)RG::kStages * RG::kStageBytes;
    const int tiles = W.rows_pad / 32, nb = W.k / 32;
    const int sms = sm_count_current();
    const int chunks = (m + kRowsMax - 1) / kRowsMax, mc = std::min(m, kRowsMax);
    // splits: fill the GPU (at most one CTA per SM per tile-split and chunk, 8
    // blocks per split at least) and make the chunk's x slices fit beside the ring
    int S = 1;
    auto fits = [&](int sp) { return ring + (size_t)mc * ((nb + sp - 1) / sp) * 32 * 4 <= (size_t)kRowsMaxSmem; };
    while (S < 8 && (!fits(S) || ((int64_t)tiles * chunks * (S + 1) <= sms && nb / (S + 1) >= 8))) ++S;
    if (!fits(S) || chunks > 65535) return cudaErrorInvalidValue;
    const size_t smem = ring + (size_t)mc * ((nb + S - 1) / S) * 32 * 4;
    GemvRowsArgs a{W, X, m, ldx, e, S, err};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * S, chunks);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int n = 0;
    if (S > 1) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = S;
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
    return cudaLaunchKernelEx(&cfg, q8_gemv_rows_kernel<EPI, RG>, a);
}

bool gemv_rows_fits(int64_t m, int64_t k) {
    constexpr size_t ring = (size_t)RingDeep::kStages * RingDeep::kStageBytes;
    const int64_t mc = std::min<int64_t>(m, kRowsMax), nb = k / 32;
    return ring + (size_t)mc * ((nb + 7) / 8) * 32 * 4 <= (size_t)kRowsMaxSmem;
}

cudaError_t launch_gemv_rows(const PackedQ8& W, const float* X, int m, int ldx, int epi, const EpiArgs& e, bool pdl,
                             int* err, cudaStream_t s) {
    if (m < 1 || ldx % 4) return cudaErrorInvalidValue;
    switch (epi) {
        case EPI_STORE: return gemv_rows_launch<EPI_STORE>(W, X, m, ldx, e, pdl, err, s);
        case EPI_RESIDUAL: return gemv_rows_launch<EPI_RESIDUAL>(W, X, m, ldx, e, pdl, err, s);
        case EPI_QKV: return gemv_rows_launch<EPI_QKV>(W, X, m, ldx, e, pdl, err, s);
        case EPI_SILU: return gemv_rows_launch<EPI_SILU>(W, X, m, ldx, e, pdl, err, s);
    }
    return cudaErrorInvalidValue;
}

// CTAs of one instantiation resident per SM with `smem` bytes of dynamic
// shared memory (occupancy query, remembered per kernel and size).
static int resident_ctas(void (*kernel)(GemvArgs), size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<const void*, size_t>, int> known;
    std::lock_guard<std::mutex> lock(mu);
    const std::pair<const void*, size_t> key((const void*)kernel, smem);
    auto it = known.find(key);
    if (it != known.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kGemvThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    n = n > 0 ? n : 1;
    known[key] = n;
    return n;
}

template <int EPI, bool NORM, typename RG>
static cudaError_t gemv_launch_ring(const PackedQ8& W, const float* x, const float* g, float eps, const EpiArgs& e,
                                    bool pdl, int* err, cudaStream_t s, const GemvPreSum* pre, int force_splits) {
    constexpr int kStages = RG::kStages, kStageBytes = RG::kStageBytes;
    const int tiles = W.rows_pad / 32, nb = W.k / 32;
    const int sms = sm_count_current();
    const int S = force_splits > 0 ? force_splits : gemv_splits(tiles, nb, sms, RG::kCtasPerSm);
    const int max_blk = (nb + S - 1) / S;
    const int n_part = (NORM && pre) ? pre->n_part : 0;
    // x (its slice, or all of it for the norm) and the added partials
    const size_t x_floats = NORM ? (size_t)W.k * (1 + n_part) : (size_t)max_blk * 32;
    const size_t smem = (size_t)kStages * kStageBytes + x_floats * sizeof(float);
    if (smem > (size_t)kGemvMaxSmem) return cudaErrorInvalidValue;
    GemvArgs a{W, x, g, eps, e, S, err, (NORM && pre) ? *pre : GemvPreSum{}};
    // S == 1: persistent CTAs, as many as are resident at once (each takes every
    // grid-th row tile); S > 1: one cluster per tile
    int grid = tiles * S;
    if (S == 1) grid = std::min(tiles, sms * resident_ctas(q8_gemv_kernel<EPI, NORM, RG>, smem));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int n = 0;
    if (S > 1) {
        attrs[n].id = cudaLaunchAttributeClusterDimension;
        attrs[n].val.clusterDim.x = S;
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
    return cudaLaunchKernelEx(&cfg, q8_gemv_kernel<EPI, NORM, RG>, a);
}

template <int EPI, bool NORM>
static cudaError_t gemv_launch_one(const PackedQ8& W, const float* x, const float* g, float eps, const EpiArgs& e,
                                   bool pdl, int* err, cudaStream_t s, const GemvPreSum* pre, int force_splits) {
    const int tiles = W.rows_pad / 32;
    if (tiles >= 2 * sm_count_current())
        return gemv_launch_ring<EPI, NORM, RingWide>(W, x, g, eps, e, pdl, err, s, pre, force_splits);
    return gemv_launch_ring<EPI, NORM, RingDeep>(W, x, g, eps, e, pdl, err, s, pre, force_splits);
}

template <int EPI>
static cudaError_t gemv_set_attr() {
    cudaError_t err = cudaSuccess;
    auto one = [&](auto kernel) {
        if (err == cudaSuccess) err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemvMaxSmem);
    };
    one(q8_gemv_kernel<EPI, true, RingWide>);
    one(q8_gemv_kernel<EPI, false, RingWide>);
    one(q8_gemv_kernel<EPI, true, RingDeep>);
    one(q8_gemv_kernel<EPI, false, RingDeep>);
    if (EPI != EPI_ARGMAX && err == cudaSuccess)
        err = cudaFuncSetAttribute(q8_gemv_rows_kernel<EPI == EPI_ARGMAX ? EPI_STORE : EPI, RingDeep>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, kRowsMaxSmem);
    return err;
}

// Raise the dynamic shared-memory limit of every instantiation once per device
// (before any stream capture).
cudaError_t init_gemv_attributes() {
    sm_count_current();
    cudaError_t err = gemv_set_attr<EPI_STORE>();
    if (err == cudaSuccess) err = gemv_set_attr<EPI_RESIDUAL>();
    if (err == cudaSuccess) err = gemv_set_attr<EPI_QKV>();
    if (err == cudaSuccess) err = gemv_set_attr<EPI_SILU>();
    if (err == cudaSuccess) err = gemv_set_attr<EPI_ARGMAX>();
    return err;
}

size_t gemv_max_k() {
    // stages + the x slice of an unsplit unit must fit in shared memory
    constexpr int ring = RingWide::kStages * RingWide::kStageBytes > RingDeep::kStages * RingDeep::kStageBytes
                             ? RingWide::kStages * RingWide::kStageBytes
                             : RingDeep::kStages * RingDeep::kStageBytes;
    return (size_t)(kGemvMaxSmem - ring) / sizeof(float) / 32 * 32;
}

cudaError_t launch_gemv(const PackedQ8& W, const float* x, const float* norm_g, float eps, int epi,
                        const EpiArgs& e, bool pdl, int* err, cudaStream_t s, const GemvPreSum* pre,
                        int force_splits) {
    const bool norm = norm_g != nullptr;
    if (force_splits < 0 || force_splits > 8 || (force_splits > 0 && W.k / 32 < force_splits))
        return cudaErrorInvalidValue;
    const int f = force_splits;
    switch (epi) {
        case EPI_STORE:
            return norm ? gemv_launch_one<EPI_STORE, true>(W, x, norm_g, eps, e, pdl, err, s, pre, f)
                        : gemv_launch_one<EPI_STORE, false>(W, x, norm_g, eps, e, pdl, err, s, pre, f);
        case EPI_RESIDUAL:
            return norm ? gemv_launch_one<EPI_RESIDUAL, true>(W, x, norm_g, eps, e, pdl, err, s, pre, f)
                        : gemv_launch_one<EPI_RESIDUAL, false>(W, x, norm_g, eps, e, pdl, err, s, pre, f);
        case EPI_QKV:
            return norm ? gemv_launch_one<EPI_QKV, true>(W, x, norm_g, eps, e, pdl, err, s, pre, f)
                        : gemv_launch_one<EPI_QKV, false>(W, x, norm_g, eps, e, pdl, err, s, pre, f);
        case EPI_SILU:
            return norm ? gemv_launch_one<EPI_SILU, true>(W, x, norm_g, eps, e, pdl, err, s, pre, f)
                        : gemv_launch_one<EPI_SILU, false>(W, x, norm_g, eps, e, pdl, err, s, pre, f);
        case EPI_ARGMAX:
            return norm ? gemv_launch_one<EPI_ARGMAX, true>(W, x, norm_g, eps, e, pdl, err, s, pre, f)
                        : gemv_launch_one<EPI_ARGMAX, false>(W, x, norm_g, eps, e, pdl, err, s, pre, f);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lq8
