// Q8_0 matrix-matrix product for prefill rows on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory): C[t][n] = X[t][:] . W[n][:]
// for T > 16 tokens, the dense contraction of the prefill path ("生成一个
// token", prefill 和 decode：同一个 forward，不同的路: many rows go to the
// matrix-matrix kernel).
//
// Precision: split-TF32 ("3xTF32"). A dequantised weight d*q (f32, at most 18
// significant bits) is exactly hi + lo with hi = tf32(w) and lo = w - hi (at
// most 7 bits, exact in tf32). An activation x is hi + lo with hi = tf32(x)
// and lo = x - hi (lo truncated to tf32 by the MMA: 22 significant bits kept).
// Three MMAs per k-step, w_hi.x_hi + w_hi.x_lo + w_lo.x_hi, accumulate in f32
// in TMEM; the dropped w_lo.x_lo term is below 2^-22 relative.
//
// CTA tile: 128 weight rows (MMA M) x 128 tokens (MMA N), k-step 32 (one Q8_0
// block = one 128-byte swizzle row of tf32). Raw k-blocks (codes, scales,
// activation rows) arrive by cp.async three blocks ahead; all 8 warps
// dequantise/split the current block into one of two operand slots
// (128-byte swizzled K-major layout the MMA reads through its descriptors)
// while the tensor core works on the other; one thread issues the MMAs and
// commits each slot to an mbarrier that releases it. The epilogue reads TMEM with tcgen05.ld (warp w
// reads lanes 32*(w%4).., column half w/4) and applies the shared epilogues.
#include "epilogue.cuh"
#include "ptx.cuh"

namespace lq8 {

constexpr int kTcBM = 128;
constexpr int kTcBN = 128;
constexpr int kTcSlots = 2;                     // operand slots (ping-pong with the tensor core)
constexpr int kTcThreads = 256;
constexpr int kTileBytes = 128 * 128;           // 128 rows x 128 bytes
constexpr int kSlotBytes = 4 * kTileBytes;      // A_hi, A_lo, B_hi, B_lo
constexpr int kRawStages = 4;                   // raw k-blocks in flight (cp.async)
constexpr int kRawBytes = 4096 + 256 + 128 * 128;  // codes, scales, activations of one k-block
constexpr int kTcSmem = kTcSlots * kSlotBytes + kRawStages * kRawBytes + 1024;  // + alignment slack

// ---- tcgen05 wrappers ---------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* holder, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(holder)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);         // start address
    d |= (uint64_t)(16 >> 4) << 16;                   // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset
    d |= (uint64_t)1 << 46;                           // descriptor version
    d |= (uint64_t)2 << 61;                           // 128-byte swizzle
    return d;
}

// Instruction descriptor: D f32, A/B tf32, both K-major, M = 128, N = 128.
constexpr uint32_t kIdescTf32 = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(kTcBN >> 3) << 17) |
                                ((uint32_t)(kTcBM >> 4) << 24);

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdescTf32), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ float tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Byte offset of the 16-byte chunk `c` (0..7) of row `r` in a 128-row x 128-byte
// K-major tile with the 128-byte swizzle.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Exact f32 values of 16 codes (4 words) times the block scale.
__device__ __forceinline__ void dequant16(const uint4& q, float d, float (&w)[16]) {
    const uint32_t ws[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t u = ws[i] ^ 0x80808080u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float biased = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540 + j));
            w[4 * i + j] = d * (biased - 8388736.0f);
        }
    }
}

// ---- cp.async (16-byte global -> shared copies, zero-filled when src_bytes = 0)
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Epilogue of one output element pair/element (row r of W, token t).
template <int EPI>
__device__ __forceinline__ void tc_epilogue_one(const EpiArgs& e, int m, int rows, int t, int r, float val,
                                                float other) {
    if (EPI == EPI_QKV || EPI == EPI_SILU) {
        if (t < m && r < rows && !(r & 1)) {
            if (EPI == EPI_QKV) epi_qkv_pair(e, t, e.pos0 + t, r, val, other);
            else e.a_out[(int64_t)t * e.lda + (r >> 1)] = silu_f32(val) * other;
        }
    } else if (t < m && r < rows) {
        if (EPI == EPI_STORE) e.y[(int64_t)t * e.ldy + r] = val;
        else if (EPI == EPI_RESIDUAL) e.y[(int64_t)t * e.ldy + r] += val;
    }
}

constexpr int kPartStride = kTcBN + 4;  // floats per row of a partial tile in shared memory

// SPLIT: the CTAs of a cluster (blockIdx.z = cluster rank) take equal shares
// of the k-blocks; each stores its partial tile in its shared memory and,
// after a cluster barrier, rank z sums rows [z * 128 / S, (z + 1) * 128 / S)
// over the S partials (in rank order, through distributed shared memory) and
// applies the epilogue to them.
template <int EPI, bool SPLIT>
__global__ void __launch_bounds__(kTcThreads, 1) q8_gemm_tc_kernel(PackedQ8 W, const float* __restrict__ X, int m,
                                                                    int ldx, EpiArgs e, int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ops = smem;                                 // kTcSlots operand slots (A_hi, A_lo, B_hi, B_lo)
    uint8_t* raw = smem + kTcSlots * kSlotBytes;         // kRawStages raw k-blocks
    __shared__ __align__(8) uint64_t mma_done[kTcSlots];
    __shared__ uint32_t tmem_holder;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k = W.k, nb_all = k >> 5;
    const int S = SPLIT ? (int)gridDim.z : 1, z = SPLIT ? (int)blockIdx.z : 0;
    const int kb0 = (z * nb_all) / S, nb = ((z + 1) * nb_all) / S - kb0;  // this CTA's k-blocks
    const int m0 = blockIdx.x * kTcBM;  // weight rows
    const int t0 = blockIdx.y * kTcBN;  // tokens
    const int tile0 = m0 >> 5;
    const int n_tiles = W.rows_pad >> 5;

    if (tid == 0) {
        for (int s = 0; s < kTcSlots; ++s) mbar_init(&mma_done[s], 1);
        fence_mbar_init();
    }
    if (warp == 0) tmem_alloc(&tmem_holder, kTcBN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_holder;

    pdl_wait();
    if (tid == 0) pdl_launch_dependents();

    // Raw k-block: codes of the CTA's 4 row tiles (1 KiB each, contiguous in
    // the packed layout), their scales (64 B each) and the 128 token rows of
    // activations (128 B each). Thread tid copies 16 B of codes, threads < 16
    // 16 B of scales, and 4 x 16 B of activations.
    auto issue_raw = [&](int kbr) {
        uint8_t* r = raw + (kbr % kRawStages) * kRawBytes;
        const int kb = kb0 + kbr;
        {
            const int t = tid >> 6, within = (tid & 63) * 16;
            const bool ok = tile0 + t < n_tiles;
            const int8_t* src = W.qs + ((int64_t)(ok ? tile0 + t : 0) * k * 32 + (int64_t)kb * 1024 + within);
            cp_async16(r + t * 1024 + within, src, ok ? 16u : 0u);
        }
        if (tid < 16) {
            const int t = tid >> 2, within = (tid & 3) * 16;
            const bool ok = tile0 + t < n_tiles;
            const uint8_t* src = reinterpret_cast<const uint8_t*>(W.d) +
                                 ((int64_t)(ok ? tile0 + t : 0) * nb_all + kb) * 64 + within;
            cp_async16(r + 4096 + t * 64 + within, src, ok ? 16u : 0u);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int f = tid + i * kTcThreads;
            const int row = f >> 3, c = f & 7;
            const bool ok = t0 + row < m;
            const float* src = X + (int64_t)(ok ? t0 + row : 0) * ldx + kb * 32 + c * 4;
            cp_async16(r + 4096 + 256 + row * 128 + c * 16, src, ok ? 16u : 0u);
        }
        cp_async_commit();
    };

    for (int j = 0; j < kRawStages - 1; ++j) {
        if (j < nb) issue_raw(j);
        else cp_async_commit();  // keep the group count uniform
    }

    const int a_row = tid >> 1, a_half = tid & 1;
    for (int kb = 0; kb < nb; ++kb) {
        cp_async_wait<kRawStages - 2>();
        __syncthreads();  // raw block kb complete for every thread; raw slot (kb-1) fully converted
        if (kb + kRawStages - 1 < nb) issue_raw(kb + kRawStages - 1);
        else cp_async_commit();
        const int slot = kb % kTcSlots;
        if (kb >= kTcSlots) mbar_wait_bounded(&mma_done[slot], ((kb / kTcSlots) - 1) & 1, err, 11);
        const uint8_t* r = raw + (kb % kRawStages) * kRawBytes;
        uint8_t* sA_hi = ops + slot * kSlotBytes;
        uint8_t* sA_lo = sA_hi + kTileBytes;
        uint8_t* sB_hi = sA_lo + kTileBytes;
        uint8_t* sB_lo = sB_hi + kTileBytes;
        {
            const int t = a_row >> 5, ln = a_row & 31;
            const uint4 qa = *reinterpret_cast<const uint4*>(r + t * 1024 + a_half * 512 + ln * 16);
            const float da = __half2float(reinterpret_cast<const __half*>(r + 4096)[t * 32 + ln]);
            float w[16];
            dequant16(qa, da, w);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float4 hi, lo;
                hi.x = tf32_rna(w[4 * c + 0]); lo.x = w[4 * c + 0] - hi.x;
                hi.y = tf32_rna(w[4 * c + 1]); lo.y = w[4 * c + 1] - hi.y;
                hi.z = tf32_rna(w[4 * c + 2]); lo.z = w[4 * c + 2] - hi.z;
                hi.w = tf32_rna(w[4 * c + 3]); lo.w = w[4 * c + 3] - hi.w;
                const uint32_t off = sw128_off(a_row, a_half * 4 + c);
                *reinterpret_cast<float4*>(sA_hi + off) = hi;
                *reinterpret_cast<float4*>(sA_lo + off) = lo;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int f = tid + i * kTcThreads;
            const int row = f >> 3, c = f & 7;
            const float4 x = *reinterpret_cast<const float4*>(r + 4096 + 256 + row * 128 + c * 16);
            float4 hi, lo;
            hi.x = tf32_rna(x.x); lo.x = x.x - hi.x;
            hi.y = tf32_rna(x.y); lo.y = x.y - hi.y;
            hi.z = tf32_rna(x.z); lo.z = x.z - hi.z;
            hi.w = tf32_rna(x.w); lo.w = x.w - hi.w;
            const uint32_t off = sw128_off(row, c);
            *reinterpret_cast<float4*>(sB_hi + off) = hi;
            *reinterpret_cast<float4*>(sB_lo + off) = lo;
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t a_hi = smem_u32(sA_hi), a_lo = smem_u32(sA_lo);
            const uint32_t b_hi = smem_u32(sB_hi), b_lo = smem_u32(sB_lo);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint32_t o = kk * 32;
                mma_tf32(tmem, sw128_desc(a_hi + o), sw128_desc(b_hi + o), (kb | kk) != 0);
                mma_tf32(tmem, sw128_desc(a_hi + o), sw128_desc(b_lo + o), 1u);
                mma_tf32(tmem, sw128_desc(a_lo + o), sw128_desc(b_hi + o), 1u);
            }
            mma_commit(&mma_done[slot]);
        }
    }
    cp_async_wait<0>();
    // all MMAs are complete once the last slot's commit has arrived
    mbar_wait_bounded(&mma_done[(nb - 1) % kTcSlots], ((nb - 1) / kTcSlots) & 1, err, 12);
    tc_fence_after();

    // ---- epilogue: warp w reads TMEM lanes 32*(w%4).. and token columns of half w/4
    const int quarter = warp & 3, half = warp >> 2;
    const int r = m0 + quarter * 32 + lane;
    if (!SPLIT) {
        for (int c0 = half * (kTcBN / 2); c0 < (half + 1) * (kTcBN / 2); c0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float other = (EPI == EPI_QKV || EPI == EPI_SILU) ? __shfl_xor_sync(0xffffffffu, v[j], 1) : 0.f;
                tc_epilogue_one<EPI>(e, m, W.rows, t0 + c0 + j, r, v[j], other);
            }
        }
    } else {
        // partial tile -> own shared memory (the operand slots are free now)
        float* part = reinterpret_cast<float*>(ops);  // [128 rows][kPartStride]
        const int row = quarter * 32 + lane;
        for (int c0 = half * (kTcBN / 2); c0 < (half + 1) * (kTcBN / 2); c0 += 16) {
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
            for (int j = 0; j < 16; j += 4)
                *reinterpret_cast<float4*>(part + row * kPartStride + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
        cluster_sync();
        // rank z sums its rows over the S partials; thread -> (row pair, 4 tokens)
        const int rows_per = kTcBM / S;
        const int ra = z * rows_per;
        for (int f = tid; f < (rows_per / 2) * (kTcBN / 4); f += kTcThreads) {
            const int rp = f % (rows_per / 2), t = (f / (rows_per / 2)) * 4;
            const int lr = ra + 2 * rp;
            float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
            for (int zz = 0; zz < S; ++zz) {
                const float4 a = ld_dsmem_f32x4(part + lr * kPartStride + t, (uint32_t)zz);
                const float4 b = ld_dsmem_f32x4(part + (lr + 1) * kPartStride + t, (uint32_t)zz);
                v0.x += a.x; v0.y += a.y; v0.z += a.z; v0.w += a.w;
                v1.x += b.x; v1.y += b.y; v1.z += b.z; v1.w += b.w;
            }
            const float e0[4] = {v0.x, v0.y, v0.z, v0.w}, e1[4] = {v1.x, v1.y, v1.z, v1.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (EPI == EPI_QKV || EPI == EPI_SILU) {
                    tc_epilogue_one<EPI>(e, m, W.rows, t0 + t + j, m0 + lr, e0[j], e1[j]);
                } else {
                    tc_epilogue_one<EPI>(e, m, W.rows, t0 + t + j, m0 + lr, e0[j], 0.f);
                    tc_epilogue_one<EPI>(e, m, W.rows, t0 + t + j, m0 + lr + 1, e1[j], 0.f);
                }
            }
        }
        cluster_sync();  // peers keep their shared memory until every rank has read it
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTcBN);
}

static int g_tc_sms = 0;

// k-splits per output tile: enough CTAs to cover the GPU once, at most 8 (a
// portable cluster), at least two k-blocks per CTA.
static int gemm_tc_splits(int tiles, int nb) {
    if (g_tc_sms <= 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_tc_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_tc_sms <= 0) g_tc_sms = 148;
    }
    int S = 1;
    while (S < 8 && tiles * S * 2 <= g_tc_sms && nb / (S * 2) >= 2) S *= 2;
    return S;
}

template <int EPI>
static cudaError_t gemm_tc_one(const PackedQ8& W, const float* X, int m, int ldx, const EpiArgs& e, bool pdl,
                               int* err, cudaStream_t s) {
    const int gx = (W.rows_pad + kTcBM - 1) / kTcBM, gy = (m + kTcBN - 1) / kTcBN;
    const int S = gemm_tc_splits(gx * gy, W.k / 32);
    if (S == 1)
        return launch_ex(q8_gemm_tc_kernel<EPI, false>, dim3(gx, gy), dim3(kTcThreads), (size_t)kTcSmem, s, pdl, W,
                         X, m, ldx, e, err);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, gy, S);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = (size_t)kTcSmem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = 1;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = S;
    int n = 1;
    if (pdl) {
        attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[1].val.programmaticStreamSerializationAllowed = 1;
        n = 2;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, q8_gemm_tc_kernel<EPI, true>, W, X, m, ldx, e, err);
}

template <int EPI>
static cudaError_t gemm_tc_attr() {
    cudaError_t err = cudaFuncSetAttribute(q8_gemm_tc_kernel<EPI, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kTcSmem);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(q8_gemm_tc_kernel<EPI, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    return err;
}

cudaError_t init_gemm_tc_attributes() {
    cudaError_t err = gemm_tc_attr<EPI_STORE>();
    if (err == cudaSuccess) err = gemm_tc_attr<EPI_RESIDUAL>();
    if (err == cudaSuccess) err = gemm_tc_attr<EPI_QKV>();
    if (err == cudaSuccess) err = gemm_tc_attr<EPI_SILU>();
    return err;
}

cudaError_t launch_gemm_tc(const PackedQ8& W, const float* X, int m, int ldx, int epi, const EpiArgs& e, bool pdl,
                           int* err, cudaStream_t s) {
    switch (epi) {
        case EPI_STORE: return gemm_tc_one<EPI_STORE>(W, X, m, ldx, e, pdl, err, s);
        case EPI_RESIDUAL: return gemm_tc_one<EPI_RESIDUAL>(W, X, m, ldx, e, pdl, err, s);
        case EPI_QKV: return gemm_tc_one<EPI_QKV>(W, X, m, ldx, e, pdl, err, s);
        case EPI_SILU: return gemm_tc_one<EPI_SILU>(W, X, m, ldx, e, pdl, err, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lq8
