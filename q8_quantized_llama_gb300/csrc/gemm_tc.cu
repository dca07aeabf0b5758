// Q8_0 matrix-matrix product for prefill rows on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory): C[t][n] = X[t][:] . W[n][:]
// for T > 16 tokens, the dense contraction of the prefill path ("生成一个
// token", prefill 和 decode：同一个 forward，不同的路: many rows go to the
// matrix-matrix kernel).
//
// Precision: the int8 codes q of a Q8_0 block are exact in f16, and the
// block scale d is one number per (row, k-block), so the tensor cores compute
// per k-block the block partial P = sum_k q.x' in f16 x f16 -> f32 MMAs
// (kind::f16), with each token's activations scaled by a power of two 2^s
// (the row's largest magnitude brought into [2^14, 2^15)) and split as
// x' = x 2^s = hi + lo (hi = x' rounded to f16, lo = x' - hi rounded to f16):
// two MMAs per 16-wide k-step, f32 accumulation in TMEM. The scaling and the
// split are done once per token row, before the product, by the kernel that
// finds the row's maximum (the RMSNorm that produced x, or a short pass), which
// writes the split rows in the MMA's operand layout: per k-block one 128-byte
// row of 32 hi then 32 lo halves. Accumulator warps add d.P to the running sums in
// registers; the epilogue multiplies each token's sums by 2^-s (exact). Each
// product q.x is off by at most 2^-22 relative, plus 2^-39 of the row's
// largest |x| times |q| where lo falls below the f16 normal range, then one
// f32 rounding per block partial.
//
// CTA tile: 128 weight rows (MMA M) x 128 tokens (MMA N), k-block 32 (one
// Q8_0 block). Warp roles (18 warps):
//  - producer warp: per k-block three tensor copies: the split activation
//    tile (2-D, 128 token rows x 128 bytes of hi and lo, 128-byte swizzle:
//    the MMA's K-major B layout, used in place), and the codes and scales of
//    the CTA's four 32-row tiles (3-D views [tile][k-block][1 KiB or 64 B] of
//    the packed weights, one box each; tiles past the matrix read as zeros);
//  - two groups of 4 converter warps, taking k-blocks in turn: write each
//    row's 32 codes as f16 pairs into tensor memory (tcgen05.st; A operand,
//    row r in lane r);
//  - MMA warp: one thread issues the 4 MMAs of a k-block (A from tensor
//    memory) into one of two block-partial buffers and commits them to the
//    stage's "done" barrier (frees the stage for the producer) and to the
//    buffer's "full" barrier;
//  - 8 accumulator warps (4 lane quarters x 2 column halves): per k-block read
//    the block partial, free the buffer, and add it times the row's d (read
//    from global memory one block ahead) into 64 registers.
// Stages and buffers are handed on with mbarriers (no CTA-wide barrier in the
// k loop). Token tiles vary fastest in the grid: the CTAs that share a weight
// tile run at the same time and read it from DRAM once. At the end the
// accumulators return the tile to tensor memory and all 16 converter and
// accumulator warps apply the epilogue, 32 token columns each.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "epilogue.cuh"
#include "ptx.cuh"

namespace lq8 {

constexpr int kTcBM = 128;
constexpr int kTcBN = 128;
// Stages in flight (6 or 8 measured no faster).
// The count stays a multiple of the converter groups: each stage is always
// converted by the same group, whose parity waits then never see a barrier
// two phases behind.
constexpr int kTcStagesMax = 4;
constexpr int kTcStagesSplit = 4;
constexpr int kTcConvGroups = 2;                      // converter groups, taking k-blocks in turn
constexpr int kTcGroupWarps = 4;                      // warps of one group (one k-block, 32 rows each)
constexpr int kTcConvWarps = kTcConvGroups * kTcGroupWarps;
constexpr int kTcAccWarps = 8;                        // accumulator warps: 4 lane quarters x 2 column halves
constexpr int kTcAccWarp0 = kTcConvWarps;
constexpr int kTcThreads = (kTcConvWarps + kTcAccWarps + 2) * 32;  // + producer, MMA issuer
static_assert(kTcStagesMax % kTcConvGroups == 0 && kTcStagesSplit % kTcConvGroups == 0,
              "each stage is converted by one group");
constexpr int kTcProducerWarp = kTcConvWarps + kTcAccWarps, kTcMmaWarp = kTcProducerWarp + 1;
constexpr int kTileBytes = 128 * 128;                 // 128 rows x 128 bytes
// one stage: the split activation tile (128 tokens x 128 bytes: hi in the
// first 64 bytes of each row, lo in the second, 128-byte swizzle), codes of 4
// row tiles, their scales
constexpr int kStHiLo = 0, kStCodes = kTileBytes;
constexpr int kStScales = kStCodes + 4096;
constexpr int kStageBytes = (kStScales + 256 + 1023) / 1024 * 1024;
constexpr int kTcSmem = kTcStagesMax * kStageBytes + 1024;  // + alignment slack
constexpr int kPartStride = kTcBN + 4;                   // floats per row of a partial tile in shared memory
// split-K: a receive buffer of the S partials of this rank's rows, [S][128 / S][kPartStride]
constexpr int kRecvBytes = kTcBM * kPartStride * 4;
constexpr int kTcSmemSplit = kTcStagesSplit * kStageBytes + 1024 + kRecvBytes;
static_assert(kTcSmem <= 227 * 1024 && kTcSmemSplit <= 227 * 1024, "shared memory per CTA");
// tensor memory: two block-partial buffers of 128 columns, then per stage the
// 32 codes of each row as 16 f16 pairs (A operand)
constexpr int kTmemCols = 512;
constexpr int kTmemA = 2 * kTcBN;
constexpr int kTmemACols = 16;  // columns of one stage's A
static_assert(kTmemA + kTcStagesMax * kTmemACols <= kTmemCols, "tensor memory columns");

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

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle (16-byte
// chunk c of row r stored at chunk c ^ (r % 8)), 8-row groups 1024 bytes
// apart. A start address 32 or 64 bytes into the row selects the next 16
// k-values or the lo half.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);         // start address
    d |= (uint64_t)(16 >> 4) << 16;                   // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;                 // stride byte offset
    d |= (uint64_t)1 << 46;                           // descriptor version
    d |= (uint64_t)2 << 61;                           // 128-byte swizzle
    return d;
}

// Instruction descriptor: D f32, A and B f16, both K-major, M = 128, N = 128.
constexpr uint32_t kIdescF16 = (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(kTcBN >> 3) << 17) |
                               ((uint32_t)(kTcBM >> 4) << 24);

// D (tensor memory) += A (tensor memory, row i in lane i, k along columns) * B (shared memory)
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(kIdescF16), "r"(accumulate)
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
// 16 consecutive columns of this thread's lane (the warp's 32 lanes at taddr).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 3-D tensor copy global -> shared, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tensor copy global -> shared, completing on an mbarrier; coordinates in
// elements (x innermost).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Four codes (one word) as two f16 pairs, exactly: each byte u = q + 128
// becomes the f16 1024 + u (exponent 10, u in the mantissa), minus 1152.
__device__ __forceinline__ void codes_to_f16x2(uint32_t q, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = q ^ 0x80808080u;
    const __half2 bias = __halves2half2(__ushort_as_half((unsigned short)0x6480u), __ushort_as_half((unsigned short)0x6480u));
    uint32_t a = __byte_perm(u, 0x64646464u, 0x4140), b = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
    const __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
    lo = *reinterpret_cast<const uint32_t*>(&ha);
    hi = *reinterpret_cast<const uint32_t*>(&hb);
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

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

// SPLIT: the CTAs of a cluster (blockIdx.z = cluster rank) take equal shares
// of the k-blocks. Rank z owns rows [z * 128 / S, (z + 1) * 128 / S) of the
// tile: every rank sends the partial rows of each owner straight from tensor
// memory into slot [its rank] of the owner's receive buffer (asynchronous
// stores that count bytes on the owner's mbarrier), and the owner sums the S
// slots in rank order and applies the epilogue. A cluster barrier arrived at
// start and waited before the first send makes every peer's mbarrier valid;
// one arrived after the owner's data is complete and waited before exit keeps
// every CTA alive until all sends have landed.
template <int EPI, bool SPLIT>
__global__ void __launch_bounds__(kTcThreads, 1)
    q8_gemm_tc_kernel(PackedQ8 W, const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap dmap, int m, const float* __restrict__ rowmax, EpiArgs e,
                      int* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int kTcStages = SPLIT ? kTcStagesSplit : kTcStagesMax;
    __shared__ __align__(8) uint64_t full_bar[kTcStages];  // producer's copies landed
    __shared__ __align__(8) uint64_t conv_bar[kTcStages];  // converters wrote A (TMEM)
    __shared__ float row_inv[kTcBN];                        // each token's 2^-s, for the epilogue
    __shared__ __align__(8) uint64_t done_bar[kTcStages];  // MMAs of the stage complete
    __shared__ __align__(8) uint64_t part_full[2];          // a block partial is in tensor memory
    __shared__ __align__(8) uint64_t part_empty[2];         // the accumulator warps have read it
    __shared__ __align__(8) uint64_t recv_bar;              // split-K: peers' partial rows landed
    __shared__ uint32_t tmem_holder;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k = W.k, nb_all = k >> 5;
    const int S = SPLIT ? (int)gridDim.z : 1, z = SPLIT ? (int)blockIdx.z : 0;
    const int kb0 = (z * nb_all) / S, nb = ((z + 1) * nb_all) / S - kb0;  // this CTA's k-blocks
    // token tiles vary fastest, so the CTAs sharing a weight tile run together
    const int m0 = blockIdx.y * kTcBM;  // weight rows
    const int t0 = blockIdx.x * kTcBN;  // tokens
    const int tile0 = m0 >> 5;
    const int n_tiles = W.rows_pad >> 5;
    const int valid_tiles = min(4, n_tiles - tile0);

    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full_bar[s], 1);
            mbar_init(&conv_bar[s], kTcGroupWarps);
            mbar_init(&done_bar[s], 1);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(&part_full[p], 1);
            mbar_init(&part_empty[p], kTcAccWarps);
        }
        mbar_init(&recv_bar, 1);
        fence_mbar_init();
    }
    if (warp == kTcMmaWarp) tmem_alloc(&tmem_holder, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (SPLIT) cluster_arrive();  // waited before the first send
    const uint32_t tmem = tmem_holder;
    bool alive = true;  // cleared by a wait that ran out; later waits are skipped

    if (warp == kTcProducerWarp) {
        // lane 0 registers a stage's bytes (full boxes: tiles past the matrix
        // and token rows past m arrive as zeros), then lane 17 copies the codes
        // of the four tiles, lane 18 their scales and lane 16 the split
        // activation tile
        constexpr uint32_t stage_tx = (uint32_t)kTileBytes + 4u * (1024u + 64u);
        auto issue_weights = [&](int kb) {
            uint8_t* st = smem + (kb % kTcStages) * kStageBytes;
            uint64_t* bar = &full_bar[kb % kTcStages];
            if (lane == 0) mbar_arrive_expect_tx(bar, stage_tx);
            __syncwarp();
            if (lane == 17) tma_load_3d(st + kStCodes, &qmap, 0, kb0 + kb, tile0, bar);
            else if (lane == 18) tma_load_3d(st + kStScales, &dmap, 0, kb0 + kb, tile0, bar);
        };
        auto issue_x = [&](int kb) {
            if (lane == 16)
                tma_load_2d(smem + (kb % kTcStages) * kStageBytes + kStHiLo, &xmap, (kb0 + kb) * 64, t0,
                            &full_bar[kb % kTcStages]);
        };
        // the first stages' weights stream before the dependency on the previous kernel
        const int pre = min(kTcStages, nb);
        for (int kb = 0; kb < pre; ++kb) issue_weights(kb);
        pdl_wait();
        for (int kb = 0; kb < pre; ++kb) issue_x(kb);
        for (int kb = pre; kb < nb; ++kb) {
            const int s = kb % kTcStages;
            if (lane == 0 && alive) alive = mbar_wait_bounded(&done_bar[s], ((kb / kTcStages) - 1) & 1, err, 13);
            __syncwarp();
            issue_weights(kb);
            issue_x(kb);
        }
        // every copy has landed before the CTA may exit
        if (lane == 0)
            for (int kb = max(0, nb - kTcStages); kb < nb; ++kb)
                if (alive) alive = mbar_wait_bounded(&full_bar[kb % kTcStages], (kb / kTcStages) & 1, err, 14);
        __syncwarp();
    } else if (warp == kTcMmaWarp) {
        pdl_wait();
        if (lane == 0) {
            for (int kb = 0; kb < nb; ++kb) {
                const int s = kb % kTcStages, p = kb & 1;
                // the activation tile has landed (tensor copy) and A is in tensor memory
                if (alive) alive = mbar_wait_bounded(&full_bar[s], (kb / kTcStages) & 1, err, 18);
                if (alive) alive = mbar_wait_bounded(&conv_bar[s], (kb / kTcStages) & 1, err, 15);
                // the partial buffer of k-block kb - 2 has been read by the accumulator warps
                if (kb >= 2 && alive) alive = mbar_wait_bounded(&part_empty[p], ((kb >> 1) - 1) & 1, err, 17);
                tc_fence_after();
                const uint32_t xs = smem_u32(smem + s * kStageBytes);
                const uint32_t a = tmem + (uint32_t)(kTmemA + s * kTmemACols);
                const uint32_t d = tmem + (uint32_t)(p * kTcBN);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {  // two 16-wide k-steps, 32 bytes apart in the rows
                    const uint64_t b_hi = sw128_desc(xs + kStHiLo + kk * 32), b_lo = sw128_desc(xs + kStHiLo + 64 + kk * 32);
                    mma_f16_ts(d, a + kk * 8, b_hi, kk != 0);
                    mma_f16_ts(d, a + kk * 8, b_lo, 1u);
                }
                mma_commit(&done_bar[s]);
                mma_commit(&part_full[p]);
            }
        }
        __syncwarp();
    } else if (warp >= kTcConvWarps) {
        pdl_wait();  // accumulator warps: they write the outputs
    } else {
        pdl_wait();
        if (tid == 0) pdl_launch_dependents();
        // converter group g takes k-blocks g, g + G, ...; warp w of the group
        // writes the 32 codes (as exact f16) of row r = 32 * (w % 4) + lane
        const int group = warp / kTcGroupWarps, gtid = tid - group * kTcGroupWarps * 32;
        const int quarter = warp & 3;
        const bool row_ok = quarter < valid_tiles;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        // token gtid's 2^-s for the epilogue, from its row maximum (rows past m: any)
        const int tok = t0 + gtid;
        if (group == 0) row_inv[gtid] = pow2f(-row_shift(tok < m ? rowmax[tok] : 0.0f));
        for (int kb = group; kb < nb; kb += kTcConvGroups) {
            const int s = kb % kTcStages;
            if (alive) alive = mbar_wait_bounded(&full_bar[s], (kb / kTcStages) & 1, err, 11);
            tc_fence_after();
            uint8_t* st = smem + s * kStageBytes;
            const uint32_t a = tmem + lane_base + (uint32_t)(kTmemA + s * kTmemACols);
            {
                uint32_t u[16];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint4 qa = make_uint4(0u, 0u, 0u, 0u);
                    if (row_ok) qa = *reinterpret_cast<const uint4*>(st + kStCodes + quarter * 1024 + h * 512 + lane * 16);
                    codes_to_f16x2(qa.x, u[8 * h + 0], u[8 * h + 1]);
                    codes_to_f16x2(qa.y, u[8 * h + 2], u[8 * h + 3]);
                    codes_to_f16x2(qa.z, u[8 * h + 4], u[8 * h + 5]);
                    codes_to_f16x2(qa.w, u[8 * h + 6], u[8 * h + 7]);
                }
                tmem_st16(a, u);  // column c: codes 2c, 2c + 1
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&conv_bar[s]);
        }
    }

    // ---- accumulator warps: warp 8 + w holds rows 32*(w%4) + lane and token
    // columns [64*(w/4), 64*(w/4) + 64) of the tile in registers; per k-block
    // it reads the block partial from tensor memory, frees the buffer and adds
    // it times the block scale d of its row
    const int aw = warp - kTcAccWarp0;
    const bool accw = aw >= 0 && aw < kTcAccWarps;
    const int quarter = aw & 3, half = aw >> 2;
    constexpr int kColsPer = kTcBN / 2;
    float acc[kColsPer];
#pragma unroll
    for (int j = 0; j < kColsPer; ++j) acc[j] = 0.0f;
    if (accw) {
        const bool row_ok = quarter < valid_tiles;
        const __half* drow = W.d + ((int64_t)(tile0 + (row_ok ? quarter : 0)) * nb_all + kb0) * 32 + lane;
        float dnext = row_ok ? __half2float(drow[0]) : 0.0f;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        for (int kb = 0; kb < nb; ++kb) {
            const int p = kb & 1;
            const float d = dnext;
            if (kb + 1 < nb && row_ok) dnext = __half2float(drow[(int64_t)(kb + 1) * 32]);
            if (alive) alive = mbar_wait_bounded(&part_full[p], (kb >> 1) & 1, err, 12);
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < kColsPer; c += 16) {
                float t16[16];
                tmem_ld16(tmem + lane_base + (uint32_t)(p * kTcBN + half * kColsPer + c), t16);
#pragma unroll
                for (int j = 0; j < 16; ++j) acc[c + j] = fmaf(d, t16[j], acc[c + j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&part_empty[p]);
        }
    }

    if (!SPLIT) {
        // the finished tile goes back to tensor memory (partial buffer 0: every
        // MMA is complete, and each accumulator warp overwrites only the region
        // it alone read), then all 16 converter and accumulator warps apply the
        // epilogue, 32 token columns each: warp w reads lanes 32*(w%4) and
        // columns [32*(w/4), 32*(w/4) + 32)
        if (accw) {
            const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
#pragma unroll
            for (int c = 0; c < kColsPer; c += 16) {
                uint32_t u[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) u[j] = __float_as_uint(acc[c + j]);
                tmem_st16(tmem + lane_base + (uint32_t)(half * kColsPer + c), u);
            }
            tmem_wait_st();
        }
        if (warp < kTcConvWarps + kTcAccWarps) {
            tc_fence_before();
            named_bar_sync(1, (kTcConvWarps + kTcAccWarps) * 32);
            tc_fence_after();
            const int eq = warp & 3, part = warp >> 2;
            const int r = m0 + eq * 32 + lane;
            for (int c0 = part * 32; c0 < part * 32 + 32; c0 += 16) {
                float v[16];
                tmem_ld16(tmem + ((uint32_t)(eq * 32) << 16) + (uint32_t)c0, v);
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] *= row_inv[c0 + j];
                if (EPI == EPI_RESIDUAL) {
                    // the 16 residual reads first, then the 16 writes: no chain of dependent round trips
                    float y0[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = t0 + c0 + j;
                        y0[j] = (t < m && r < W.rows) ? e.y[(int64_t)t * e.ldy + r] : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = t0 + c0 + j;
                        if (t < m && r < W.rows) e.y[(int64_t)t * e.ldy + r] = y0[j] + v[j];
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float other =
                            (EPI == EPI_QKV || EPI == EPI_SILU) ? __shfl_xor_sync(0xffffffffu, v[j], 1) : 0.f;
                        tc_epilogue_one<EPI>(e, m, W.rows, t0 + c0 + j, r, v[j], other);
                    }
                }
            }
        }
    } else {
        const int rows_per = kTcBM / S;
        float* recv = reinterpret_cast<float*>(smem + kTcStages * kStageBytes);  // [S][rows_per][kPartStride]
        if (tid == 0 && alive)
            mbar_arrive_expect_tx(&recv_bar, (uint32_t)((S - 1) * rows_per * kTcBN * 4));
        cluster_wait();  // every peer's receive barrier is initialised
        if (accw) {
            const int row = quarter * 32 + lane;
            const int owner = row / rows_per, orow = row - owner * rows_per;
            float* dst = recv + ((size_t)z * rows_per + orow) * kPartStride + half * kColsPer;
#pragma unroll
            for (int j = 0; j < kColsPer; j += 4) {
                const float4 f = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
                if (owner == z) *reinterpret_cast<float4*>(dst + j) = f;
                else st_async_f32x4(dst + j, (uint32_t)owner, f, &recv_bar);
            }
        }
        if (alive) alive = mbar_wait_bounded(&recv_bar, 0, err, 16);
        __syncthreads();  // this rank's own slot is written too
        cluster_arrive();  // waited before exit: every send in the cluster has landed by then
        // rank z sums its rows over the S slots in rank order; thread -> (row pair, 4 tokens)
        const int ra = z * rows_per;
        for (int f = tid; f < (rows_per / 2) * (kTcBN / 4); f += kTcThreads) {
            const int rp = f % (rows_per / 2), t = (f / (rows_per / 2)) * 4;
            const int lr = 2 * rp;
            float4 v0 = make_float4(0.f, 0.f, 0.f, 0.f), v1 = v0;
            for (int zz = 0; zz < S; ++zz) {
                const float4 a4 = *reinterpret_cast<const float4*>(recv + ((size_t)zz * rows_per + lr) * kPartStride + t);
                const float4 b4 =
                    *reinterpret_cast<const float4*>(recv + ((size_t)zz * rows_per + lr + 1) * kPartStride + t);
                v0.x += a4.x; v0.y += a4.y; v0.z += a4.z; v0.w += a4.w;
                v1.x += b4.x; v1.y += b4.y; v1.z += b4.z; v1.w += b4.w;
            }
            const float i0 = row_inv[t], i1 = row_inv[t + 1], i2 = row_inv[t + 2], i3 = row_inv[t + 3];
            const float e0[4] = {v0.x * i0, v0.y * i1, v0.z * i2, v0.w * i3};
            const float e1[4] = {v1.x * i0, v1.y * i1, v1.z * i2, v1.w * i3};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (EPI == EPI_QKV || EPI == EPI_SILU) {
                    tc_epilogue_one<EPI>(e, m, W.rows, t0 + t + j, m0 + ra + lr, e0[j], e1[j]);
                } else {
                    tc_epilogue_one<EPI>(e, m, W.rows, t0 + t + j, m0 + ra + lr, e0[j], 0.f);
                    tc_epilogue_one<EPI>(e, m, W.rows, t0 + t + j, m0 + ra + lr + 1, e1[j], 0.f);
                }
            }
        }
        cluster_wait();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// CTAs of the tensor-core GEMM that can be resident at once with S CTAs per
// cluster: one per SM without a split; with a split, the occupancy API's count
// of co-resident S-CTA clusters (a cluster takes S SMs of one GPC, so on this
// GPU 16 clusters of 8 do not all fit at once). Queried once per device.
static int g_tc_capacity[64][4] = {};

static int gemm_tc_capacity(int S) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
    const int slot = S == 1 ? 0 : S == 2 ? 1 : S == 4 ? 2 : 3;
    int& cap = g_tc_capacity[dev][slot];
    if (cap > 0) return cap;
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    if (S == 1) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q8_gemm_tc_kernel<EPI_STORE, false>, kTcThreads,
                                                          (size_t)kTcSmem) != cudaSuccess || per_sm < 1) {
            cudaGetLastError();
            per_sm = 1;
        }
        cap = sms * per_sm;
        return cap;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, S);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = (size_t)kTcSmemSplit;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = S;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, q8_gemm_tc_kernel<EPI_STORE, true>, &cfg) != cudaSuccess ||
        clusters < 1) {
        cudaGetLastError();
        clusters = sms / S;
    }
    cap = clusters * S;
    return cap;
}

// k-splits per output tile over S in {1, 2, 4, 8} CTAs of a cluster (S divides
// the 128 rows of a tile, at least two k-blocks per CTA): the least estimated
// time, counted in k-blocks per wave of co-resident CTAs, with split_cost(S)
// k-blocks' worth for the exchange of partial rows (measured with per-CTA
// timestamps at 203 tokens: 0.64 us per k-block in steady state, ~2 us from
// the last block partial to the peers' rows landing with S = 2, ~3.7 us with
// S = 8), taken only when it beats the next smaller choice by more than 10%.
static int split_cost(int S) { return 2 + S / 2; }

static int gemm_tc_splits(int tiles, int nb) {
    int best = 1;
    const int cap1 = gemm_tc_capacity(1);
    long best_cost = (long)((tiles + cap1 - 1) / cap1) * nb;
    for (int S = 2; S <= 8; S *= 2) {
        if (nb / S < 2) break;
        const int cap = gemm_tc_capacity(S);
        const long waves = ((long)tiles * S + cap - 1) / cap;
        const long cost = waves * ((nb + S - 1) / S + split_cost(S));
        if (cost * 10 < best_cost * 9) {  // a split only for a clear (> 10%) gain
            best = S;
            best_cost = cost;
        }
    }
    return best;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on the driver library).
static PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

static cudaError_t get_encode_tiled() {
    if (!g_encode_tiled) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return cudaErrorNotSupported;
        g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return cudaSuccess;
}

// Tensor map of the split activations hl[m][2k] (f16): boxes of one k-block
// (64 halves = 128 bytes: 32 hi, 32 lo) x 128 rows with the 128-byte swizzle;
// rows past m read as zeros. The box's x coordinate is 64 kb: 128 bytes, a
// multiple of 16.
static cudaError_t make_hl_map(CUtensorMap* map, const __half* hl, int m, int k) {
    if ((uintptr_t)hl & 15) return cudaErrorInvalidValue;
    cudaError_t e = get_encode_tiled();
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[2] = {(cuuint64_t)2 * k, (cuuint64_t)m};
    const cuuint64_t strides[1] = {(cuuint64_t)2 * k * sizeof(__half)};
    const cuuint32_t box[2] = {64, (cuuint32_t)kTcBN};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(hl), dims, strides,
                                      box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D views of the packed weights as 32-bit words: codes [tile][k-block][256]
// (1 KiB per 32-row tile and k-block) and scales [tile][k-block][16] (64 B);
// one box = the CTA's four tiles at one k-block, tiles past the matrix zero.
static cudaError_t make_w_maps(CUtensorMap* qmap, CUtensorMap* dmap, const PackedQ8& W) {
    if (((uintptr_t)W.qs | (uintptr_t)W.d) & 15) return cudaErrorInvalidValue;
    cudaError_t e = get_encode_tiled();
    if (e != cudaSuccess) return e;
    const cuuint64_t tiles = (cuuint64_t)(W.rows_pad / 32), nb = (cuuint64_t)(W.k / 32);
    const cuuint32_t elem[3] = {1, 1, 1};
    const cuuint64_t qdims[3] = {256, nb, tiles};
    const cuuint64_t qstrides[2] = {1024, nb * 1024};
    const cuuint32_t qbox[3] = {256, 1, 4};
    CUresult r = g_encode_tiled(qmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<int8_t*>(W.qs), qdims, qstrides,
                                qbox, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const cuuint64_t ddims[3] = {16, nb, tiles};
    const cuuint64_t dstrides[2] = {64, nb * 64};
    const cuuint32_t dbox[3] = {16, 1, 4};
    r = g_encode_tiled(dmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<__half*>(W.d), ddims, dstrides, dbox, elem,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The product's operand from X[m][ldx] (k columns): each row's largest |x|
// into rowmax, then the row scaled by its power of two and split into hi / lo
// (common.cuh) into hl. One CTA per row (enough CTAs to stream the widest
// inputs, 14336 columns, at HBM speed), float4 loads; the second pass reads
// the row again from L1. After the grid dependency wait, since X comes from
// the preceding kernel.
constexpr int kRowSplitThreads = 256;
__global__ void __launch_bounds__(kRowSplitThreads) row_split_kernel(const float* __restrict__ X, int k, int ldx,
                                                                     float* __restrict__ rowmax,
                                                                     __half* __restrict__ hl) {
    __shared__ float red[kRowSplitThreads / 32];
    pdl_wait();
    pdl_launch_dependents();
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* row = X + (size_t)t * ldx;
    float mx = 0.0f;
    for (int i = threadIdx.x * 4; i < k; i += kRowSplitThreads * 4) {
        const float4 v = *reinterpret_cast<const float4*>(row + i);
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    mx = warp_max(mx);
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = 0.0f;
#pragma unroll
    for (int w = 0; w < kRowSplitThreads / 32; ++w) mx = fmaxf(mx, red[w]);
    if (threadIdx.x == 0) rowmax[t] = mx;
    const float sc = pow2f(row_shift(mx));
    __half* hr = hl + (size_t)t * 2 * k;
    for (int i = threadIdx.x * 4; i < k; i += kRowSplitThreads * 4) {
        const float4 v = *reinterpret_cast<const float4*>(row + i);
        store_split4(hr, i, v.x * sc, v.y * sc, v.z * sc, v.w * sc);
    }
}

template <int EPI>
static cudaError_t gemm_tc_one(const PackedQ8& W, const float* X, int m, int ldx, const EpiArgs& e, bool pdl,
                               int* err, cudaStream_t s, const SplitRows& split, bool split_ready) {
    if (!split.rowmax || !split.hl) return cudaErrorInvalidValue;
    if (!split_ready) {
        if (((uintptr_t)X & 15) || (ldx & 3) || ldx < W.k) return cudaErrorInvalidValue;
        cudaError_t rerr = launch_ex(row_split_kernel, dim3(m), dim3(kRowSplitThreads), 0, s, pdl, X, W.k, ldx,
                                     split.rowmax, split.hl);
        if (rerr != cudaSuccess) return rerr;
        pdl = true;  // the product follows its own operand pass
    }
    CUtensorMap xmap, qmap, dmap;
    cudaError_t merr = make_hl_map(&xmap, split.hl, m, W.k);
    if (merr == cudaSuccess) merr = make_w_maps(&qmap, &dmap, W);
    if (merr != cudaSuccess) return merr;
    const float* rowmax = split.rowmax;
    const int gx = (W.rows_pad + kTcBM - 1) / kTcBM, gy = (m + kTcBN - 1) / kTcBN;
    const int S = gemm_tc_splits(gx * gy, W.k / 32);
    if (S == 1)
        return launch_ex(q8_gemm_tc_kernel<EPI, false>, dim3(gy, gx), dim3(kTcThreads), (size_t)kTcSmem, s, pdl, W,
                         xmap, qmap, dmap, m, rowmax, e, err);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gy, gx, S);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = (size_t)kTcSmemSplit;
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
    return cudaLaunchKernelEx(&cfg, q8_gemm_tc_kernel<EPI, true>, W, xmap, qmap, dmap, m, rowmax, e, err);
}

template <int EPI>
static cudaError_t gemm_tc_attr() {
    cudaError_t err = cudaFuncSetAttribute(q8_gemm_tc_kernel<EPI, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kTcSmem);
    if (err == cudaSuccess)
        err = cudaFuncSetAttribute(q8_gemm_tc_kernel<EPI, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kTcSmemSplit);
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
                           int* err, cudaStream_t s, const SplitRows& split, bool split_ready) {
    switch (epi) {
        case EPI_STORE: return gemm_tc_one<EPI_STORE>(W, X, m, ldx, e, pdl, err, s, split, split_ready);
        case EPI_RESIDUAL: return gemm_tc_one<EPI_RESIDUAL>(W, X, m, ldx, e, pdl, err, s, split, split_ready);
        case EPI_QKV: return gemm_tc_one<EPI_QKV>(W, X, m, ldx, e, pdl, err, s, split, split_ready);
        case EPI_SILU: return gemm_tc_one<EPI_SILU>(W, X, m, ldx, e, pdl, err, s, split, split_ready);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lq8
