// Matrix-vector product for the other GGUF block formats of a Q4_K_M file:
// Q5_0 (32 weights in 22 bytes), Q4_K and Q6_K (256 weights in 144 / 210
// bytes). "速度" (CPU GGUF：decode 快，prefill 慢) times QMatMul in these
// formats and lists a 135M Q4_K_M file as mostly Q5_0 with Q4K / Q6K for the
// down projections; the block layouts are the published GGUF definitions.
//
// Device layout (llama_q8_pack_fmt): rows in tiles of 32, each (tile, block)
// one contiguous record of 32 x the block's bytes, its fields regrouped so that
// lane l (row l of the tile) reads 16-byte chunks that sit next to the other
// lanes' (conflict-free shared-memory loads):
//   Q5_0 (704 B): qs 32 x 16 | qh 32 x 4 | d 32 x 2
//   Q4_K (4608 B): 8 chunks of qs, each 32 x 16 | d, dmin, 12 scale bytes 32 x 16
//   Q6_K (6720 B): 8 chunks of ql | 4 chunks of qh | 16 int8 scales 32 x 16 | d 32 x 2
// A tile's block range is one contiguous run of records, streamed into a
// shared-memory ring by a producer warp with bulk async copies, as in the
// Q8_0 kernel. Eight consumer warps take units (a Q5_0 block, half a Q4_K
// block of four sub-blocks, two Q6_K sub-blocks of 16) and turn codes into
// exact f32 with the offset folded in: bytes 0x4B0000cc are 2^23 + c, and
// subtracting 2^23 + offset leaves c - offset.
#include <algorithm>
#include <map>
#include <mutex>

#include "kernels.cuh"
#include "ptx.cuh"

namespace lq8 {

namespace {

constexpr int kFmtCWarps = 8;
constexpr int kFmtThreads = (kFmtCWarps + 1) * 32;
constexpr int kFmtStages = 4;
constexpr int kFmtMaxSmem = 227 * 1024 - 4096;

template <int T>
struct Fmt;
template <>
struct Fmt<kGgufQ5_0> {
    static constexpr int kW = 32, kBytes = 22, kRec = 32 * 22, kUnits = 1, kUnitW = 32, kStageRecs = 16;
};
template <>
struct Fmt<kGgufQ4_K> {
    // a unit is half a block (four sub-blocks): the scale bytes are read and
    // unpacked once per unit, and each 32-byte chunk pair serves two sub-blocks
    static constexpr int kW = 256, kBytes = 144, kRec = 32 * 144, kUnits = 2, kUnitW = 128, kStageRecs = 4;
};
template <>
struct Fmt<kGgufQ6_K> {
    static constexpr int kW = 256, kBytes = 210, kRec = 32 * 210, kUnits = 8, kUnitW = 32, kStageRecs = 2;
};

// Four codes held as bytes of c (each < 256 - 2^23 rounding is exact) minus
// `off`, times x[0..3], into two packed partial sums.
__device__ __forceinline__ uint64_t dot4_codes(uint32_t c, float4 x, float off, uint64_t acc) {
    const uint32_t b0 = __byte_perm(c, 0x4B000000u, 0x7540);
    const uint32_t b1 = __byte_perm(c, 0x4B000000u, 0x7541);
    const uint32_t b2 = __byte_perm(c, 0x4B000000u, 0x7542);
    const uint32_t b3 = __byte_perm(c, 0x4B000000u, 0x7543);
    const float bias = 8388608.0f + off;  // 2^23 + offset
    const uint64_t lo = sub_f2((uint64_t)b0 | ((uint64_t)b1 << 32), pack_f2(bias, bias));
    const uint64_t hi = sub_f2((uint64_t)b2 | ((uint64_t)b3 << 32), pack_f2(bias, bias));
    acc = fma_f2(lo, pack_f2(x.x, x.y), acc);
    return fma_f2(hi, pack_f2(x.z, x.w), acc);
}

// Four bits b (bits 0..3) to bit 4 of each byte: bit i -> bit 8 i + 4.
__device__ __forceinline__ uint32_t spread4_to_bit4(uint32_t b) { return ((b * 0x00204081u) & 0x01010101u) << 4; }

__device__ __forceinline__ uint4 lds_u4(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Dot of one 32-weight unit u of a record (lane = row) with x[0..32) of that unit.
template <int T>
__device__ __forceinline__ float unit_dot(const uint8_t* rec, int u, int lane, const float* x, const float* xsum);

template <>
__device__ __forceinline__ float unit_dot<kGgufQ5_0>(const uint8_t* rec, int, int lane, const float* x,
                                                     const float*) {
    const uint4 qs = lds_u4(rec + lane * 16);
    const uint32_t qh = *reinterpret_cast<const uint32_t*>(rec + 512 + lane * 4);
    const float d = __half2float(*reinterpret_cast<const __half*>(rec + 640 + lane * 2));
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint64_t a0 = 0, a1 = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w = word(qs, i);
        const uint32_t lo = (w & 0x0F0F0F0Fu) | spread4_to_bit4((qh >> (4 * i)) & 0xFu);         // weights 4i..
        const uint32_t hi = ((w >> 4) & 0x0F0F0F0Fu) | spread4_to_bit4((qh >> (16 + 4 * i)) & 0xFu);  // 16 + 4i..
        a0 = dot4_codes(lo, x4[i], 16.0f, a0);
        a1 = dot4_codes(hi, x4[4 + i], 16.0f, a1);
    }
    return d * ((f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1)));
}

template <>
__device__ __forceinline__ float unit_dot<kGgufQ4_K>(const uint8_t* rec, int u, int lane, const float* x,
                                                     const float* xsum) {
    // unit u: sub-blocks 4u .. 4u + 3, the low and high nibbles of qs bytes
    // [64u, 64u + 64) (chunks 4u .. 4u + 3). The lane's 16 metadata bytes in one
    // load: fp16 d, fp16 dmin, then the 12 scale bytes; the unit's four 6-bit
    // scales and minima unpacked as the bytes of one word each.
    const uint4 meta = lds_u4(rec + 4096 + lane * 16);
    const float d = __half2float(__ushort_as_half((unsigned short)(meta.x & 0xFFFFu)));
    const float dmin = __half2float(__ushort_as_half((unsigned short)(meta.x >> 16)));
    uint32_t scw, mnw;
    if (u == 0) {  // sub-blocks 0..3: low six bits of scale bytes 0..3 and 4..7
        scw = meta.y & 0x3F3F3F3Fu;
        mnw = meta.z & 0x3F3F3F3Fu;
    } else {  // sub-blocks 4..7: nibbles of bytes 8..11, top two bits from bytes 0..3 / 4..7
        scw = (meta.w & 0x0F0F0F0Fu) | ((meta.y >> 2) & 0x30303030u);
        mnw = ((meta.w >> 4) & 0x0F0F0F0Fu) | ((meta.z >> 2) & 0x30303030u);
    }
    const float4* x4 = reinterpret_cast<const float4*>(x);
    float qacc = 0.0f, macc = 0.0f;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const uint4 q0 = lds_u4(rec + (4 * u + 2 * p) * 512 + lane * 16);      // weights 0..15 of sub-blocks 2p, 2p + 1
        const uint4 q1 = lds_u4(rec + (4 * u + 2 * p + 1) * 512 + lane * 16);  // weights 16..31
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int jj = 2 * p + h;  // sub-block within the unit: low nibbles (h = 0) or high
            uint64_t a0 = 0, a1 = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a0 = dot4_codes((word(q0, i) >> (4 * h)) & 0x0F0F0F0Fu, x4[8 * jj + i], 0.0f, a0);
                a1 = dot4_codes((word(q1, i) >> (4 * h)) & 0x0F0F0F0Fu, x4[8 * jj + 4 + i], 0.0f, a1);
            }
            const float qx = (f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1));
            qacc = fmaf((float)((scw >> (8 * jj)) & 0xFFu), qx, qacc);
            macc = fmaf((float)((mnw >> (8 * jj)) & 0xFFu), xsum[jj], macc);
        }
    }
    return d * qacc - dmin * macc;
}

template <>
__device__ __forceinline__ float unit_dot<kGgufQ6_K>(const uint8_t* rec, int u, int lane, const float* x,
                                                     const float*) {
    // unit u = weights [32 u, 32 u + 32): half h, group g of that half
    const int h = u >> 2, g = u & 3;
    const int lc = 4 * h + 2 * (g & 1);  // ql chunk pair
    const int hc = 2 * h;                // qh chunk pair
    const int lsh = (g >> 1) * 4, hsh = 2 * g;
    const uint4 l0 = lds_u4(rec + lc * 512 + lane * 16);
    const uint4 l1 = lds_u4(rec + (lc + 1) * 512 + lane * 16);
    const uint4 h0 = lds_u4(rec + 4096 + hc * 512 + lane * 16);
    const uint4 h1 = lds_u4(rec + 4096 + (hc + 1) * 512 + lane * 16);
    const int8_t* scales = reinterpret_cast<const int8_t*>(rec + 6144 + lane * 16);
    const float d = __half2float(*reinterpret_cast<const __half*>(rec + 6656 + lane * 2));
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint64_t a0 = 0, a1 = 0;  // weights 0..15 (scale 2u), 16..31 (scale 2u + 1)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c0 = ((word(l0, i) >> lsh) & 0x0F0F0F0Fu) | (((word(h0, i) >> hsh) & 0x03030303u) << 4);
        const uint32_t c1 = ((word(l1, i) >> lsh) & 0x0F0F0F0Fu) | (((word(h1, i) >> hsh) & 0x03030303u) << 4);
        a0 = dot4_codes(c0, x4[i], 32.0f, a0);
        a1 = dot4_codes(c1, x4[4 + i], 32.0f, a1);
    }
    return d * ((float)scales[2 * u] * (f2_lo(a0) + f2_hi(a0)) + (float)scales[2 * u + 1] * (f2_lo(a1) + f2_hi(a1)));
}

struct FmtArgs {
    const uint8_t* W;  // packed records
    int rows, rows_pad, k;
    const float* x;
    float* y;
    int splits;
    int* err;
};

// Grid as in the Q8_0 kernel: S == 1 persistent CTAs over row tiles, S > 1 one
// cluster per tile with the block range split over its ranks.
template <int T>
__global__ void __launch_bounds__(kFmtThreads) fmt_gemv_kernel(FmtArgs a) {
    using F = Fmt<T>;
    constexpr int kStageBytes = F::kStageRecs * F::kRec;
    constexpr int kUnitsPerStage = F::kStageRecs * F::kUnits;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* stages = smem;
    float* xs = reinterpret_cast<float*>(smem + kFmtStages * kStageBytes);
    __shared__ __align__(8) uint64_t full[kFmtStages];
    __shared__ __align__(8) uint64_t empty[kFmtStages];
    __shared__ __align__(8) uint64_t xbar;
    __shared__ float red[2][kFmtCWarps][32];
    __shared__ float part[32];

    const int nb = a.k / F::kW;
    const int S = a.splits;
    const int tiles = a.rows_pad >> 5;
    const int cl_id = blockIdx.x / S, split = blockIdx.x % S, n_cl = gridDim.x / S;
    const int my_tiles = cl_id < tiles ? (tiles - cl_id + n_cl - 1) / n_cl : 0;
    const int b0 = (split * nb) / S, b1 = ((split + 1) * nb) / S;
    const int nblk = b1 - b0;
    const int n_stage = (nblk + F::kStageRecs - 1) / F::kStageRecs;
    const int total = my_tiles * n_stage;
    const int xn = nblk * F::kW;  // this unit's slice of x
    float* xsum = xs + xn;        // Q4_K: sum of x over each 32-weight sub-block of the slice
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kFmtStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kFmtCWarps);
        }
        mbar_init(&xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kFmtCWarps) {
        if (lane == 0) {
            auto issue = [&](int g) {
                const int slot = g % kFmtStages;
                if (g >= kFmtStages) mbar_wait_bounded(&empty[slot], ((g / kFmtStages) - 1) & 1, a.err, 31);
                const int tile = cl_id + (g / n_stage) * n_cl, j = g % n_stage;
                const int bs = b0 + j * F::kStageRecs;
                const int nbs = min(F::kStageRecs, b1 - bs);
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(nbs * F::kRec));
                bulk_g2s(stages + slot * kStageBytes, a.W + ((size_t)tile * nb + bs) * F::kRec,
                         (uint32_t)(nbs * F::kRec), &full[slot]);
            };
            const int first = min(kFmtStages, total);
            for (int g = 0; g < first; ++g) issue(g);  // weights: no kernel writes them
            pdl_wait();                                // x: written by the preceding kernel
            mbar_arrive_expect_tx(&xbar, (uint32_t)(xn * 4));
            bulk_g2s(xs, a.x + (size_t)b0 * F::kW, (uint32_t)(xn * 4), &xbar);
            for (int g = first; g < total; ++g) issue(g);
        }
    } else {
        pdl_wait();
        if (tid == 0) pdl_launch_dependents();
        constexpr int kCT = kFmtCWarps * 32;
        mbar_wait_bounded(&xbar, 0, a.err, 32);
        if (T == kGgufQ4_K) {
            for (int i = warp; i < xn / 32; i += kFmtCWarps) {
                const float v = warp_sum(xs[i * 32 + lane]);
                if (lane == 0) xsum[i] = v;
            }
            named_bar_sync(1, kCT);
        }
        for (int ti = 0; ti < my_tiles; ++ti) {
            const int tile = cl_id + ti * n_cl;
            float acc = 0.0f;
            for (int j = 0; j < n_stage; ++j) {
                const int g = ti * n_stage + j;
                const int slot = g % kFmtStages;
                mbar_wait_bounded(&full[slot], (g / kFmtStages) & 1, a.err, 33);
                const int nbs = min(F::kStageRecs, nblk - j * F::kStageRecs);
                const uint8_t* st = stages + slot * kStageBytes;
#pragma unroll
                for (int v = warp; v < kUnitsPerStage; v += kFmtCWarps) {
                    const int r = v / F::kUnits, u = v % F::kUnits;
                    if (r < nbs) {
                        const int w0 = (j * F::kStageRecs + r) * F::kW + u * F::kUnitW;  // relative to the slice
                        acc += unit_dot<T>(st + r * F::kRec, u, lane, xs + w0, xsum + w0 / 32);
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
                for (int w = 0; w < kFmtCWarps; ++w) v += red[ti & 1][w][lane];
                const int row = tile * 32 + lane;
                if (S == 1) {
                    if (row < a.rows) a.y[row] = v;
                } else {
                    part[lane] = v;
                }
            }
        }
        if (S > 1) {
            __syncwarp();
            cluster_sync();
            if (split == 0 && warp == 0 && my_tiles > 0) {
                float v = part[lane];
                for (int rnk = 1; rnk < S; ++rnk) v += ld_dsmem_f32(&part[lane], (uint32_t)rnk);
                const int row = cl_id * 32 + lane;
                if (row < a.rows) a.y[row] = v;
            }
            cluster_sync();
        }
        return;
    }
    if (S > 1) {
        __syncwarp();
        cluster_sync();
        cluster_sync();
    }
}

template <int T>
size_t fmt_smem(int max_blk) {
    return (size_t)kFmtStages * Fmt<T>::kStageRecs * Fmt<T>::kRec + (size_t)max_blk * Fmt<T>::kW * 4 +
           (size_t)max_blk * Fmt<T>::kW / 32 * 4;
}

int fmt_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

template <int T>
int fmt_resident(size_t smem) {
    static std::mutex mu;
    static std::map<size_t, int> known;
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(smem);
    if (it != known.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fmt_gemv_kernel<T>, kFmtThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        n = 1;
    }
    n = std::max(n, 1);
    known[smem] = n;
    return n;
}

template <int T>
cudaError_t fmt_launch(const uint8_t* W, int rows, int k, const float* x, float* y, bool pdl, int* err,
                       cudaStream_t s) {
    using F = Fmt<T>;
    const int tiles = (rows + 31) / 32, nb = k / F::kW;
    const int sms = fmt_sm_count();
    const size_t smem1 = fmt_smem<T>(nb);
    const int cap = sms * fmt_resident<T>(smem1);
    // split each tile's block range over a cluster when the tiles cannot fill the
    // GPU, keeping at least 512 weights per split, at most 8 splits
    int S = 1;
    while (S < 8 && tiles * (S + 1) <= cap && nb / (S + 1) * F::kW >= 512) ++S;
    const size_t smem = fmt_smem<T>((nb + S - 1) / S);
    if (smem > (size_t)kFmtMaxSmem) return cudaErrorInvalidValue;
    const int grid = S == 1 ? std::min(tiles, cap) : tiles * S;
    FmtArgs a{W, rows, tiles * 32, k, x, y, S, err};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFmtThreads);
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
    return cudaLaunchKernelEx(&cfg, fmt_gemv_kernel<T>, a);
}

// ---- repack: one thread per (row, block) ---------------------------------------------
template <int T>
__global__ void pack_fmt_kernel(const uint8_t* __restrict__ src, int64_t rows, int64_t nb, uint8_t* __restrict__ dst) {
    using F = Fmt<T>;
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * nb) return;
    const int64_t n = idx / nb, b = idx % nb;
    const uint8_t* blk = src + idx * F::kBytes;
    const int64_t tile = n >> 5;
    const int lane = (int)(n & 31);
    uint8_t* rec = dst + (tile * nb + b) * F::kRec;
    if (T == kGgufQ5_0) {
        for (int i = 0; i < 16; ++i) rec[lane * 16 + i] = blk[6 + i];
        for (int i = 0; i < 4; ++i) rec[512 + lane * 4 + i] = blk[2 + i];
        for (int i = 0; i < 2; ++i) rec[640 + lane * 2 + i] = blk[i];
    } else if (T == kGgufQ4_K) {
        for (int c = 0; c < 8; ++c)
            for (int i = 0; i < 16; ++i) rec[c * 512 + lane * 16 + i] = blk[16 + 16 * c + i];
        for (int i = 0; i < 16; ++i) rec[4096 + lane * 16 + i] = blk[i];
    } else {
        for (int c = 0; c < 8; ++c)
            for (int i = 0; i < 16; ++i) rec[c * 512 + lane * 16 + i] = blk[16 * c + i];
        for (int c = 0; c < 4; ++c)
            for (int i = 0; i < 16; ++i) rec[4096 + c * 512 + lane * 16 + i] = blk[128 + 16 * c + i];
        for (int i = 0; i < 16; ++i) rec[6144 + lane * 16 + i] = blk[192 + i];
        for (int i = 0; i < 2; ++i) rec[6656 + lane * 2 + i] = blk[208 + i];
    }
}

template <int T>
cudaError_t fmt_pack(const uint8_t* src, int64_t rows, int64_t k, uint8_t* dst, cudaStream_t s) {
    const int64_t nb = k / Fmt<T>::kW, total = rows * nb;
    cudaError_t e = cudaMemsetAsync(dst, 0, (size_t)fmt_packed_bytes(T, rows, k), s);
    if (e != cudaSuccess || total == 0) return e;
    pack_fmt_kernel<T><<<(unsigned)((total + 255) / 256), 256, 0, s>>>(src, rows, nb, dst);
    return cudaGetLastError();
}

}  // namespace

bool fmt_supported(int type) { return type == kGgufQ5_0 || type == kGgufQ4_K || type == kGgufQ6_K; }

int fmt_block_weights(int type) {
    switch (type) {
        case kGgufQ5_0: return Fmt<kGgufQ5_0>::kW;
        case kGgufQ4_K: return Fmt<kGgufQ4_K>::kW;
        case kGgufQ6_K: return Fmt<kGgufQ6_K>::kW;
    }
    return 0;
}

int64_t fmt_packed_bytes(int type, int64_t rows, int64_t k) {
    const int64_t rp = round_up32(rows);
    switch (type) {
        case kGgufQ5_0: return rp * (k / 32) * 22;
        case kGgufQ4_K: return rp * (k / 256) * 144;
        case kGgufQ6_K: return rp * (k / 256) * 210;
    }
    return 0;
}

int64_t fmt_max_k(int type) {
    // the x slice of an unsplit unit must fit in shared memory beside the ring
    const int w = fmt_block_weights(type);
    if (!w) return 0;
    int64_t ring = 0;
    switch (type) {
        case kGgufQ5_0: ring = fmt_smem<kGgufQ5_0>(0); break;
        case kGgufQ4_K: ring = fmt_smem<kGgufQ4_K>(0); break;
        case kGgufQ6_K: ring = fmt_smem<kGgufQ6_K>(0); break;
    }
    return (kFmtMaxSmem - ring) * 32 / 132 / w * w;  // 4 bytes of x + 4 / 32 of a sub-block sum per weight
}

cudaError_t launch_pack_fmt(int type, const uint8_t* src, int64_t rows, int64_t k, uint8_t* dst, cudaStream_t s) {
    switch (type) {
        case kGgufQ5_0: return fmt_pack<kGgufQ5_0>(src, rows, k, dst, s);
        case kGgufQ4_K: return fmt_pack<kGgufQ4_K>(src, rows, k, dst, s);
        case kGgufQ6_K: return fmt_pack<kGgufQ6_K>(src, rows, k, dst, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_gemv_fmt(int type, const uint8_t* packed, int rows, int k, const float* x, float* y, bool pdl,
                            int* err, cudaStream_t s) {
    switch (type) {
        case kGgufQ5_0: return fmt_launch<kGgufQ5_0>(packed, rows, k, x, y, pdl, err, s);
        case kGgufQ4_K: return fmt_launch<kGgufQ4_K>(packed, rows, k, x, y, pdl, err, s);
        case kGgufQ6_K: return fmt_launch<kGgufQ6_K>(packed, rows, k, x, y, pdl, err, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t init_gemv_fmt_attributes() {
    cudaError_t e = cudaFuncSetAttribute(fmt_gemv_kernel<kGgufQ5_0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kFmtMaxSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fmt_gemv_kernel<kGgufQ4_K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kFmtMaxSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fmt_gemv_kernel<kGgufQ6_K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kFmtMaxSmem);
    return e;
}

}  // namespace lq8
