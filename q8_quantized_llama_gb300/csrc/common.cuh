// Shared device helpers for the sm_103a kernels: the packed Q8_0 layout,
// exact int8 -> f32 conversion, packed f32x2 arithmetic and warp reductions.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace lq8 {

// ---------------------------------------------------------------------------
// Packed device layout of a Q8_0 matrix W[rows][k] (k % 32 == 0).
//
// Rows are grouped in tiles of 32 (rows padded with zero rows up to a
// multiple of 32). Codes: for tile t and 16-code chunk j of the row, the 32
// rows' 16-byte pieces lie next to each other, so one warp-wide 128-bit load
// (lane = row within the tile) reads 512 contiguous bytes:
//   qs byte offset(n, kk) = ((n / 32) * (k / 16) + kk / 16) * 512 + (n % 32) * 16 + kk % 16
// Scales: fp16, for tile t and block b the 32 rows' scales are contiguous:
//   d index(n, b) = ((n / 32) * (k / 32) + b) * 32 + n % 32
// Same 34 bytes per 32 weights as the Q8_0 block; only the order differs.
// ---------------------------------------------------------------------------
struct PackedQ8 {
    const int8_t* qs;
    const __half* d;
    int rows;      // logical rows
    int rows_pad;  // rows rounded up to 32
    int k;
};

__host__ __device__ inline int64_t packed_qs_bytes(int64_t rows_pad, int64_t k) { return rows_pad * k; }
__host__ __device__ inline int64_t packed_d_count(int64_t rows_pad, int64_t k) { return rows_pad * (k / 32); }
__host__ __device__ inline int64_t round_up32(int64_t x) { return (x + 31) / 32 * 32; }
// Total bytes, with the scale array starting 256-byte aligned after the codes.
__host__ __device__ inline int64_t packed_total_bytes(int64_t rows, int64_t k) {
    int64_t rp = round_up32(rows);
    int64_t qb = (packed_qs_bytes(rp, k) + 255) / 256 * 256;
    return qb + packed_d_count(rp, k) * 2;
}
__host__ __device__ inline int64_t packed_d_offset_bytes(int64_t rows, int64_t k) {
    int64_t rp = round_up32(rows);
    return (packed_qs_bytes(rp, k) + 255) / 256 * 256;
}

// ---------------------------------------------------------------------------
// Exact int8 -> f32: the byte b (two's complement q) is XORed with 0x80 to give
// u = q + 128 in [0, 255]; the float with bit pattern 0x4B0000uu is 2^23 + u
// exactly, and subtracting 2^23 + 128 leaves q exactly. One PRMT per code plus
// one packed subtraction per two codes.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
    return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t sub_f2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Two codes (bytes i and i+1 of the XORed word u) as an exact f32 pair.
template <int I>
__device__ __forceinline__ uint64_t codes2_f2(uint32_t u) {
    const uint32_t lo = __byte_perm(u, 0x4B000000u, 0x7540 + I);
    const uint32_t hi = __byte_perm(u, 0x4B000000u, 0x7540 + I + 1);
    const uint64_t biased = (uint64_t)lo | ((uint64_t)hi << 32);
    const float off = 8388736.0f;  // 2^23 + 128
    return sub_f2(biased, pack_f2(off, off));
}

// acc (two partial sums) += codes(4 bytes of w) * x[0..3]
__device__ __forceinline__ uint64_t dot4_acc(uint32_t w, float4 x, uint64_t acc) {
    const uint32_t u = w ^ 0x80808080u;
    acc = fma_f2(codes2_f2<0>(u), pack_f2(x.x, x.y), acc);
    acc = fma_f2(codes2_f2<2>(u), pack_f2(x.z, x.w), acc);
    return acc;
}

// One Q8_0 block of a 32-row tile against 32 values of x (lane = row): codes
// at blk (two 512-byte halves, 16 bytes per lane), as two packed partial sums.
__device__ __forceinline__ float block_dot_lane(const uint8_t* blk, int lane, const float* x) {
    const uint4 q0 = *reinterpret_cast<const uint4*>(blk + lane * 16);
    const uint4 q1 = *reinterpret_cast<const uint4*>(blk + 512 + lane * 16);
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint64_t a0 = 0, a1 = 0;
    a0 = dot4_acc(q0.x, x4[0], a0); a1 = dot4_acc(q1.x, x4[4], a1);
    a0 = dot4_acc(q0.y, x4[1], a0); a1 = dot4_acc(q1.y, x4[5], a1);
    a0 = dot4_acc(q0.z, x4[2], a0); a1 = dot4_acc(q1.z, x4[6], a1);
    a0 = dot4_acc(q0.w, x4[3], a0); a1 = dot4_acc(q1.w, x4[7], a1);
    return (f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1));
}

// sum over blocks b = b0, b0 + step, ... < b1 of d_b (codes_b . x_b) for one
// 32-row tile held in shared memory (codes of block b at tw + 1024 b, the fp16
// scales after nb_all blocks, x of block b at xs + 32 b). Two blocks per step
// with independent chains, so the second block's loads and products overlap
// the first's (the latency of these short loops is what the decode kernels
// wait on).
__device__ __forceinline__ float tile_blocks_dot(const uint8_t* tw, int nb_all, int b0, int step, int b1, int lane,
                                                 const float* xs) {
    const __half* ds = reinterpret_cast<const __half*>(tw + (size_t)nb_all * 1024);
    float acc0 = 0.0f, acc1 = 0.0f;
    int b = b0;
    for (; b + step < b1; b += 2 * step) {
        const float d0 = __half2float(ds[b * 32 + lane]);
        const float d1 = __half2float(ds[(b + step) * 32 + lane]);
        const float s0 = block_dot_lane(tw + (size_t)b * 1024, lane, xs + b * 32);
        const float s1 = block_dot_lane(tw + (size_t)(b + step) * 1024, lane, xs + (b + step) * 32);
        acc0 = fmaf(d0, s0, acc0);
        acc1 = fmaf(d1, s1, acc1);
    }
    if (b < b1) acc0 = fmaf(__half2float(ds[b * 32 + lane]), block_dot_lane(tw + (size_t)b * 1024, lane, xs + b * 32), acc0);
    return acc0 + acc1;
}

// Exact scalar code extraction (used where speed does not matter).
__device__ __forceinline__ float code_to_f32(int8_t q) { return (float)q; }

// ---------------------------------------------------------------------------
// Warp reductions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// ---------------------------------------------------------------------------
// Tensor-core operand of prefill rows: each token row x is scaled by 2^s, s
// the exponent that brings the row's largest |x| into [2^14, 2^15) (clamped so
// that 2^s and 2^-s are normal f32 numbers), and x 2^s = hi + lo is split into
// two f16 numbers (hi = x 2^s rounded to f16, lo = the remainder rounded to
// f16). Row layout: per 32-wide k-block the 32 hi values, then the 32 lo
// values (2k halves per row; one 128-byte row per k-block, the MMA's K-major
// operand row).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int row_shift(float mx) {
    const int e = (int)((__float_as_uint(mx) >> 23) & 0xFFu) - 127;
    return max(-126, min(126, 14 - e));
}
__device__ __forceinline__ float pow2f(int s) { return __uint_as_float((uint32_t)(s + 127) << 23); }

// Elements i .. i + 3 (i a multiple of 4) of a row, already multiplied by the
// row's 2^s, into the row's hi / lo halves (hl = the row's first half).
__device__ __forceinline__ void store_split4(__half* hl, int i, float a, float b, float c, float d) {
    const __half2 h0 = __floats2half2_rn(a, b), h1 = __floats2half2_rn(c, d);
    const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
    const __half2 l0 = __floats2half2_rn(a - f0.x, b - f0.y), l1 = __floats2half2_rn(c - f1.x, d - f1.y);
    __half* blk = hl + (size_t)(i >> 5) * 64 + (i & 31);
    uint2 hw, lw;
    hw.x = *reinterpret_cast<const uint32_t*>(&h0);
    hw.y = *reinterpret_cast<const uint32_t*>(&h1);
    lw.x = *reinterpret_cast<const uint32_t*>(&l0);
    lw.y = *reinterpret_cast<const uint32_t*>(&l1);
    *reinterpret_cast<uint2*>(blk) = hw;
    *reinterpret_cast<uint2*>(blk + 32) = lw;
}

// Streaming 128-bit load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ unsigned short ld_stream_u16(const void* p) {
    unsigned short r;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// Order-preserving map of an f32 to u32 (for a packed max / lowest-index key).
__device__ __forceinline__ uint32_t f32_order_key(float v) {
    uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    return ((unsigned long long)f32_order_key(v) << 32) | (unsigned long long)(~(uint32_t)idx);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long key) {
    return (int)(~(uint32_t)(key & 0xffffffffull));
}

}  // namespace lq8
