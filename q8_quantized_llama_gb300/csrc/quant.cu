// Q8_0 quantisation, repacking into the device layout, embedding gather and
// the stand-alone RMSNorm used by the prefill path.
#include "kernels.cuh"
#include "ptx.cuh"

namespace lq8 {

PackedQ8 packed_view(const uint8_t* base, int64_t rows, int64_t k) {
    PackedQ8 p;
    p.qs = reinterpret_cast<const int8_t*>(base);
    p.d = reinterpret_cast<const __half*>(base + packed_d_offset_bytes(rows, k));
    p.rows = (int)rows;
    p.rows_pad = (int)round_up32(rows);
    p.k = (int)k;
    return p;
}

// ---------------------------------------------------------------------------
// Quantise: one thread per 32-weight block. d = max|w| / 127 with an IEEE f32
// division, codes q = round(w / d) (IEEE f32 division, roundf = ties away from
// zero, clamp to +-127, d == 0 -> 0), d stored as fp16 round-to-nearest-even.
// ---------------------------------------------------------------------------
__global__ void quantize_q8_0_kernel(const float* __restrict__ w, int64_t n_blocks,
                                     uint16_t* __restrict__ out) {
    int64_t blk = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (blk >= n_blocks) return;
    const float4* src = reinterpret_cast<const float4*>(w + blk * 32);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4 f = src[i];
        v[4 * i + 0] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float d = __fdiv_rn(amax, 127.0f);
    const __half dh = __float2half_rn(d);
    uint8_t q[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        float r = 0.0f;
        if (d != 0.0f) {
            r = roundf(__fdiv_rn(v[i], d));
            r = fminf(fmaxf(r, -127.0f), 127.0f);
        }
        q[i] = (uint8_t)(int8_t)(int)r;
    }
    // 34-byte record, 2-byte aligned: 17 half-words, little-endian.
    uint16_t* dst = out + blk * 17;
    dst[0] = __half_as_ushort(dh);
#pragma unroll
    for (int i = 0; i < 16; ++i) dst[1 + i] = (uint16_t)q[2 * i] | ((uint16_t)q[2 * i + 1] << 8);
}

cudaError_t launch_quantize(const float* w, int64_t rows, int64_t k, uint8_t* out, cudaStream_t s) {
    int64_t nb = rows * (k / 32);
    if (nb == 0) return cudaSuccess;
    const int threads = 256;
    int64_t grid = (nb + threads - 1) / threads;
    quantize_q8_0_kernel<<<(unsigned)grid, threads, 0, s>>>(w, nb, reinterpret_cast<uint16_t*>(out));
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Repack: one thread per (source row, block). Source row n lands on packed row
// row_offset + n * row_stride (used to concatenate Q/K/V and to interleave the
// gate and up rows).
// ---------------------------------------------------------------------------
__global__ void pack_q8_0_kernel(const uint16_t* __restrict__ src, int64_t rows, int64_t k,
                                 uint8_t* __restrict__ qs, __half* __restrict__ dsc,
                                 int64_t row_offset, int64_t row_stride) {
    const int64_t nb = k / 32;
    int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * nb) return;
    const int64_t n = idx / nb, b = idx % nb;
    const uint16_t* rec = src + idx * 17;
    uint32_t words[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) words[i] = (uint32_t)rec[1 + 2 * i] | ((uint32_t)rec[2 + 2 * i] << 16);
    const int64_t dn = row_offset + n * row_stride;
    const int64_t tile = dn >> 5, lane = dn & 31;
    dsc[(tile * nb + b) * 32 + lane] = __ushort_as_half(rec[0]);
    uint8_t* q0 = qs + ((tile * (k / 16) + 2 * b) * 512 + lane * 16);
    *reinterpret_cast<uint4*>(q0) = make_uint4(words[0], words[1], words[2], words[3]);
    *reinterpret_cast<uint4*>(q0 + 512) = make_uint4(words[4], words[5], words[6], words[7]);
}

cudaError_t launch_pack(const uint8_t* q8, int64_t rows, int64_t k, uint8_t* packed_base,
                        int64_t dst_rows, int64_t row_offset, int64_t row_stride, cudaStream_t s) {
    int64_t total = rows * (k / 32);
    if (total == 0) return cudaSuccess;
    uint8_t* qs = packed_base;
    __half* d = reinterpret_cast<__half*>(packed_base + packed_d_offset_bytes(dst_rows, k));
    const int threads = 256;
    pack_q8_0_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, s>>>(
        reinterpret_cast<const uint16_t*>(q8), rows, k, qs, d, row_offset, row_stride);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Embedding: x[t] = dequant(E[id_t]); ids from device memory, or (decode) the
// token in the device state. An id outside [0, n_vocab) is recorded in
// st_err->err and row 0 is used.
// ---------------------------------------------------------------------------
__global__ void embed_kernel(PackedQ8 E, const int32_t* __restrict__ ids, const DevState* st_token,
                             DevState* st_err, float* __restrict__ x, int n_vocab, unsigned long long* stamp) {
    if (threadIdx.x == 0) stamp_at(stamp, 0);
    pdl_wait();
    pdl_launch_dependents();
    if (threadIdx.x == 0) stamp_at(stamp, 1);
    const int t = blockIdx.x;
    int id = ids ? ids[t] : st_token->token;
    if (id < 0 || id >= n_vocab) {
        if (threadIdx.x == 0 && st_err) st_err->err = 4;  // LQ8_ERR_TOKEN
        id = 0;
    }
    const int k = E.k, nchunk = k >> 4;
    const int64_t tile = id >> 5, lane = id & 31;
    const int8_t* qrow = E.qs + tile * (int64_t)k * 32 + lane * 16;
    const __half* drow = E.d + tile * (int64_t)(k >> 5) * 32 + lane;
    float* xo = x + (int64_t)t * k;
    for (int j = threadIdx.x; j < nchunk; j += blockDim.x) {
        const uint4 w = *reinterpret_cast<const uint4*>(qrow + (int64_t)j * 512);
        const float d = __half2float(drow[(j >> 1) * 32]);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        float out[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) out[i] = d * (float)(int8_t)((ws[i >> 2] >> (8 * (i & 3))) & 0xff);
        float4* dst = reinterpret_cast<float4*>(xo + j * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(out[4 * i], out[4 * i + 1], out[4 * i + 2], out[4 * i + 3]);
    }
}

cudaError_t launch_embed(const PackedQ8& E, const int32_t* ids, int T, const DevState* st_token,
                         DevState* st_err, float* x, int n_vocab, bool pdl, cudaStream_t s,
                         unsigned long long* stamp) {
    return launch_ex(embed_kernel, dim3(T), dim3(128), 0, s, pdl, E, ids, st_token, st_err, x, n_vocab, stamp);
}

__global__ void stamp_kernel(unsigned long long* stamp) {
    if (threadIdx.x == 0) stamp_at(stamp, 0);
    pdl_wait();
    if (threadIdx.x == 0) stamp_at(stamp, 1);
}

cudaError_t launch_stamp(unsigned long long* stamp, cudaStream_t s) {
    return launch_ex(stamp_kernel, dim3(1), dim3(32), 0, s, true, stamp);
}

// ---------------------------------------------------------------------------
// RMSNorm rows: y = x * g / sqrt(mean(x^2) + eps), f32.
// ---------------------------------------------------------------------------
// y is written when non-null. With hl, the kernel also writes the operand of
// the tensor-core product that reads the normalised rows: rowmax[row] = the
// row's largest |y| and hl[row] = y scaled by the row's power of two and split
// into f16 hi / lo (common.cuh), from the same f32 values y holds.
__global__ void rmsnorm_kernel(const float* __restrict__ x, const float* __restrict__ g, float eps,
                               int k, float* __restrict__ y, float* __restrict__ rowmax, __half* __restrict__ hl) {
    __shared__ float red[32];
    pdl_wait();
    pdl_launch_dependents();
    const float* xr = x + (int64_t)blockIdx.x * k;
    float ss = 0.0f;
    for (int i = threadIdx.x * 4; i < k; i += blockDim.x * 4) {
        float4 v = *reinterpret_cast<const float4*>(xr + i);
        ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
        v = warp_sum(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float r = 1.0f / sqrtf(red[0] / (float)k + eps);
    auto norm4 = [&](int i) {
        const float4 v = *reinterpret_cast<const float4*>(xr + i);
        const float4 gg = *reinterpret_cast<const float4*>(g + i);
        return make_float4(v.x * r * gg.x, v.y * r * gg.y, v.z * r * gg.z, v.w * r * gg.w);
    };
    float mx = 0.0f;
    for (int i = threadIdx.x * 4; i < k; i += blockDim.x * 4) {
        const float4 o = norm4(i);
        if (y) *reinterpret_cast<float4*>(y + (int64_t)blockIdx.x * k + i) = o;
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(o.x), fabsf(o.y)), fmaxf(fabsf(o.z), fabsf(o.w))));
    }
    if (!hl) return;
    mx = warp_max(mx);
    __syncthreads();  // every thread has read the sum of squares from red[0]
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
        v = warp_max(v);
        if (threadIdx.x == 0) {
            rowmax[blockIdx.x] = v;
            red[0] = v;
        }
    }
    __syncthreads();
    const float sc = pow2f(row_shift(red[0]));
    __half* hr = hl + (int64_t)blockIdx.x * 2 * k;
    for (int i = threadIdx.x * 4; i < k; i += blockDim.x * 4) {
        const float4 o = norm4(i);  // the same products as above: the same f32 values
        store_split4(hr, i, o.x * sc, o.y * sc, o.z * sc, o.w * sc);
    }
}

cudaError_t launch_rmsnorm(const float* x, const float* g, float eps, int m, int k, float* y, bool pdl,
                           cudaStream_t s, const SplitRows* split) {
    return launch_ex(rmsnorm_kernel, dim3(m), dim3(256), 0, s, pdl, x, g, eps, k, y,
                     split ? split->rowmax : nullptr, split ? split->hl : nullptr);
}

__global__ void set_state_kernel(DevState* st, int pos, int token, int n_out) {
    if (pos >= 0) st->pos = pos;
    if (token >= 0) st->token = token;
    if (n_out >= 0) st->n_out = n_out;
}

cudaError_t launch_set_state(DevState* st, int pos, int token, int n_out, cudaStream_t s) {
    set_state_kernel<<<1, 1, 0, s>>>(st, pos, token, n_out);
    return cudaGetLastError();
}

// A barrier that nothing completes: the bounded wait gives up after ~1 s and
// records `code` (the failure path every kernel takes on a lost wait).
__global__ void wait_timeout_kernel(int* err, int code) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    mbar_wait_bounded(&bar, 0, err, code);
}

cudaError_t launch_wait_timeout(int* err, int code, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(err, code);
    return cudaGetLastError();
}

}  // namespace lq8
