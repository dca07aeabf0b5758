// Q8_0 matrix-vector product for one token (decode, and the lm_head of every
// forward): the counterpart of the quantised mat-vec kernel the pages name on
// "生成一个 token" (prefill 和 decode：同一个 forward，不同的路), written for
// sm_103a.
//
// One CTA (8 warps) per tile of 32 output rows. The activation vector is staged
// once in shared memory (RMSNorm applied there when the step fuses it); each
// warp takes a contiguous range of 32-weight blocks, lane l owns row
// tile*32 + l and streams its codes with 128-bit loads: a warp instruction
// reads 512 contiguous bytes of the packed layout. Codes become f32 exactly
// (byte-permute into 2^23 + u, one packed subtraction per pair) and are
// multiplied into f32x2 accumulators; each block's sum is scaled by its fp16
// d. Warp partials are summed in shared memory in warp order (deterministic),
// then warp 0 runs the epilogue on its 32 rows.
#include "epilogue.cuh"

namespace lq8 {

constexpr int kGemvWarps = 8;
constexpr int kGemvThreads = kGemvWarps * 32;
constexpr int kGemvUnroll = 4;

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

template <int EPI, bool NORM>
__global__ void __launch_bounds__(kGemvThreads) q8_gemv_kernel(PackedQ8 W, const float* __restrict__ x,
                                                               const float* __restrict__ g, float eps,
                                                               EpiArgs e) {
    extern __shared__ float4 smem4[];
    float* sx = reinterpret_cast<float*>(smem4);
    __shared__ float red[kGemvWarps][33];
    __shared__ float s_rscale;

    const int k = W.k, nb = k >> 5, tile = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- prologue: stage x (and normalise it) ----------------------------
    float ss = 0.0f;
    for (int i = tid * 4; i < k; i += kGemvThreads * 4) {
        const float4 v = *reinterpret_cast<const float4*>(x + i);
        *reinterpret_cast<float4*>(sx + i) = v;
        if (NORM) {
            ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss);
            ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
        }
    }
    if (NORM) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp][0] = ss;
        __syncthreads();
        if (tid == 0) {
            float t = 0.0f;
#pragma unroll
            for (int w = 0; w < kGemvWarps; ++w) t += red[w][0];
            s_rscale = 1.0f / sqrtf(t / (float)k + eps);
        }
        __syncthreads();
        const float r = s_rscale;
        for (int i = tid * 4; i < k; i += kGemvThreads * 4) {
            float4 v = *reinterpret_cast<float4*>(sx + i);
            const float4 gg = *reinterpret_cast<const float4*>(g + i);
            v.x = v.x * r * gg.x; v.y = v.y * r * gg.y; v.z = v.z * r * gg.z; v.w = v.w * r * gg.w;
            *reinterpret_cast<float4*>(sx + i) = v;
        }
    }
    __syncthreads();

    // ---- main loop -----------------------------------------------------------
    const int b0 = (warp * nb) / kGemvWarps, b1 = ((warp + 1) * nb) / kGemvWarps;
    const int8_t* qp = W.qs + (int64_t)tile * k * 32 + lane * 16;
    const __half* dp = W.d + (int64_t)tile * nb * 32 + lane;
    float acc = 0.0f;
    int b = b0;
    for (; b + kGemvUnroll <= b1; b += kGemvUnroll) {
        uint4 q[2 * kGemvUnroll];
        unsigned short dh[kGemvUnroll];
#pragma unroll
        for (int u = 0; u < kGemvUnroll; ++u) {
            q[2 * u] = ld_stream_u4(qp + (int64_t)(2 * (b + u)) * 512);
            q[2 * u + 1] = ld_stream_u4(qp + (int64_t)(2 * (b + u) + 1) * 512);
            dh[u] = ld_stream_u16(dp + (b + u) * 32);
        }
#pragma unroll
        for (int u = 0; u < kGemvUnroll; ++u)
            acc = fmaf(__half2float(__ushort_as_half(dh[u])), block_dot32(q[2 * u], q[2 * u + 1], sx + 32 * (b + u)), acc);
    }
    for (; b < b1; ++b) {
        const uint4 q0 = ld_stream_u4(qp + (int64_t)(2 * b) * 512);
        const uint4 q1 = ld_stream_u4(qp + (int64_t)(2 * b + 1) * 512);
        const unsigned short dh = ld_stream_u16(dp + b * 32);
        acc = fmaf(__half2float(__ushort_as_half(dh)), block_dot32(q0, q1, sx + 32 * b), acc);
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp != 0) return;

    // ---- epilogue (warp 0, rows tile*32 + lane) -------------------------------
    float v = 0.0f;
#pragma unroll
    for (int w = 0; w < kGemvWarps; ++w) v += red[w][lane];
    const int r = tile * 32 + lane;
    const bool valid = r < W.rows;
    if (EPI == EPI_STORE) {
        if (valid) e.y[r] = v;
    } else if (EPI == EPI_RESIDUAL) {
        if (valid) e.y[r] += v;
    } else if (EPI == EPI_QKV) {
        const float other = __shfl_xor_sync(0xffffffffu, v, 1);
        const int pos = e.state ? e.state->pos : e.pos0;
        if (!(lane & 1) && valid) epi_qkv_pair(e, 0, pos, r, v, other);
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
        if (lane == 0) {
            atomicMax(e.best_key, key);
            __threadfence();
            const unsigned int ticket = atomicAdd(e.done_count, 1u);
            if (ticket == gridDim.x - 1) {
                __threadfence();
                const unsigned long long best = atomicExch(e.best_key, 0ull);
                atomicExch(e.done_count, 0u);
                const int tok = argmax_key_index(best);
                DevState* st = e.st;
                st->token = tok;
                if (e.out_ids) e.out_ids[st->n_out] = tok;
                st->n_out += 1;
                st->pos = e.pos_after >= 0 ? e.pos_after : st->pos + 1;
            }
        }
    }
}

template <int EPI, bool NORM>
static cudaError_t gemv_launch_one(const PackedQ8& W, const float* x, const float* g, float eps,
                                   const EpiArgs& e, cudaStream_t s) {
    const size_t smem = (size_t)W.k * sizeof(float);
    q8_gemv_kernel<EPI, NORM><<<W.rows_pad / 32, kGemvThreads, smem, s>>>(W, x, g, eps, e);
    return cudaGetLastError();
}

constexpr int kGemvMaxSmem = 200 * 1024;  // activation vectors up to 51200 floats

template <int EPI>
static cudaError_t gemv_set_attr() {
    cudaError_t err = cudaFuncSetAttribute(q8_gemv_kernel<EPI, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kGemvMaxSmem);
    if (err != cudaSuccess) return err;
    return cudaFuncSetAttribute(q8_gemv_kernel<EPI, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kGemvMaxSmem);
}

// Raise the dynamic shared-memory limit of every instantiation once per device
// (before any stream capture).
cudaError_t init_gemv_attributes() {
    cudaError_t err = gemv_set_attr<EPI_STORE>();
    if (err == cudaSuccess) err = gemv_set_attr<EPI_RESIDUAL>();
    if (err == cudaSuccess) err = gemv_set_attr<EPI_QKV>();
    if (err == cudaSuccess) err = gemv_set_attr<EPI_SILU>();
    if (err == cudaSuccess) err = gemv_set_attr<EPI_ARGMAX>();
    return err;
}

cudaError_t launch_gemv(const PackedQ8& W, const float* x, const float* norm_g, float eps, int epi,
                        const EpiArgs& e, cudaStream_t s) {
    const bool norm = norm_g != nullptr;
    switch (epi) {
        case EPI_STORE:
            return norm ? gemv_launch_one<EPI_STORE, true>(W, x, norm_g, eps, e, s)
                        : gemv_launch_one<EPI_STORE, false>(W, x, norm_g, eps, e, s);
        case EPI_RESIDUAL:
            return norm ? gemv_launch_one<EPI_RESIDUAL, true>(W, x, norm_g, eps, e, s)
                        : gemv_launch_one<EPI_RESIDUAL, false>(W, x, norm_g, eps, e, s);
        case EPI_QKV:
            return norm ? gemv_launch_one<EPI_QKV, true>(W, x, norm_g, eps, e, s)
                        : gemv_launch_one<EPI_QKV, false>(W, x, norm_g, eps, e, s);
        case EPI_SILU:
            return norm ? gemv_launch_one<EPI_SILU, true>(W, x, norm_g, eps, e, s)
                        : gemv_launch_one<EPI_SILU, false>(W, x, norm_g, eps, e, s);
        case EPI_ARGMAX:
            return norm ? gemv_launch_one<EPI_ARGMAX, true>(W, x, norm_g, eps, e, s)
                        : gemv_launch_one<EPI_ARGMAX, false>(W, x, norm_g, eps, e, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lq8
