// Q8_0 matrix-matrix product for prefill rows (T > 1): C[t][n] = X[t][:] . W[n][:],
// the counterpart of the quantised mat-mat kernel on "生成一个 token"
// (prefill 和 decode：同一个 forward，不同的路).
//
// CUDA-core version: a 64-token x 64-row tile per CTA, 32-weight (one Q8_0
// block) k-steps. The CTA dequantises its weight block into shared memory
// (d * q, exact in f32), stages the matching activation block, and each
// thread accumulates a 4 x 4 sub-tile in f32. The epilogues are the ones of
// the matrix-vector kernel, applied per (token, row pair).
#include "epilogue.cuh"
#include "ptx.cuh"

namespace lq8 {

constexpr int kBM = 64;   // tokens per CTA
constexpr int kBN = 64;   // weight rows per CTA
constexpr int kBK = 32;   // one Q8_0 block
constexpr int kGemmThreads = 256;

template <int EPI>
__global__ void __launch_bounds__(kGemmThreads) q8_gemm_simt_kernel(PackedQ8 W, const float* __restrict__ X,
                                                                    int m, int ldx, EpiArgs e) {
    __shared__ __align__(16) float Xs[kBK][kBM + 4];
    __shared__ __align__(16) float Ws[kBK][kBN + 4];
    pdl_wait();
    pdl_launch_dependents();
    const int k = W.k, nb = k >> 5;
    const int n0 = blockIdx.x * kBN, t0 = blockIdx.y * kBM;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

    for (int kb = 0; kb < nb; ++kb) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int f = tid + i * kGemmThreads;
            const int row = f >> 3, c4 = f & 7;
            const int t = t0 + row;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < m) v = *reinterpret_cast<const float4*>(X + (int64_t)t * ldx + kb * 32 + c4 * 4);
            Xs[c4 * 4 + 0][row] = v.x;
            Xs[c4 * 4 + 1][row] = v.y;
            Xs[c4 * 4 + 2][row] = v.z;
            Xs[c4 * 4 + 3][row] = v.w;
        }
        if (tid < 128) {
            const int rr = tid >> 1, c = tid & 1;
            const int n = n0 + rr;
            float w[16];
            if (n < W.rows_pad) {
                const int64_t tile = n >> 5, lane = n & 31;
                const uint4 q = *reinterpret_cast<const uint4*>(
                    W.qs + ((tile * (k >> 4) + 2 * kb + c) * 512 + lane * 16));
                const float d = __half2float(W.d[(tile * nb + kb) * 32 + lane]);
                const uint32_t ws[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = d * (float)(int8_t)((ws[i >> 2] >> (8 * (i & 3))) & 0xff);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Ws[c * 16 + i][rr] = w[i];
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < kBK; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&Xs[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&Ws[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = t0 + ty * 4 + i;
        if (t >= m) continue;
        const int n = n0 + tx * 4;
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
            const int r = n + j;
            if (r >= W.rows) continue;
            const float a = acc[i][j], b = acc[i][j + 1];
            if (EPI == EPI_STORE) {
                e.y[(int64_t)t * e.ldy + r] = a;
                if (r + 1 < W.rows) e.y[(int64_t)t * e.ldy + r + 1] = b;
            } else if (EPI == EPI_RESIDUAL) {
                e.y[(int64_t)t * e.ldy + r] += a;
                if (r + 1 < W.rows) e.y[(int64_t)t * e.ldy + r + 1] += b;
            } else if (EPI == EPI_QKV) {
                epi_qkv_pair(e, t, e.pos0 + t, r, a, b);
            } else if (EPI == EPI_SILU) {
                e.a_out[(int64_t)t * e.lda + (r >> 1)] = silu_f32(a) * b;
            }
        }
    }
}

cudaError_t launch_gemm(const PackedQ8& W, const float* X, int m, int ldx, int epi,
                        const EpiArgs& e, bool pdl, cudaStream_t s) {
    dim3 grid((W.rows_pad + kBN - 1) / kBN, (m + kBM - 1) / kBM);
    dim3 block(kGemmThreads);
    switch (epi) {
        case EPI_STORE: return launch_ex(q8_gemm_simt_kernel<EPI_STORE>, grid, block, 0, s, pdl, W, X, m, ldx, e);
        case EPI_RESIDUAL: return launch_ex(q8_gemm_simt_kernel<EPI_RESIDUAL>, grid, block, 0, s, pdl, W, X, m, ldx, e);
        case EPI_QKV: return launch_ex(q8_gemm_simt_kernel<EPI_QKV>, grid, block, 0, s, pdl, W, X, m, ldx, e);
        case EPI_SILU: return launch_ex(q8_gemm_simt_kernel<EPI_SILU>, grid, block, 0, s, pdl, W, X, m, ldx, e);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lq8
