// The MLP half of a decode layer (T = 1) as ONE kernel: RMSNorm -> gate/up +
// SiLU -> down projection ("量化 llama 的一次前向", forward, mlp: the same
// steps as the gate/up and down kernels, one launch). CTA c owns 16 entries
// of the SiLU product a = silu(W_g y) * (W_u y) (gate/up row tile c of the
// row-interleaved [W_g;W_u]) and multiplies them into the matching 16-column
// half of W_down's block column c / 2 (one 512-byte chunk of every row tile
// in the packed layout): a partial of W_down a over all h rows. The CTAs form
// clusters of 16; each partial row goes (st.async, completing the receiver's
// mbarrier) to the CTA of its cluster that owns the row, which adds the 16 in
// rank order and writes the cluster's partial. The next kernel adds the
// clusters' partials to the residual in a fixed order, so the result is
// deterministic. Weights and the norm weight are requested before the grid
// dependency wait; the input x + attention partials are read after it.
#include "epilogue.cuh"
#include "ptx.cuh"

namespace lq8 {

constexpr int kMlpCl = 16;      // CTAs per cluster (non-portable size)
constexpr int kMlpProd = 16;    // SiLU products per CTA
constexpr int kMlpWarps = 8;    // consumer warps
constexpr int kMlpCT = kMlpWarps * 32;
constexpr int kMlpThreads = kMlpCT + 32;

struct MlpPlan {
    int gu, wd, wds, xs, red_in, red, floats;  // offsets in floats
};
__host__ __device__ inline int mlp_round(int n) { return (n + 31) / 32 * 32; }
__host__ __device__ inline int mlp_rows_per_owner(int h) { return (h / kMlpCl + 3) / 4 * 4; }
__host__ __device__ inline MlpPlan mlp_plan(int h) {
    MlpPlan p;
    const int nbx = h / 32, tiles_h = h / 32;
    int o = 0;
    auto take = [&](int n) { const int r = o; o += mlp_round(n); return r; };
    p.gu = take(nbx * 1088 / 4);        // the gate/up tile: codes then scales
    p.wd = take(tiles_h * 512 / 4);     // W_down: this CTA's 16-code chunk of each row tile
    p.wds = take(tiles_h * 64 / 4);     // and the scales of its block
    p.xs = take(h);                     // x * g
    p.red_in = take(kMlpCl * mlp_rows_per_owner(h));  // partials of the rows this CTA owns
    p.red = take(kMlpWarps * 33);
    p.floats = o;
    return p;
}

__global__ void __launch_bounds__(kMlpThreads, 1) decode_mlp_kernel(MlpArgs ma) {
    extern __shared__ __align__(128) float smf[];
    __shared__ __align__(8) uint64_t w_bar, red_bar;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) stamp_at(ma.stamp, 0);
    const int c = blockIdx.x;                 // a entries [16c, 16c + 16): W_down chunk c
    const int q = (int)cluster_rank();        // rank in the cluster
    const int cl_id = c / kMlpCl;
    const int h = ma.wgu.k, nbx = h >> 5, tiles_h = h >> 5;
    const int nbf = ma.wdown.k >> 5;
    const int rpo = mlp_rows_per_owner(h);
    const MlpPlan pl = mlp_plan(h);
    uint8_t* GU = reinterpret_cast<uint8_t*>(smf + pl.gu);
    uint8_t* WD = reinterpret_cast<uint8_t*>(smf + pl.wd);
    uint8_t* WDS = reinterpret_cast<uint8_t*>(smf + pl.wds);
    float* XS = smf + pl.xs;
    float* RIN = smf + pl.red_in;
    float* RED = smf + pl.red;
    const int own0 = q * rpo, own1 = min(h, own0 + rpo);  // rows this CTA reduces

    if (tid == 0) {
        mbar_init(&w_bar, 1);
        mbar_init(&red_bar, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&red_bar, (uint32_t)(kMlpCl * max(0, own1 - own0) * 4));
    }
    __syncthreads();
    cluster_sync();  // every CTA's barrier exists and expects its bytes before any peer stores

    if (warp == kMlpWarps) {
        if (lane == 0) {  // constant weights, before the dependency wait
            mbar_arrive_expect_tx(&w_bar, (uint32_t)(nbx * 1088 + tiles_h * (512 + 64)));
            bulk_g2s(GU, reinterpret_cast<const uint8_t*>(ma.wgu.qs) + (size_t)c * h * 32, (uint32_t)(nbx * 1024),
                     &w_bar);
            bulk_g2s(GU + nbx * 1024, reinterpret_cast<const uint8_t*>(ma.wgu.d) + (size_t)c * nbx * 64,
                     (uint32_t)(nbx * 64), &w_bar);
            for (int t = 0; t < tiles_h; ++t) {
                // 16-code chunk c of row tile t: block c / 2, its first or second half
                bulk_g2s(WD + (size_t)t * 512,
                         reinterpret_cast<const uint8_t*>(ma.wdown.qs) + (size_t)t * ma.wdown.k * 32 + (size_t)c * 512,
                         512u, &w_bar);
                bulk_g2s(WDS + (size_t)t * 64,
                         reinterpret_cast<const uint8_t*>(ma.wdown.d) + ((size_t)t * nbf + (c >> 1)) * 64, 64u, &w_bar);
            }
        }
        return;
    }

    // ---- consumers: x' = x + attention partials (in order), RMSNorm ---------------------
    constexpr int kGPre = 2;  // h <= 2048 floats: float4s per thread
    float4 gpre[kGPre];
#pragma unroll
    for (int u = 0; u < kGPre; ++u) {
        const int i = tid * 4 + u * kMlpCT * 4;
        gpre[u] = i < h ? *reinterpret_cast<const float4*>(ma.g + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    pdl_wait();
    if (tid == 0) {
        pdl_launch_dependents();
        stamp_at(ma.stamp, 1);
    }
    float ss = 0.0f;
    // x and every attention partial are requested before any is used: one round trip
    constexpr int kMaxParts = 8;
    float4 xin[kGPre], xp[kGPre][kMaxParts];
#pragma unroll
    for (int u = 0; u < kGPre; ++u) {
        const int i = tid * 4 + u * kMlpCT * 4;
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        xin[u] = i < h ? *reinterpret_cast<const float4*>(ma.x + i) : z;
#pragma unroll
        for (int p = 0; p < kMaxParts; ++p)
            xp[u][p] = (i < h && p < ma.n_attn_part)
                           ? *reinterpret_cast<const float4*>(ma.attn_part + (size_t)p * h + i)
                           : z;
    }
#pragma unroll
    for (int u = 0; u < kGPre; ++u) {
        const int i = tid * 4 + u * kMlpCT * 4;
        if (i < h) {
            float4 v = xin[u];
#pragma unroll
            for (int p = 0; p < kMaxParts; ++p) {
                if (p < ma.n_attn_part) {
                    const float4 w = xp[u][p];
                    v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
                }
            }
            if (c == 0) *reinterpret_cast<float4*>(ma.xr_out + i) = v;
            ss = fmaf(v.x, v.x, ss); ss = fmaf(v.y, v.y, ss); ss = fmaf(v.z, v.z, ss); ss = fmaf(v.w, v.w, ss);
            const float4 gg = gpre[u];
            *reinterpret_cast<float4*>(XS + i) = make_float4(v.x * gg.x, v.y * gg.y, v.z * gg.z, v.w * gg.w);
        }
    }
    ss = warp_sum(ss);
    if (lane == 0) RED[warp * 33 + 32] = ss;
    named_bar_sync(1, kMlpCT);
    float t_ss = 0.0f;
#pragma unroll
    for (int w = 0; w < kMlpWarps; ++w) t_ss += RED[w * 33 + 32];
    const float r_norm = 1.0f / sqrtf(t_ss / (float)h + ma.eps);
    mbar_wait_bounded(&w_bar, 0, ma.err, 51);

    // ---- gate/up: tile c, its blocks over the eight warps; lane = row ----------------------
    // Every warp sums the eight warp partials and forms the 16 SiLU products
    // itself (the same sums in the same order in every warp), so the down
    // projection needs no further barrier.
    float4 a4[4];
    {
        const float acc = tile_blocks_dot(GU, nbx, warp, kMlpWarps, nbx, lane, XS);
        RED[warp * 33 + lane] = acc;
        named_bar_sync(1, kMlpCT);
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kMlpWarps; ++w) v += RED[w * 33 + lane];
        v *= r_norm;
        const float up = __shfl_xor_sync(0xffffffffu, v, 1);
        const float prod = silu_f32(v) * up;  // valid in even lanes: entry lane / 2
        float e[kMlpProd];
#pragma unroll
        for (int i = 0; i < kMlpProd; ++i) e[i] = __shfl_sync(0xffffffffu, prod, 2 * i);
#pragma unroll
        for (int i = 0; i < 4; ++i) a4[i] = make_float4(e[4 * i], e[4 * i + 1], e[4 * i + 2], e[4 * i + 3]);
    }

    // ---- down: this CTA's 16 columns of W_down times a, every row tile; lane = row ---------
    // each row's partial goes straight to the cluster CTA owning the row:
    // RIN[source rank][r - owner's first row]
#pragma unroll 2
    for (int t = warp; t < tiles_h; t += kMlpWarps) {
        const uint4 q0 = *reinterpret_cast<const uint4*>(WD + (size_t)t * 512 + lane * 16);
        const float d = __half2float(reinterpret_cast<const __half*>(WDS + (size_t)t * 64)[lane]);
        uint64_t a0 = 0, a1 = 0;
        a0 = dot4_acc(q0.x, a4[0], a0); a1 = dot4_acc(q0.y, a4[1], a1);
        a0 = dot4_acc(q0.z, a4[2], a0); a1 = dot4_acc(q0.w, a4[3], a1);
        const float p = d * ((f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1)));
        const int r = t * 32 + lane, owner = r / rpo;
        st_async_f32(&RIN[q * rpo + (r - owner * rpo)], (uint32_t)owner, p, &red_bar);
    }
    mbar_wait_bounded(&red_bar, 0, ma.err, 52);  // the 8 partials of the rows this CTA owns
    for (int r = own0 + tid; r < own1; r += kMlpCT) {
        float v = 0.0f;
#pragma unroll
        for (int s = 0; s < kMlpCl; ++s) v += RIN[s * rpo + (r - own0)];
        ma.mlp_part[(size_t)cl_id * h + r] = v;
    }
}

static constexpr int kMlpSmemLimit = 227 * 1024 - 1024;
static bool g_mlp_attr = false;

static cudaLaunchConfig_t mlp_config(int grid, size_t smem, cudaStream_t s, cudaLaunchAttribute* attrs, bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kMlpThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = kMlpCl;
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

// The kernel serves the model when F / 16 is a multiple of 16 (whole
// clusters), h <= 2048 with h / 16 rows per owner a multiple of 4, the
// shared-memory plan fits, and all the clusters can be resident at once.
int decode_mlp_clusters(int h, int ff, int gu_rows) {
    if (h % 64 || ff % 32 || gu_rows != 2 * ff || h > 2048 || (h / kMlpCl) % 4) return 0;
    if ((ff / kMlpProd) % kMlpCl) return 0;
    const size_t smem = (size_t)mlp_plan(h).floats * 4;
    if (smem > (size_t)kMlpSmemLimit) return 0;
    if (!g_mlp_attr) {
        if (cudaFuncSetAttribute(decode_mlp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kMlpSmemLimit) !=
                cudaSuccess ||
            cudaFuncSetAttribute(decode_mlp_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_mlp_attr = true;
    }
    const int clusters = (ff / kMlpProd) / kMlpCl;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = mlp_config(kMlpCl, smem, 0, attrs, false);
    int resident = 0;
    if (cudaOccupancyMaxActiveClusters(&resident, decode_mlp_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return resident >= clusters ? clusters : 0;
}

cudaError_t launch_decode_mlp(const MlpArgs& ma, bool pdl, cudaStream_t s) {
    const int h = ma.wgu.k, ff = ma.wdown.k;
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = mlp_config(ff / kMlpProd, (size_t)mlp_plan(h).floats * 4, s, attrs, pdl);
    return cudaLaunchKernelEx(&cfg, decode_mlp_kernel, ma);
}

}  // namespace lq8
