// One decode layer (T = 1) as ONE kernel: a single cluster of 16 CTAs does
// RMSNorm -> Q/K/V projection + rope_i + KV append -> GQA attention -> O
// projection + residual -> RMSNorm -> gate/up + SiLU -> down projection +
// residual ("量化 llama 的一次前向", forward: the same steps as the per-kernel
// path, in one launch per layer).
//
// Why: a decode step of a small model is a chain of short dependent steps;
// as separate kernels each link costs a grid launch and completion (~0.5-0.7
// us) plus a global-memory round trip. Inside a cluster the links are
// asynchronous stores into the other CTAs' shared memory (st.async) that
// complete transaction counts on the receivers' mbarriers (bounded waits),
// and the weights of the whole layer stream into each CTA's ring of
// shared-memory stages from launch on. With programmatic dependent launch the
// next layer's kernel starts on other SMs while this one runs, so its weight
// stream overlaps this layer's arithmetic.
//
// Work of CTA c (CL = 16):
//   Q/K/V, O, gate/up: 32-row tiles c, c + 16, ... of each projection;
//   down: units (tile, half of the inner dimension) c, c + 16, ...;
//   attention: KV head c / P, position share c % P of it (P = 16 / n_kv).
// Every CTA receives every exchanged vector (new q/k/v rows, attention
// partials, the residual after the O projection, the SiLU product); the down
// partials go to the CTA that owns the tile, which writes the next residual.
#include "attn_core.cuh"
#include "epilogue.cuh"

namespace lq8 {

constexpr int kLkCl = 16;          // CTAs (one cluster)
constexpr int kLkStages = 6;       // ring stages
constexpr int kLkUnitBlocks = 24;  // at most this many 32-weight blocks per weight unit

template <int HD>
struct LkGeom {
    static constexpr int kUnitFloats = kLkUnitBlocks * 272;  // 1088 bytes per block
    static constexpr int kSlot = kUnitFloats > kCaRows * HD ? kUnitFloats : kCaRows * HD;
    static constexpr int kRing = kLkStages * kSlot;
};

struct LkPlan {
    int s, q, corr, red, red2, x, xn, xo, qa, knew, vnew, po, pm, pl, wg, om, a, dp, ga, gf, floats;
};
__host__ __device__ inline int lk_units_per_row(int k) { return (k / 32 + kLkUnitBlocks - 1) / kLkUnitBlocks; }
__host__ __device__ inline int lk_tiles_of(int rows_pad, int c) { return (rows_pad / 32 - c + kLkCl - 1) / kLkCl; }

template <int HD>
__host__ __device__ inline LkPlan lk_plan(int h, int ff, int n_head, int n_kv, int GP) {
    LkPlan p;
    const int qd = n_head * HD, kvd = n_kv * HD, G = n_head / n_kv, P = kLkCl / n_kv;
    int o = LkGeom<HD>::kRing;
    auto take = [&](int n) { const int r = o; o += (n + 31) / 32 * 32; return r; };
    p.s = take(kCaWin * GP);
    p.q = take(GP * HD);
    p.corr = take(kMaxGroup);
    p.red = take(kCaWarps * GP * HD);
    p.red2 = take(kCaWarps * 33);
    p.x = take(h);
    p.xn = take(h);
    p.xo = take(h);
    p.qa = take(qd);
    p.knew = take(kvd);
    p.vnew = take(kvd);
    p.po = take(n_kv * P * G * HD);
    p.pm = take(n_kv * P * G);
    p.pl = take(n_kv * P * G);
    p.wg = take(n_head * P);
    p.om = take(qd);
    p.a = take(ff);
    p.dp = take(((h + 31) / 32 + kLkCl - 1) / kLkCl * lk_units_per_row(ff) * 32);
    p.ga = take(h);
    p.gf = take(h);
    p.floats = o;
    return p;
}

// 32 rows of one weight unit (blocks [b0, b0 + nbs) of a tile, staged at `tw`)
// against vec[b0 * 32 ...]: lane = row; returns the row sums in warp 0.
__device__ __forceinline__ float lk_unit_dot(const uint8_t* tw, int nbs, const float* vec, float* red2, int warp,
                                             int lane) {
    float acc = 0.0f;
    for (int b = warp; b < nbs; b += kCaWarps) {
        const uint4 q0 = *reinterpret_cast<const uint4*>(tw + b * 1024 + lane * 16);
        const uint4 q1 = *reinterpret_cast<const uint4*>(tw + b * 1024 + 512 + lane * 16);
        const float d = __half2float(reinterpret_cast<const __half*>(tw + nbs * 1024)[b * 32 + lane]);
        const float4* x4 = reinterpret_cast<const float4*>(vec + b * 32);
        uint64_t a0 = 0, a1 = 0;
        a0 = dot4_acc(q0.x, x4[0], a0); a1 = dot4_acc(q1.x, x4[4], a1);
        a0 = dot4_acc(q0.y, x4[1], a0); a1 = dot4_acc(q1.y, x4[5], a1);
        a0 = dot4_acc(q0.z, x4[2], a0); a1 = dot4_acc(q1.z, x4[6], a1);
        a0 = dot4_acc(q0.w, x4[3], a0); a1 = dot4_acc(q1.w, x4[7], a1);
        acc = fmaf(d, (f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1)), acc);
    }
    red2[warp * 33 + lane] = acc;
    named_bar_sync(1, kCaCT);
    float v = 0.0f;
    if (warp == 0) {
#pragma unroll
        for (int w = 0; w < kCaWarps; ++w) v += red2[w * 33 + lane];
    }
    return v;
}

template <int HD, int GP>
__global__ void __launch_bounds__(kCaThreads, 1) decode_layer_kernel(LayerKArgs la) {
    using Geo = LkGeom<HD>;
    constexpr int CL = kLkCl, D4 = HD / 4;
    extern __shared__ __align__(128) float smf[];
    __shared__ __align__(8) uint64_t full[kLkStages];
    __shared__ __align__(8) uint64_t empty[kLkStages];
    __shared__ __align__(8) uint64_t g_bar, rows_bar, part_bar, xo_bar, a_bar, dn_bar;
    __shared__ float s_rscale;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = (int)cluster_rank();
    const int h = la.wqkv.k, ff = la.wdown.k;
    const int n_head = la.n_head, n_kv = la.n_kv, G = n_head / n_kv, P = CL / n_kv;
    const int qd = n_head * HD, kvd = n_kv * HD;
    const int upr = lk_units_per_row(ff);  // down units per tile
    const LkPlan pl = lk_plan<HD>(h, ff, n_head, n_kv, GP);
    float* S = smf + pl.s;
    float* Q = smf + pl.q;
    float* CORR = smf + pl.corr;
    float* RED = smf + pl.red;
    float* RED2 = smf + pl.red2;
    float* X = smf + pl.x;
    float* XN = smf + pl.xn;
    float* XO = smf + pl.xo;
    float* QA = smf + pl.qa;
    float* KNEW = smf + pl.knew;
    float* VNEW = smf + pl.vnew;
    float* PO = smf + pl.po;
    float* PM = smf + pl.pm;
    float* PLs = smf + pl.pl;
    float* WG = smf + pl.wg;
    float* OM = smf + pl.om;
    float* A = smf + pl.a;
    float* DP = smf + pl.dp;
    float* GA = smf + pl.ga;
    float* GF = smf + pl.gf;

    const int pos = la.st->pos;  // written two or more launches back
    const int kv_len = pos + 1, j_new = pos;
    const bool attn_cta = c < n_kv * P;
    const int kh = c / P, chunk = c % P;
    const int per = (kv_len + P - 1) / P;
    const int ja = min(kv_len, chunk * per), jb = min(kv_len, ja + per);
    const int t_qkv = la.wqkv.rows_pad >> 5, t_o = la.wo.rows_pad >> 5, t_gu = la.wgu.rows_pad >> 5;
    const int t_dn = la.wdown.rows_pad >> 5;
    const int my_dn_tiles = lk_tiles_of(la.wdown.rows_pad, c);

    if (tid == 0) {
        for (int s = 0; s < kLkStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCaWarps);
        }
        mbar_init(&g_bar, 1);
        mbar_init(&rows_bar, 1);
        mbar_init(&part_bar, 1);
        mbar_init(&xo_bar, 1);
        mbar_init(&a_bar, 1);
        mbar_init(&dn_bar, 1);
        fence_mbar_init();
        // bytes each exchange brings into this CTA
        mbar_arrive_expect_tx(&rows_bar, (uint32_t)((qd + 2 * kvd) * 4));
        mbar_arrive_expect_tx(&part_bar, (uint32_t)(n_kv * P * (G * HD + 2 * G) * 4));
        mbar_arrive_expect_tx(&xo_bar, (uint32_t)(h * 4));
        mbar_arrive_expect_tx(&a_bar, (uint32_t)(ff * 4));
        mbar_arrive_expect_tx(&dn_bar, (uint32_t)(my_dn_tiles * upr * 32 * 4));
    }
    __syncthreads();
    cluster_sync();  // every CTA's barriers exist and expect their bytes before any peer stores

    if (warp == kCaWarps) {
        // ================= producer: the layer's weights, in consumption order =========
        if (lane == 0) {
            mbar_arrive_expect_tx(&g_bar, (uint32_t)(2 * h * 4));
            bulk_g2s(GA, la.g_attn, (uint32_t)(h * 4), &g_bar);
            bulk_g2s(GF, la.g_ffn, (uint32_t)(h * 4), &g_bar);
            int j = 0;
            auto unit = [&](const PackedQ8& W, int t, int b0, int nbs) {
                const int slot = j % kLkStages;
                if (j >= kLkStages) mbar_wait_bounded(&empty[slot], ((j / kLkStages) - 1) & 1, la.err, 31);
                uint8_t* dst = reinterpret_cast<uint8_t*>(smf + slot * Geo::kSlot);
                const int nb = W.k >> 5;
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(nbs * 1088));
                bulk_g2s(dst, reinterpret_cast<const uint8_t*>(W.qs) + (size_t)t * W.k * 32 + (size_t)b0 * 1024,
                         (uint32_t)(nbs * 1024), &full[slot]);
                bulk_g2s(dst + nbs * 1024, reinterpret_cast<const uint8_t*>(W.d) + ((size_t)t * nb + b0) * 64,
                         (uint32_t)(nbs * 64), &full[slot]);
                ++j;
            };
            for (int t = c; t < t_qkv; t += CL) unit(la.wqkv, t, 0, h >> 5);
            if (attn_cta) {
                bool waited = false;
                ca_produce_head<HD, kLkStages, Geo::kSlot>(smf, full, empty, la.kc + (int64_t)kh * la.stride * HD,
                                                           la.vc + (int64_t)kh * la.stride * HD, ja, jb, j_new,
                                                           true, waited, j, la.err);
            }
            for (int t = c; t < t_o; t += CL) unit(la.wo, t, 0, qd >> 5);
            for (int t = c; t < t_gu; t += CL) unit(la.wgu, t, 0, h >> 5);
            const int nbd = ff >> 5;
            for (int u = c; u < t_dn * upr; u += CL) {
                const int t = u / upr, part = u % upr;
                const int b0 = (part * nbd) / upr, b1 = ((part + 1) * nbd) / upr;
                unit(la.wdown, t, b0, b1 - b0);
            }
        }
        return;
    }

    // ===================== consumers ===============================================
    int j = 0;  // ring stage counter, mirrors the producer
    auto stage = [&]() -> const uint8_t* {
        const int slot = j % kLkStages;
        mbar_wait_bounded(&full[slot], (j / kLkStages) & 1, la.err, 32);
        return reinterpret_cast<const uint8_t*>(smf + slot * Geo::kSlot);
    };
    auto release = [&]() {  // every consumer warp is done with the current stage
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[j % kLkStages]);
        ++j;
    };
    auto rms_norm = [&](const float* src, const float* g, float* dst) {
        float ss = 0.0f;
        for (int i = tid; i < h; i += kCaCT) ss = fmaf(src[i], src[i], ss);
        ss = warp_sum(ss);
        if (lane == 0) RED2[warp * 33 + 32] = ss;
        named_bar_sync(1, kCaCT);
        if (tid == 0) {
            float t = 0.0f;
            for (int w = 0; w < kCaWarps; ++w) t += RED2[w * 33 + 32];
            s_rscale = 1.0f / sqrtf(t / (float)h + la.eps);
        }
        named_bar_sync(1, kCaCT);
        const float r = s_rscale;
        for (int i = tid; i < h; i += kCaCT) dst[i] = src[i] * r * g[i];
        named_bar_sync(1, kCaCT);
    };

    pdl_wait();
    if (tid == 0) pdl_launch_dependents();
    for (int i = tid; i < h; i += kCaCT) X[i] = la.x_in[i];
    mbar_wait_bounded(&g_bar, 0, la.err, 33);
    named_bar_sync(1, kCaCT);
    rms_norm(X, GA, XN);

    // ---- Q/K/V rows of this CTA's tiles: rope_i, KV append, rows to every CTA ----
    {
        const int half = HD >> 1;
        const float* cosr = la.rope_cos + (int64_t)pos * half;
        const float* sinr = la.rope_sin + (int64_t)pos * half;
        for (int t = c; t < t_qkv; t += CL) {
            const uint8_t* tw = stage();
            const float v = lk_unit_dot(tw, h >> 5, XN, RED2, warp, lane);
            release();
            if (warp == 0) {
                const float other = __shfl_xor_sync(0xffffffffu, v, 1);
                const int r = t * 32 + lane;
                if (r < qd + kvd) {
                    const int rr = r < qd ? r : r - qd;
                    const int d = rr % HD;
                    const float cs = cosr[d >> 1], sn = sinr[d >> 1];
                    const float rot = (lane & 1) ? other * sn + v * cs : v * cs - other * sn;
                    if (r < qd) {
#pragma unroll 4
                        for (int p = 0; p < CL; ++p) st_async_f32(&QA[r], (uint32_t)p, rot, &rows_bar);
                    } else {
                        la.kc[((int64_t)(rr / HD) * la.stride + pos) * HD + d] = rot;
#pragma unroll 4
                        for (int p = 0; p < CL; ++p) st_async_f32(&KNEW[rr], (uint32_t)p, rot, &rows_bar);
                    }
                } else if (r < qd + 2 * kvd) {
                    const int rr = r - qd - kvd;
                    la.vc[((int64_t)(rr / HD) * la.stride + pos) * HD + rr % HD] = v;
#pragma unroll 4
                    for (int p = 0; p < CL; ++p) st_async_f32(&VNEW[rr], (uint32_t)p, v, &rows_bar);
                }
            }
            named_bar_sync(1, kCaCT);  // RED2 is reused by the next unit
        }
    }
    mbar_wait_bounded(&rows_bar, 0, la.err, 34);  // q, k, v of the new position

    // ---- attention: KV head kh over this CTA's position share -------------------------
    if (attn_cta) {
        for (int i = tid; i < GP * HD; i += kCaCT) Q[i] = i < G * HD ? QA[kh * G * HD + i] : 0.0f;
        named_bar_sync(1, kCaCT);
        float4 qr[GP], o[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            qr[g] = *reinterpret_cast<const float4*>(Q + g * HD + (lane % D4) * 4);
            o[g] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float m_run = -INFINITY, l_run = 0.0f;
        bool first = true;
        ca_consume_head<HD, GP, kLkStages, Geo::kSlot>(smf, full, empty, S, CORR, qr, G, ja, jb, la.scale, j, first,
                                                       o, m_run, l_run, la.err, j_new, KNEW + kh * HD,
                                                       VNEW + kh * HD);
        const int d4 = tid % D4;
        if (D4 < 32) {  // head_dim 64: two position slices per warp
#pragma unroll
            for (int g = 0; g < GP; ++g) {
                o[g].x += __shfl_xor_sync(0xffffffffu, o[g].x, 16);
                o[g].y += __shfl_xor_sync(0xffffffffu, o[g].y, 16);
                o[g].z += __shfl_xor_sync(0xffffffffu, o[g].z, 16);
                o[g].w += __shfl_xor_sync(0xffffffffu, o[g].w, 16);
            }
        }
        named_bar_sync(1, kCaCT);
        if (lane < D4) {
#pragma unroll
            for (int g = 0; g < GP; ++g)
                if (g < G) *reinterpret_cast<float4*>(RED + (warp * GP + g) * HD + d4 * 4) = o[g];
        }
        named_bar_sync(1, kCaCT);
        for (int e4 = tid; e4 < G * HD / 4; e4 += kCaCT) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            const int g = (e4 * 4) / HD, d = (e4 * 4) % HD;
#pragma unroll
            for (int w = 0; w < kCaWarps; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(RED + (w * GP + g) * HD + d);
                acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
            }
#pragma unroll 4
            for (int p = 0; p < CL; ++p)
                st_async_f32x4(&PO[c * G * HD + e4 * 4], (uint32_t)p, acc, &part_bar);
        }
        if (warp < G && lane < CL) {
            st_async_f32(&PM[c * G + warp], (uint32_t)lane, m_run, &part_bar);
            st_async_f32(&PLs[c * G + warp], (uint32_t)lane, l_run, &part_bar);
        }
    }
    mbar_wait_bounded(&part_bar, 0, la.err, 35);  // every attention CTA's partial result

    // ---- merge: weights per (query head, source CTA), then the attention output --------
    for (int hq = warp; hq < n_head; hq += kCaWarps) {
        const int g = hq % G, kv = hq / G;
        const int src = kv * P + lane;  // source CTA of this head's share `lane`
        const float m_r = lane < P ? PM[src * G + g] : -INFINITY;
        const float M = warp_max(m_r);
        const float w = (lane < P && m_r != -INFINITY) ? expf(m_r - M) : 0.0f;
        const float L = warp_sum(lane < P ? w * PLs[src * G + g] : 0.0f);
        if (lane < P) WG[hq * P + lane] = w / L;
    }
    named_bar_sync(1, kCaCT);
    for (int e = tid; e < qd; e += kCaCT) {
        const int hq = e / HD, g = hq % G, kv = hq / G, d = e % HD;
        float acc = 0.0f;
        for (int p = 0; p < P; ++p) acc = fmaf(WG[hq * P + p], PO[(kv * P + p) * G * HD + g * HD + d], acc);
        OM[e] = acc;
    }
    named_bar_sync(1, kCaCT);

    // ---- O projection + residual: x' rows to every CTA -------------------------------
    for (int t = c; t < t_o; t += CL) {
        const uint8_t* tw = stage();
        const float v = lk_unit_dot(tw, qd >> 5, OM, RED2, warp, lane);
        release();
        if (warp == 0) {
            const int r = t * 32 + lane;
            if (r < h) {
                const float xr = X[r] + v;
#pragma unroll 4
                for (int p = 0; p < CL; ++p) st_async_f32(&XO[r], (uint32_t)p, xr, &xo_bar);
            }
        }
        named_bar_sync(1, kCaCT);
    }
    mbar_wait_bounded(&xo_bar, 0, la.err, 36);
    rms_norm(XO, GF, XN);

    // ---- gate/up + SiLU: the product to every CTA --------------------------------------
    // This CTA's tiles are taken a ring-full at a time, one whole tile per warp
    // (lane = row, no cross-warp reduction), so the tiles run side by side.
    {
        const int nbx = h >> 5;
        int t0 = c;
        while (t0 < t_gu) {
            int n = 0;  // tiles of this group
            while (n < kLkStages && n < kCaWarps && t0 + n * CL < t_gu) ++n;
            if (warp < n) {
                const int slot = (j + warp) % kLkStages;
                mbar_wait_bounded(&full[slot], ((j + warp) / kLkStages) & 1, la.err, 32);
                const uint8_t* tw = reinterpret_cast<const uint8_t*>(smf + slot * Geo::kSlot);
                uint64_t a0 = 0, a1 = 0;
                float acc = 0.0f;
                for (int b = 0; b < nbx; ++b) {
                    const uint4 q0 = *reinterpret_cast<const uint4*>(tw + b * 1024 + lane * 16);
                    const uint4 q1 = *reinterpret_cast<const uint4*>(tw + b * 1024 + 512 + lane * 16);
                    const float d = __half2float(reinterpret_cast<const __half*>(tw + nbx * 1024)[b * 32 + lane]);
                    const float4* x4 = reinterpret_cast<const float4*>(XN + b * 32);
                    a0 = 0; a1 = 0;
                    a0 = dot4_acc(q0.x, x4[0], a0); a1 = dot4_acc(q1.x, x4[4], a1);
                    a0 = dot4_acc(q0.y, x4[1], a0); a1 = dot4_acc(q1.y, x4[5], a1);
                    a0 = dot4_acc(q0.z, x4[2], a0); a1 = dot4_acc(q1.z, x4[6], a1);
                    a0 = dot4_acc(q0.w, x4[3], a0); a1 = dot4_acc(q1.w, x4[7], a1);
                    acc = fmaf(d, (f2_lo(a0) + f2_hi(a0)) + (f2_lo(a1) + f2_hi(a1)), acc);
                }
                const float up = __shfl_xor_sync(0xffffffffu, acc, 1);
                const int r = (t0 + warp * CL) * 32 + lane;
                if (!(lane & 1) && r < la.wgu.rows) {
                    const float av = silu_f32(acc) * up;
#pragma unroll 4
                    for (int p = 0; p < CL; ++p) st_async_f32(&A[r >> 1], (uint32_t)p, av, &a_bar);
                }
            }
            named_bar_sync(1, kCaCT);  // every tile of the group is read
            if (lane == 0)
                for (int u = 0; u < n; ++u) mbar_arrive(&empty[(j + u) % kLkStages]);
            j += n;
            t0 += n * CL;
        }
    }
    mbar_wait_bounded(&a_bar, 0, la.err, 37);

    // ---- down projection: partial rows to the tile's owner -----------------------------
    {
        const int nbd = ff >> 5;
        for (int u = c; u < t_dn * upr; u += CL) {
            const int t = u / upr, part = u % upr;
            const int b0 = (part * nbd) / upr, b1 = ((part + 1) * nbd) / upr;
            const uint8_t* tw = stage();
            const float v = lk_unit_dot(tw, b1 - b0, A + b0 * 32, RED2, warp, lane);
            release();
            if (warp == 0) {
                const int owner = t % CL, slot_t = t / CL;
                st_async_f32(&DP[(slot_t * upr + part) * 32 + lane], (uint32_t)owner, v, &dn_bar);
            }
            named_bar_sync(1, kCaCT);
        }
    }
    mbar_wait_bounded(&dn_bar, 0, la.err, 38);
    // ---- residual of the tiles this CTA owns --------------------------------------------
    for (int f = tid; f < my_dn_tiles * 32; f += kCaCT) {
        const int i = f >> 5, ln = f & 31;
        const int r = (c + i * CL) * 32 + ln;
        float v = XO[r < h ? r : 0];
        for (int p = 0; p < upr; ++p) v += DP[(i * upr + p) * 32 + ln];
        if (r < h) la.x_out[r] = v;
    }
}

// ---- host side -------------------------------------------------------------------------
static constexpr int kLkSmemLimit = 227 * 1024 - 1024;

template <int HD, int GP>
static cudaLaunchConfig_t lk_config(const LayerKArgs& la, size_t smem, cudaStream_t s, cudaLaunchAttribute* attrs,
                                    bool pdl) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kLkCl);
    cfg.blockDim = dim3(kCaThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = kLkCl;
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
    (void)la;
    return cfg;
}

template <int HD, int GP>
static size_t lk_smem(const LayerKArgs& la) {
    return (size_t)lk_plan<HD>(la.wqkv.k, la.wdown.k, la.n_head, la.n_kv, GP).floats * 4;
}

template <int HD, int GP>
static bool lk_supported_t(const LayerKArgs& la) {
    const size_t smem = lk_smem<HD, GP>(la);
    if (smem > (size_t)kLkSmemLimit) return false;
    if (cudaFuncSetAttribute(decode_layer_kernel<HD, GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(decode_layer_kernel<HD, GP>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = lk_config<HD, GP>(la, smem, 0, attrs, false);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_layer_kernel<HD, GP>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return n >= 2;  // this layer and the next one (started early) side by side
}

// The layer kernel serves the model when: head_dim 64 or 128; the group of
// query heads per KV head <= 8; n_kv divides into 16 CTAs; every projection's
// inner dimension gives units of <= 24 blocks except the down projection
// (split in halves or more); the shared-memory plan fits.
bool decode_layer_supported(const LayerKArgs& la, int head_dim) {
    const int n_head = la.n_head, n_kv = la.n_kv;
    if (n_kv <= 0 || n_head % n_kv || n_head / n_kv > kMaxGroup || n_kv > kLkCl) return false;
    const int G = n_head / n_kv;
    if (G * head_dim % 32 || la.wqkv.k % 32 || la.wdown.k % 32) return false;
    const int h = la.wqkv.k;
    if (h / 32 > kLkUnitBlocks || (n_head * head_dim) / 32 > kLkUnitBlocks) return false;  // one unit per tile
    if (la.wo.k != n_head * head_dim || la.wgu.k != h || la.wgu.rows != 2 * la.wdown.k || la.wo.rows != h ||
        la.wdown.rows != h)
        return false;
    const bool wide = G > 4;
    if (head_dim == 64) return wide ? lk_supported_t<64, 8>(la) : lk_supported_t<64, 4>(la);
    if (head_dim == 128) return wide ? lk_supported_t<128, 8>(la) : lk_supported_t<128, 4>(la);
    return false;
}

template <int HD, int GP>
static cudaError_t lk_launch(const LayerKArgs& la, bool pdl, cudaStream_t s) {
    cudaLaunchAttribute attrs[2];
    cudaLaunchConfig_t cfg = lk_config<HD, GP>(la, lk_smem<HD, GP>(la), s, attrs, pdl);
    return cudaLaunchKernelEx(&cfg, decode_layer_kernel<HD, GP>, la);
}

cudaError_t launch_decode_layer(const LayerKArgs& la, int head_dim, bool pdl, cudaStream_t s) {
    if (!la.st || la.x_in == la.x_out) return cudaErrorInvalidValue;
    const bool wide = la.n_head / la.n_kv > 4;
    if (head_dim == 64) return wide ? lk_launch<64, 8>(la, pdl, s) : lk_launch<64, 4>(la, pdl, s);
    if (head_dim == 128) return wide ? lk_launch<128, 8>(la, pdl, s) : lk_launch<128, 4>(la, pdl, s);
    return cudaErrorInvalidValue;
}

}  // namespace lq8
