// Shared pieces of the decode attention kernels: the 64-position stage
// geometry, the producer and consumer sides of one KV head's position share
// (two passes per window through a ring of shared-memory stages), the
// butterfly reduce-scatter of the K pass, and distributed-shared-memory
// stores. Included by attention.cu.
#pragma once

#include "kernels.cuh"
#include "ptx.cuh"

namespace lq8 {

constexpr int kMaxGroup = 8;  // query heads per KV head handled by the decode kernels

constexpr int kCaRows = 64;                // positions per stage
constexpr int kCaStages = 4;
constexpr int kCaWin = 256;                // positions per window
constexpr int kCaWarps = 8;                // consumer warps
constexpr int kCaCT = kCaWarps * 32;
constexpr int kCaThreads = kCaCT + 32;     // + producer warp
constexpr int kCaRowsPerWarp = kCaRows / kCaWarps;

template <int HD>
struct CaGeom {
    static constexpr int kSlot = kCaRows * HD;             // ring slot (floats)
    static constexpr int kRing = kCaStages * kSlot;
    static constexpr int kSlices = kCaCT / (HD / 4);       // position slices in the V pass
    static_assert(kSlices * kMaxGroup * HD <= kRing, "slice sums reuse the ring");
};
struct CaPlan {
    int s, q, corr, po, pm, pl, om, red2, wo, floats;
};
__host__ __device__ inline int ca_round(int n) { return (n + 31) / 32 * 32; }
// wo_bytes: the W_o slice one CTA holds when the kernel also applies the O
// projection (0 otherwise).
template <int HD>
__host__ __device__ inline CaPlan ca_plan(int G, int GP, int cl, int wo_bytes) {
    CaPlan p;
    int o = CaGeom<HD>::kRing;
    auto take = [&](int n) { const int r = o; o += ca_round(n); return r; };
    p.s = take(kCaWin * GP);        // [kCaWin][GP] scores, then weights
    p.q = take(GP * HD);            // [GP][HD]
    p.corr = take(kMaxGroup);
    p.po = take(cl * G * HD);       // [cl][G][HD]
    p.pm = take(cl * G);            // [cl][G]
    p.pl = take(cl * G);
    p.om = take(wo_bytes ? G * HD : 0);          // merged output of the group (O projection input)
    p.red2 = take(wo_bytes ? kCaWarps * 33 : 0);
    p.wo = take(wo_bytes / 4);                   // W_o tiles: per tile, codes then scales
    p.floats = o;
    return p;
}
inline int ca_group_pad(int G) { return G <= 4 ? 4 : 8; }

// The O projection applied inside the decode attention kernel: cluster kh
// multiplies its query heads' output o (G * head_dim values) by the matching
// column blocks of W_o and writes the partial product part[kh][0..rows); the
// n_kv partials sum to W_o o.
struct AttnOproj {
    PackedQ8 wo;
    float* part;
    int part_stride;
    unsigned long long* stamp;  // timeline stamps (instrumented decode graph), or null
};
constexpr int kFoMaxWoBytes = 32 * 1024;  // W_o bytes one CTA may hold
__host__ __device__ inline int fo_tiles_per_cta(int rows_pad, int cl) { return (rows_pad / 32 + cl - 1) / cl; }
__host__ __device__ inline int fo_wo_bytes(int rows_pad, int G, int hd, int cl) {
    return fo_tiles_per_cta(rows_pad, cl) * (G * hd / 32) * 1088;
}

__device__ __forceinline__ void st_dsmem_f32(float* local_ptr, uint32_t rank, float v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_ptr)), "r"(rank));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Butterfly reduce-scatter over groups of LPR lanes: on entry every lane
// holds NV partial values; on exit v[k] (k < NV / LPR) holds the sum over the
// group of value index (NV / LPR) * (lane % LPR) + k.
template <int NV, int LPR>
__device__ __forceinline__ void reduce_scatter(float (&v)[NV], int lane) {
    int n = NV;
#pragma unroll
    for (int o = LPR / 2; o >= 1; o >>= 1) {
        const int half = n >> 1;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < NV / 2; ++k) {
            if (k < half) {
                const float send = upper ? v[k] : v[k + half];
                const float keep = upper ? v[k + half] : v[k];
                v[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
            }
        }
        n = half;
    }
}

// Producer side of one KV head's share [ja, jb): per window, the K stages then
// the V stages, one bulk copy each, through the ring. Rows at or after j_new
// (written by the preceding kernel) are requested only after the grid
// dependency wait; with skip_new the row j_new is not requested at all (the
// consumers take it from shared memory). Run by one thread.
template <int HD, int STAGES = kCaStages, int SLOT = CaGeom<HD>::kSlot>
__device__ __forceinline__ void ca_produce_head(float* smf, uint64_t* full, uint64_t* empty, const float* kb,
                                                const float* vb, int ja, int jb, int j_new, bool skip_new,
                                                bool& waited, int& j, int* err) {
    for (int wa = ja; wa < jb; wa += kCaWin) {
        const int wn = min(kCaWin, jb - wa);
        for (int pass = 0; pass < 2; ++pass) {
            for (int r0 = 0; r0 < wn; r0 += kCaRows, ++j) {
                const int a = wa + r0;
                int n = min(kCaRows, wn - r0);
                const int slot = j % STAGES;
                if (skip_new && a + n > j_new) n = j_new - a;  // rows before the newest one
                else if (!waited && a + n > j_new) {
                    pdl_wait();
                    waited = true;
                }
                if (j >= STAGES) mbar_wait_bounded(&empty[slot], ((j / STAGES) - 1) & 1, err, 21);
                mbar_arrive_expect_tx(&full[slot], (uint32_t)(n * HD * 4));
                if (n > 0)
                    bulk_g2s(smf + slot * SLOT, (pass == 0 ? kb : vb) + (int64_t)a * HD,
                             (uint32_t)(n * HD * 4), &full[slot]);
            }
        }
    }
}

// Consumer side of one KV head's share [ja, jb) (all consumer threads): the
// K pass, softmax and V pass of every window. qr: this lane's q chunk of every
// head of the group; o, m_run, l_run: running state (m/l valid in warp g < G
// for head g). `first`: no earlier window used S in this kernel.
template <int HD, int GP, int STAGES = kCaStages, int SLOT = CaGeom<HD>::kSlot>
__device__ __forceinline__ void ca_consume_head(const float* smf, uint64_t* full, uint64_t* empty, float* S,
                                                float* CORR, const float4 (&qr)[GP], int G, int ja, int jb,
                                                float scale, int& j, bool& first, float4 (&o)[GP], float& m_run,
                                                float& l_run, int* err, int j_new = -1,
                                                const float* knew = nullptr, const float* vnew = nullptr) {
    using Geo = CaGeom<HD>;
    constexpr int D4 = HD / 4;
    constexpr int LPR = D4;                          // lanes per K row in the K pass
    constexpr int RPI = 32 / LPR;                    // rows per warp-wide load
    constexpr int RS = kCaRowsPerWarp / RPI;         // row slots per lane
    constexpr int NV = RS * GP;                      // partial scores per lane
    constexpr int R = NV / LPR;                      // finished scores per lane
    static_assert(R >= 1 && NV % LPR == 0, "K pass shape");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kc4 = lane % LPR, khalf = lane / LPR;   // K pass: chunk, row within a load
    const int d4 = tid % D4, slice = tid / D4;        // V pass

    for (int wa = ja; wa < jb; wa += kCaWin) {
        const int wn = min(kCaWin, jb - wa);
        if (!first) named_bar_sync(1, kCaCT);  // every thread is done with the previous weights in S
        first = false;
        // ---- K pass: scores of every head of the group --------------------------------
        for (int r0 = 0; r0 < wn; r0 += kCaRows, ++j) {
            const int slot = j % STAGES, n = min(kCaRows, wn - r0);
            mbar_wait_bounded(&full[slot], (j / STAGES) & 1, err, 22);
            const float* Ks = smf + slot * SLOT;
            float v[NV];
#pragma unroll
            for (int rs = 0; rs < RS; ++rs) {
                const int row = warp * kCaRowsPerWarp + rs * RPI + khalf;
                const float* kr = (knew && wa + r0 + row == j_new) ? knew : Ks + row * HD;
                const float4 kv = row < n ? *reinterpret_cast<const float4*>(kr + kc4 * 4)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int g = 0; g < GP; ++g) {
                    float a = qr[g].x * kv.x;
                    a = fmaf(qr[g].y, kv.y, a);
                    a = fmaf(qr[g].z, kv.z, a);
                    v[rs * GP + g] = fmaf(qr[g].w, kv.w, a);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            reduce_scatter<NV, LPR>(v, lane);
#pragma unroll
            for (int k = 0; k < R; ++k) {
                const int idx = R * kc4 + k, rs = idx / GP, g = idx % GP;
                const int row = warp * kCaRowsPerWarp + rs * RPI + khalf;
                if (row < n) S[(r0 + row) * GP + g] = v[k] * scale;
            }
        }
        named_bar_sync(1, kCaCT);
        // ---- softmax statistics over the window, weights in place ---------------------
        if (warp < G) {
            float mw = -INFINITY;
            for (int p = lane; p < wn; p += 32) mw = fmaxf(mw, S[p * GP + warp]);
            const float m_new = fmaxf(m_run, warp_max(mw));
            float sum = 0.0f;
            for (int p = lane; p < wn; p += 32) {
                const float e = expf(S[p * GP + warp] - m_new);
                S[p * GP + warp] = e;
                sum += e;
            }
            const float corr = expf(m_run - m_new);  // 0 on the first window
            l_run = l_run * corr + warp_sum(sum);
            m_run = m_new;
            if (lane == 0) CORR[warp] = corr;
        }
        named_bar_sync(1, kCaCT);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
            const float c = g < G ? CORR[g] : 0.0f;
            o[g].x *= c; o[g].y *= c; o[g].z *= c; o[g].w *= c;
        }
        // ---- V pass: weighted sum of the value rows -------------------------------------
        for (int r0 = 0; r0 < wn; r0 += kCaRows, ++j) {
            const int slot = j % STAGES, n = min(kCaRows, wn - r0);
            mbar_wait_bounded(&full[slot], (j / STAGES) & 1, err, 23);
            const float* Vs = smf + slot * SLOT;
            for (int jj = slice; jj < n; jj += Geo::kSlices) {
                const float* vr = (vnew && wa + r0 + jj == j_new) ? vnew : Vs + jj * HD;
                const float4 vv = *reinterpret_cast<const float4*>(vr + d4 * 4);
                const float* pw = S + (r0 + jj) * GP;
#pragma unroll
                for (int g4 = 0; g4 < GP; g4 += 4) {
                    const float4 p4 = *reinterpret_cast<const float4*>(pw + g4);
                    const float pp[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float4& acc = o[g4 + u];
                        acc.x = fmaf(pp[u], vv.x, acc.x); acc.y = fmaf(pp[u], vv.y, acc.y);
                        acc.z = fmaf(pp[u], vv.z, acc.z); acc.w = fmaf(pp[u], vv.w, acc.w);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
    }
}


}  // namespace lq8
