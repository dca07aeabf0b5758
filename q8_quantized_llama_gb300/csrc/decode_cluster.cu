// The whole per-layer part of a decode step (T = 1) as ONE cluster of CTAs
// for models whose activations fit in shared memory: embedding, and for every
// layer RMSNorm -> Q/K/V projection + rope_i + KV append -> GQA attention ->
// O projection + residual -> RMSNorm -> gate/up + SiLU -> down projection +
// residual ("量化 llama 的一次前向", forward：mask 什么时候建 — the same steps
// as the per-kernel path). The lm_head + argmax runs after it on the whole GPU.
//
// Why: a decode step of a small model reads ~143 MB of weights (~21 us at HBM
// speed) but as ~150 dependent kernels it is bound by launch-to-launch latency
// (the pages make the same point about command submission on "生成一个
// token", 动脑筋答案). Here the dependent steps are cluster-wide barriers on
// mbarriers inside one kernel and the activations move through distributed
// shared memory: every CTA keeps a full copy of the residual stream, the
// projection outputs are broadcast to every CTA as they are produced.
//
// Work: each projection's 32-row tiles are dealt round-robin to the cluster's
// CTAs; a producer warp per CTA streams the CTA's tiles for the WHOLE step,
// layer after layer, into a ring of shared-memory stages with bulk async
// copies, never waiting on the barriers (weights are constant), so weight
// reads run ahead of the arithmetic. Attention: CTA r takes an equal share of
// the cached positions for all heads (K/V rows prefetched by cp.async at the
// start of the layer), and every CTA merges all CTAs' partial results.
#include "epilogue.cuh"
#include "ptx.cuh"

namespace lq8 {

constexpr int kCsWarps = 16;                      // consumer warps
constexpr int kCsCT = kCsWarps * 32;              // consumer threads
constexpr int kCsThreads = kCsCT + 32;            // + one producer warp
constexpr int kCsStageBlocks = 16;                // one block per consumer warp
constexpr int kCsStageBytes = kCsStageBlocks * 1024 + kCsStageBlocks * 64;
constexpr int kCsStages = 5;
constexpr int kCsSub = 16;                        // attention positions per sub-chunk

// Shared-memory plan (float offsets after the stage ring), the same on the
// host (sizing) and the device.
struct CsPlan {
    int x, xn, q, o, a, knew, vnew, katt, vatt, po, pm, pl, red, total_floats;
};
__host__ __device__ inline CsPlan cs_plan(int h, int n_head, int n_kv, int hd, int ff, int cl) {
    CsPlan p;
    const int qd = n_head * hd, kvd = n_kv * hd;
    int o = 0;
    auto take = [&](int n) { int r = o; o += (n + 31) / 32 * 32; return r; };
    p.x = take(h);
    p.xn = take(h);
    p.q = take(qd);
    p.o = take(qd);
    p.a = take(ff);
    p.knew = take(kvd);
    p.vnew = take(kvd);
    p.katt = take(2 * kCsSub * kvd);
    p.vatt = take(2 * kCsSub * kvd);
    p.po = take(cl * qd);
    p.pm = take(cl * n_head);
    p.pl = take(cl * n_head);
    p.red = take(2 * kCsWarps * 33);
    p.total_floats = o;
    return p;
}
__host__ __device__ inline size_t cs_smem_bytes(int h, int n_head, int n_kv, int hd, int ff, int cl) {
    return (size_t)kCsStages * kCsStageBytes + (size_t)cs_plan(h, n_head, n_kv, hd, ff, cl).total_floats * 4;
}

// ---- cluster helpers ------------------------------------------------------------
__device__ __forceinline__ uint32_t dsmem_addr(const void* local_ptr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local_ptr)), "r"(rank));
    return remote;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
template <int CL>
__device__ __forceinline__ void broadcast_f32(float* local_ptr, float v) {
#pragma unroll
    for (int r = 0; r < CL; ++r) st_cluster_f32(dsmem_addr(local_ptr, (uint32_t)r), v);
}
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* local_bar, uint32_t rank) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(dsmem_addr(local_bar, rank))
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ void fence_acq_rel_cluster() { asm volatile("fence.acq_rel.cluster;" ::: "memory"); }

__device__ __forceinline__ void cp_async16_cs(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit_cs() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait0_cs() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1_cs() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ float dot32_f2(const uint4& q0, const uint4& q1, const float* xs) {
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

enum CsPhase { CS_QKV = 0, CS_O = 1, CS_GU = 2, CS_DOWN = 3 };

template <int CL>
__global__ void __launch_bounds__(kCsThreads, 1) decode_cluster_kernel(ClusterStepArgs a) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t* ring = smem;
    float* F = reinterpret_cast<float*>(smem + kCsStages * kCsStageBytes);
    __shared__ __align__(8) uint64_t full[kCsStages];
    __shared__ __align__(8) uint64_t empty[kCsStages];
    __shared__ __align__(8) uint64_t phase_bar;
    __shared__ float s_r;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = (int)cluster_rank();
    const int h = a.h, hd = a.hd, n_head = a.n_head, n_kv = a.n_kv, G = n_head / n_kv;
    const int qd = n_head * hd, kvd = n_kv * hd;
    const CsPlan P = cs_plan(h, n_head, n_kv, hd, a.ff, CL);
    float* x = F + P.x;
    float* xn = F + P.xn;
    float* qv = F + P.q;
    float* ov = F + P.o;
    float* av = F + P.a;
    float* knew = F + P.knew;
    float* vnew = F + P.vnew;
    float* katt = F + P.katt;
    float* vatt = F + P.vatt;
    float* PO = F + P.po;
    float* PM = F + P.pm;
    float* PL = F + P.pl;
    float* red = F + P.red;

    if (tid == 0) {
        for (int s = 0; s < kCsStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCsWarps);
        }
        mbar_init(&phase_bar, CL);
        fence_mbar_init();
    }
    cluster_sync();  // every CTA's barriers exist before any remote arrive

    pdl_wait();
    // Let the lm_head kernel that follows start streaming its weights now; it
    // waits for this grid's completion before reading the final x.
    if (threadIdx.x == 0) pdl_launch_dependents();
    const int pos = a.st->pos;
    const int token = a.st->token;

    // The sequence of weight units (tile of one projection x all its blocks)
    // this CTA processes, in the order both the producer and the consumers walk.
    auto mat_of = [&](const LayerPtrs& L, int ph) -> const PackedQ8& {
        return ph == CS_QKV ? L.qkv : ph == CS_O ? L.o : ph == CS_GU ? L.gu : L.down;
    };

    if (warp == kCsWarps) {
        // ================= producer ======================================
        if (lane == 0) {
            int j = 0;
            for (int l = 0; l < a.n_layer; ++l) {
                const LayerPtrs& L = a.layers[l];
                for (int ph = 0; ph < 4; ++ph) {
                    const PackedQ8& W = mat_of(L, ph);
                    const int tiles = W.rows_pad >> 5, nb = W.k >> 5;
                    for (int t = c; t < tiles; t += CL) {
                        const uint8_t* gcodes = reinterpret_cast<const uint8_t*>(W.qs) + (size_t)t * W.k * 32;
                        const uint8_t* gscales = reinterpret_cast<const uint8_t*>(W.d) + (size_t)t * nb * 64;
                        for (int b = 0; b < nb; b += kCsStageBlocks, ++j) {
                            const int slot = j % kCsStages;
                            if (j >= kCsStages) mbar_wait_bounded(&empty[slot], ((j / kCsStages) - 1) & 1, a.err, 15);
                            const int nbs = min(kCsStageBlocks, nb - b);
                            uint8_t* dst = ring + slot * kCsStageBytes;
                            mbar_arrive_expect_tx(&full[slot], (uint32_t)(nbs * 1024 + nbs * 64));
                            bulk_g2s(dst, gcodes + (size_t)b * 1024, nbs * 1024, &full[slot]);
                            bulk_g2s(dst + kCsStageBlocks * 1024, gscales + (size_t)b * 64, nbs * 64, &full[slot]);
                        }
                    }
                }
            }
        }
        __syncwarp();
        cluster_sync();  // final: keep this CTA's shared memory alive for its peers
        return;
    }

    // ===================== consumers ===========================================
    int j = 0;        // stage counter (mirrors the producer)
    int red_par = 0;  // which half of `red` the next unit uses
    uint32_t phase_parity = 0;

    // Cluster-wide phase barrier: every consumer thread orders its shared and
    // global writes, one thread per CTA arrives on every CTA's barrier, and all
    // consumer threads wait on their own CTA's barrier.
    auto phase_sync = [&]() {
        fence_acq_rel_cluster();
        named_bar_sync(1, kCsCT);
        if (tid < CL) mbar_arrive_remote(&phase_bar, (uint32_t)tid);
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait_cluster(&phase_bar, phase_parity)) {
            if (global_timer_ns() - t0 > 1000000000ull) {
                if (a.err) atomicExch(a.err, 16);
                break;
            }
        }
        phase_parity ^= 1u;
    };

    // RMSNorm of the residual stream into xn (every CTA, identical result).
    auto rms_norm_into_xn = [&](const float* g) {
        float ss = 0.0f;
        for (int i = tid; i < h; i += kCsCT) ss = fmaf(x[i], x[i], ss);
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        named_bar_sync(1, kCsCT);
        if (tid == 0) {
            float t = 0.0f;
            for (int w = 0; w < kCsWarps; ++w) t += red[w];
            s_r = 1.0f / sqrtf(t / (float)h + a.eps);
        }
        named_bar_sync(1, kCsCT);
        const float r = s_r;
        for (int i = tid; i < h; i += kCsCT) xn[i] = x[i] * r * g[i];
        named_bar_sync(1, kCsCT);
    };

    // One weight unit: 32 rows of W against vector `vec`; returns (in warp 0)
    // the 32 dot products, lane = row within the tile.
    auto unit_dot = [&](const PackedQ8& W, const float* vec) -> float {
        const int nb = W.k >> 5;
        float acc = 0.0f;
        for (int b = 0; b < nb; b += kCsStageBlocks, ++j) {
            const int slot = j % kCsStages;
            mbar_wait_bounded(&full[slot], (j / kCsStages) & 1, a.err, 17);
            const int nbs = min(kCsStageBlocks, nb - b);
            if (warp < nbs) {
                const uint8_t* st = ring + slot * kCsStageBytes;
                const uint4 q0 = *reinterpret_cast<const uint4*>(st + warp * 1024 + lane * 16);
                const uint4 q1 = *reinterpret_cast<const uint4*>(st + warp * 1024 + 512 + lane * 16);
                const float d =
                    __half2float(reinterpret_cast<const __half*>(st + kCsStageBlocks * 1024)[warp * 32 + lane]);
                acc = fmaf(d, dot32_f2(q0, q1, vec + (b + warp) * 32), acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }
        float* rd = red + red_par * (kCsWarps * 33);
        rd[warp * 33 + lane] = acc;
        named_bar_sync(1, kCsCT);
        red_par ^= 1;
        float v = 0.0f;
        if (warp == 0) {
#pragma unroll
            for (int w = 0; w < kCsWarps; ++w) v += rd[w * 33 + lane];
        }
        return v;
    };

    // ---- embedding: x = dequant(E[token]) in every CTA ----------------------
    {
        int id = token;
        if (id < 0 || id >= a.n_vocab) {
            if (tid == 0 && a.err) atomicExch(a.err, 4);
            id = 0;
        }
        const int64_t tile = id >> 5, ln = id & 31;
        const int8_t* qrow = a.embd.qs + tile * (int64_t)h * 32 + ln * 16;
        const __half* drow = a.embd.d + tile * (int64_t)(h >> 5) * 32 + ln;
        for (int i = tid; i < h; i += kCsCT) {
            const int chunk = i >> 4;
            x[i] = __half2float(drow[(chunk >> 1) * 32]) * (float)qrow[(int64_t)chunk * 512 + (i & 15)];
        }
        named_bar_sync(1, kCsCT);
    }

    const int kv_len = pos + 1;
    const int per = (kv_len + CL - 1) / CL;
    const int r0 = min(kv_len, c * per), r1 = min(kv_len, r0 + per);
    const int n_rows = r1 - r0;
    const int n_sub = (n_rows + kCsSub - 1) / kCsSub;
    const int half = hd >> 1;
    const float* cosr = a.rope_cos + (int64_t)pos * half;
    const float* sinr = a.rope_sin + (int64_t)pos * half;

    // cp.async of cached K/V rows [ra, rb) (positions < kv_len - 1) into buffer b
    auto copy_kv = [&](const LayerPtrs& L, int buf, int ra, int rb) {
        const int n = rb - ra, c4 = hd / 4;
        for (int f = tid; f < n_kv * n * c4; f += kCsCT) {
            const int kh = f / (n * c4), rem = f % (n * c4), row = rem / c4, cc = rem % c4;
            const int64_t goff = ((int64_t)kh * a.max_seq + ra + row) * hd + cc * 4;
            const int soff = ((buf * n_kv + kh) * kCsSub + (ra - r0) % kCsSub + row) * hd + cc * 4;
            cp_async16_cs(katt + soff, L.kc + goff);
            cp_async16_cs(vatt + soff, L.vc + goff);
        }
    };
    auto sub_range = [&](int s, int& ra, int& rb) {
        ra = r0 + s * kCsSub;
        rb = min(r1, ra + kCsSub);
    };

    for (int l = 0; l < a.n_layer; ++l) {
        const LayerPtrs& L = a.layers[l];
        // prefetch this CTA's first K/V sub-chunk (rows cached before this step)
        if (n_sub > 0) {
            int ra, rb;
            sub_range(0, ra, rb);
            copy_kv(L, 0, ra, min(rb, kv_len - 1));
        }
        cp_async_commit_cs();

        // ---- Q/K/V + rope_i + KV append ------------------------------------
        rms_norm_into_xn(L.attn_norm);
        {
            const PackedQ8& W = L.qkv;
            for (int t = c; t < (W.rows_pad >> 5); t += CL) {
                const float v = unit_dot(W, xn);
                if (warp == 0) {
                    const int r = t * 32 + lane;
                    const float other = __shfl_xor_sync(0xffffffffu, v, 1);
                    if (r < qd + kvd) {
                        const int rr = r < qd ? r : r - qd;
                        const int i = (rr % hd) >> 1;
                        const float cs = cosr[i], sn = sinr[i];
                        const float rot = (lane & 1) ? other * sn + v * cs : v * cs - other * sn;
                        if (r < qd) {
                            broadcast_f32<CL>(&qv[r], rot);
                        } else {
                            const int kh = rr / hd, d = rr % hd;
                            L.kc[((int64_t)kh * a.max_seq + pos) * hd + d] = rot;
                            broadcast_f32<CL>(&knew[rr], rot);
                        }
                    } else if (r < qd + 2 * kvd) {
                        const int rr = r - qd - kvd;
                        const int kh = rr / hd, d = rr % hd;
                        L.vc[((int64_t)kh * a.max_seq + pos) * hd + d] = v;
                        broadcast_f32<CL>(&vnew[rr], v);
                    }
                }
            }
        }
        phase_sync();

        // ---- attention over this CTA's share of positions --------------------
        {
            int ra1 = 0, rb1 = 0;
            if (n_sub > 1) {
                sub_range(1, ra1, rb1);
                copy_kv(L, 1, ra1, min(rb1, kv_len - 1));
            }
            cp_async_commit_cs();
            float m = -INFINITY, lsum = 0.0f;
            float oacc[4] = {0.f, 0.f, 0.f, 0.f};  // hd / 32 values per lane (hd <= 128)
            const int hq = warp;                    // one query head per warp
            for (int s = 0; s < n_sub; ++s) {
                const int buf = s & 1;
                int ra, rb;
                sub_range(s, ra, rb);
                const int n = rb - ra;
                cp_async_wait1_cs();
                // the newest row comes from the broadcast copy of this step's k, v
                if (rb == kv_len) {
                    const int row = (kv_len - 1 - r0) % kCsSub;
                    for (int f = tid; f < kvd; f += kCsCT) {
                        const int kh = f / hd, d = f % hd;
                        katt[((buf * n_kv + kh) * kCsSub + row) * hd + d] = knew[f];
                        vatt[((buf * n_kv + kh) * kCsSub + row) * hd + d] = vnew[f];
                    }
                }
                named_bar_sync(1, kCsCT);
                if (hq < n_head) {
                    const int kh = hq / G;
                    const float* kbase = katt + ((buf * n_kv + kh) * kCsSub) * hd;
                    const float* vbase = vatt + ((buf * n_kv + kh) * kCsSub) * hd;
                    const float* qh = qv + hq * hd;
                    float sc = -INFINITY;
                    if (lane < n) {
                        const float* kr = kbase + lane * hd;
                        float acc0 = 0.0f, acc1 = 0.0f;
                        const int nc = hd / 4;
                        for (int cc = 0; cc < nc; cc += 2) {
                            const int c0 = (cc + lane) % nc, c1 = (cc + 1 + lane) % nc;
                            const float4 k0 = *reinterpret_cast<const float4*>(kr + c0 * 4);
                            const float4 q0 = *reinterpret_cast<const float4*>(qh + c0 * 4);
                            const float4 k1 = *reinterpret_cast<const float4*>(kr + c1 * 4);
                            const float4 q1 = *reinterpret_cast<const float4*>(qh + c1 * 4);
                            acc0 = fmaf(q0.x, k0.x, acc0); acc0 = fmaf(q0.y, k0.y, acc0);
                            acc0 = fmaf(q0.z, k0.z, acc0); acc0 = fmaf(q0.w, k0.w, acc0);
                            acc1 = fmaf(q1.x, k1.x, acc1); acc1 = fmaf(q1.y, k1.y, acc1);
                            acc1 = fmaf(q1.z, k1.z, acc1); acc1 = fmaf(q1.w, k1.w, acc1);
                        }
                        sc = (acc0 + acc1) * a.scale;
                    }
                    const float m_new = fmaxf(m, warp_max(sc));
                    const float p = lane < n ? expf(sc - m_new) : 0.0f;
                    const float corr = expf(m - m_new);  // 0 on the first sub-chunk
                    lsum = lsum * corr + warp_sum(p);
                    m = m_new;
                    const int nd = hd / 32;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (e < nd) oacc[e] *= corr;
                    for (int jj = 0; jj < n; ++jj) {
                        const float pj = __shfl_sync(0xffffffffu, p, jj);
                        const float* vr = vbase + jj * hd;
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (e < nd) oacc[e] = fmaf(pj, vr[lane + 32 * e], oacc[e]);
                    }
                }
                named_bar_sync(1, kCsCT);  // buffer `buf` is free again
                if (s + 2 < n_sub) {
                    int ra2, rb2;
                    sub_range(s + 2, ra2, rb2);
                    copy_kv(L, buf, ra2, min(rb2, kv_len - 1));
                }
                cp_async_commit_cs();
            }
            // push this CTA's partial result for every head to every CTA
            if (hq < n_head) {
                const int nd = hd / 32;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (e < nd) broadcast_f32<CL>(&PO[c * qd + hq * hd + lane + 32 * e], oacc[e]);
                if (lane == 0) {
                    broadcast_f32<CL>(&PM[c * n_head + hq], m);
                    broadcast_f32<CL>(&PL[c * n_head + hq], lsum);
                }
            }
        }
        phase_sync();
        // merge the cluster's partial results (every CTA, all heads)
        for (int e = tid; e < qd; e += kCsCT) {
            const int hh = e / hd;
            float M = -INFINITY;
#pragma unroll
            for (int r = 0; r < CL; ++r) M = fmaxf(M, PM[r * n_head + hh]);
            float Ls = 0.0f, acc = 0.0f;
#pragma unroll
            for (int r = 0; r < CL; ++r) {
                const float mr = PM[r * n_head + hh];
                const float w = mr == -INFINITY ? 0.0f : expf(mr - M);
                Ls = fmaf(w, PL[r * n_head + hh], Ls);
                acc = fmaf(w, PO[r * qd + e], acc);
            }
            ov[e] = acc / Ls;
        }
        named_bar_sync(1, kCsCT);

        // ---- O projection + residual -------------------------------------------
        {
            const PackedQ8& W = L.o;
            for (int t = c; t < (W.rows_pad >> 5); t += CL) {
                const float v = unit_dot(W, ov);
                if (warp == 0) {
                    const int r = t * 32 + lane;
                    if (r < h) broadcast_f32<CL>(&x[r], x[r] + v);
                }
            }
        }
        phase_sync();

        // ---- RMSNorm + gate/up + SiLU ------------------------------------------
        rms_norm_into_xn(L.ffn_norm);
        {
            const PackedQ8& W = L.gu;
            for (int t = c; t < (W.rows_pad >> 5); t += CL) {
                const float v = unit_dot(W, xn);
                if (warp == 0) {
                    const int r = t * 32 + lane;
                    const float up = __shfl_xor_sync(0xffffffffu, v, 1);
                    if (!(lane & 1) && r < W.rows) broadcast_f32<CL>(&av[r >> 1], silu_f32(v) * up);
                }
            }
        }
        phase_sync();

        // ---- down projection + residual ----------------------------------------
        {
            const PackedQ8& W = L.down;
            for (int t = c; t < (W.rows_pad >> 5); t += CL) {
                const float v = unit_dot(W, av);
                if (warp == 0) {
                    const int r = t * 32 + lane;
                    if (r < h) broadcast_f32<CL>(&x[r], x[r] + v);
                }
            }
        }
        phase_sync();
    }
    cp_async_wait0_cs();
    if (c == 0) {
        for (int i = tid; i < h; i += kCsCT) a.x_out[i] = x[i];
    }
    cluster_sync();  // no CTA leaves while its peers may still write into it
}

// ---- host side -------------------------------------------------------------------
template <int CL>
static cudaError_t cs_set_attrs(size_t smem) {
    cudaError_t err = cudaFuncSetAttribute(decode_cluster_kernel<CL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err == cudaSuccess && CL > 8)
        err = cudaFuncSetAttribute(decode_cluster_kernel<CL>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return err;
}

template <int CL>
static cudaLaunchConfig_t cs_config(size_t smem, cudaStream_t s, cudaLaunchAttribute* attrs) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CL);
    cfg.blockDim = dim3(kCsThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = CL;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    cfg.attrs = attrs;
    cfg.numAttrs = 1;
    return cfg;
}

// Largest usable cluster (16, then 8) for this model on the current device,
// or 0 when the activations do not fit or no such cluster can be scheduled.
int decode_cluster_size(int h, int n_head, int n_kv, int hd, int ff) {
    if (hd > 128 || n_head > kCsWarps || (hd % 32) != 0) return 0;
    int dev = 0, max_smem = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const size_t static_bytes = 2048;
    for (int cl : {16, 8}) {
        const size_t smem = cs_smem_bytes(h, n_head, n_kv, hd, ff, cl);
        if (smem + static_bytes > (size_t)max_smem) continue;
        cudaError_t err = cl == 16 ? cs_set_attrs<16>(smem) : cs_set_attrs<8>(smem);
        if (err != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        cudaLaunchAttribute attrs[1];
        cudaLaunchConfig_t cfg = cl == 16 ? cs_config<16>(smem, 0, attrs) : cs_config<8>(smem, 0, attrs);
        int n_clusters = 0;
        err = cl == 16 ? cudaOccupancyMaxActiveClusters(&n_clusters, decode_cluster_kernel<16>, &cfg)
                       : cudaOccupancyMaxActiveClusters(&n_clusters, decode_cluster_kernel<8>, &cfg);
        if (err != cudaSuccess) {
            cudaGetLastError();
            continue;
        }
        if (n_clusters >= 1) return cl;
    }
    return 0;
}

cudaError_t launch_decode_cluster(int cl, const ClusterStepArgs& args, cudaStream_t s) {
    const size_t smem = cs_smem_bytes(args.h, args.n_head, args.n_kv, args.hd, args.ff, cl);
    cudaLaunchAttribute attrs[1];
    if (cl == 16) {
        cudaLaunchConfig_t cfg = cs_config<16>(smem, s, attrs);
        return cudaLaunchKernelEx(&cfg, decode_cluster_kernel<16>, args);
    }
    if (cl == 8) {
        cudaLaunchConfig_t cfg = cs_config<8>(smem, s, attrs);
        return cudaLaunchKernelEx(&cfg, decode_cluster_kernel<8>, args);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lq8
