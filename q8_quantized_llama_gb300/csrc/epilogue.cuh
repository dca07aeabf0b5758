// Per-element epilogues shared by the matrix-vector and matrix-matrix kernels.
// The neighbouring rows (2i, 2i+1) of the projection output are the rope_i
// pairs of a head, and the gate/up rows are interleaved the same way, so both
// fused epilogues work on a pair (even row value, odd row value).
#pragma once

#include "kernels.cuh"

namespace lq8 {

__device__ __forceinline__ float silu_f32(float z) { return z / (1.0f + expf(-z)); }

// Rotate the pair (a, b) = (value of row 2i, value of row 2i+1) by the angle
// of position pos and frequency index i: (a c - b s, a s + b c).
__device__ __forceinline__ void rope_pair(const EpiArgs& e, int pos, int i, float a, float b,
                                          float& ra, float& rb) {
    const int half = e.head_dim >> 1;
    const float c = e.rope_cos[(int64_t)pos * half + i];
    const float s = e.rope_sin[(int64_t)pos * half + i];
    ra = a * c - b * s;
    rb = a * s + b * c;
}

// The rotary (cos, sin) of row r's pair at position pos (q and k rows; v rows
// are not rotated and get (1, 0)).
__device__ __forceinline__ float2 rope_cs_for_row(const EpiArgs& e, int pos, int r) {
    if (r >= e.q_rows + e.kv_rows) return make_float2(1.0f, 0.0f);
    const int half = e.head_dim >> 1;
    const int i = (((r < e.q_rows) ? r : r - e.q_rows) % e.head_dim) >> 1;
    return make_float2(e.rope_cos[(int64_t)pos * half + i], e.rope_sin[(int64_t)pos * half + i]);
}

// QKV epilogue for the pair of rows (r, r+1), r even, of token t at position
// pos, with the pair's rotary (cos, sin) already loaded.
__device__ __forceinline__ void epi_qkv_pair_cs(const EpiArgs& e, int t, int pos, int r, float a, float b,
                                                float2 cs) {
    const int hd = e.head_dim;
    if (r < e.q_rows) {
        float* q = e.q_out + (int64_t)t * e.q_rows + r;
        q[0] = a * cs.x - b * cs.y;
        q[1] = a * cs.y + b * cs.x;
    } else if (r < e.q_rows + e.kv_rows) {
        const int rr = r - e.q_rows;
        const int kh = rr / hd, d = rr % hd;
        float* k = e.k_cache + ((int64_t)kh * e.max_seq + pos) * hd + d;
        k[0] = a * cs.x - b * cs.y;
        k[1] = a * cs.y + b * cs.x;
    } else if (r < e.q_rows + 2 * e.kv_rows) {
        const int rr = r - e.q_rows - e.kv_rows;
        const int kh = rr / hd, d = rr % hd;
        float* v = e.v_cache + ((int64_t)kh * e.max_seq + pos) * hd + d;
        v[0] = a;
        v[1] = b;
    }
}

// QKV epilogue for the pair of rows (r, r+1), r even, of token t at position pos.
__device__ __forceinline__ void epi_qkv_pair(const EpiArgs& e, int t, int pos, int r, float a, float b) {
    const int hd = e.head_dim;
    if (r < e.q_rows) {
        float ra, rb;
        rope_pair(e, pos, (r % hd) >> 1, a, b, ra, rb);
        float* q = e.q_out + (int64_t)t * e.q_rows + r;
        q[0] = ra;
        q[1] = rb;
    } else if (r < e.q_rows + e.kv_rows) {
        const int rr = r - e.q_rows;
        const int kh = rr / hd, d = rr % hd;
        float ra, rb;
        rope_pair(e, pos, d >> 1, a, b, ra, rb);
        float* k = e.k_cache + ((int64_t)kh * e.max_seq + pos) * hd + d;
        k[0] = ra;
        k[1] = rb;
    } else if (r < e.q_rows + 2 * e.kv_rows) {
        const int rr = r - e.q_rows - e.kv_rows;
        const int kh = rr / hd, d = rr % hd;
        float* v = e.v_cache + ((int64_t)kh * e.max_seq + pos) * hd + d;
        v[0] = a;
        v[1] = b;
    }
}

}  // namespace lq8
