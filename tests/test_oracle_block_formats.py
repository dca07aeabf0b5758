"""Pins of the oracle's Q5_0, Q4_K and Q6_K dequantisation (reading R13).

- Byte sizes: with 22 bytes per 32 weights (Q5_0), 144 per 256 (Q4_K), 210
  per 256 (Q6_K) and 34 per 32 (Q8_0), the 135M Q4_K_M file's tensors — the
  30 ffn_down matrices (rows of 1536, a multiple of the K-quant block) split
  16 Q4_K / 14 Q6_K, 14 attn_k / attn_v in Q8_0 with token_embd, every other
  projection (rows of 576) in Q5_0 — give exactly the census on "速度"
  (CPU GGUF：decode 快，prefill 慢): 272 tensors; Q4K 16 / 7.6 MiB, Q5_0 166 /
  51.2 MiB, Q6K 14 / 9.7 MiB, Q8_0 15 / 30.3 MiB, F32 61 / 0.1 MiB.
- Layouts: each block is built here by a packer written independently from
  the block definition (the inverse direction of the oracle's unpacking), from
  per-weight codes chosen so that a swapped nibble, a wrong bit index, a wrong
  offset, a sign or endianness error gives different values; the expected
  weights are the closed forms of those codes.
"""
import numpy as np
import pytest

from oracle import q8_oracle as O

MIB = 2 ** 20


def test_block_sizes_reproduce_the_q4_k_m_census():
    h, ff, hd, nh, nkv, L, V = 576, 1536, 64, 9, 3, 30, 49152
    shapes = {"attn_q": (nh * hd, h), "attn_k": (nkv * hd, h), "attn_v": (nkv * hd, h),
              "attn_output": (h, nh * hd), "ffn_gate": (ff, h), "ffn_up": (ff, h), "ffn_down": (h, ff)}
    census = {}

    def add(kind, rows, k):
        n, b = census.get(kind, (0, 0))
        nbytes = rows * k * 4 if kind == "F32" else rows * O.block_format_row_bytes(kind, k)
        census[kind] = (n + 1, b + nbytes)

    add(O.GGUF_TYPE_Q8_0, V, h)                               # token_embd
    add("F32", 1, h)                                          # output_norm
    kv_q8 = 14
    for layer in range(L):
        add("F32", 1, h)
        add("F32", 1, h)
        for name, (rows, k) in shapes.items():
            if name == "ffn_down":
                add(O.GGUF_TYPE_Q4_K if layer < 16 else O.GGUF_TYPE_Q6_K, rows, k)
            elif name in ("attn_k", "attn_v") and kv_q8 > 0:
                kv_q8 -= 1
                add(O.GGUF_TYPE_Q8_0, rows, k)
            else:
                assert k % 256 != 0                           # 576: no K-quant block fits
                add(O.GGUF_TYPE_Q5_0, rows, k)
    got = {k: (n, round(b / MIB, 1)) for k, (n, b) in census.items()}
    assert got == {O.GGUF_TYPE_Q4_K: (16, 7.6), O.GGUF_TYPE_Q5_0: (166, 51.2), O.GGUF_TYPE_Q6_K: (14, 9.7),
                   O.GGUF_TYPE_Q8_0: (15, 30.3), "F32": (61, 0.1)}
    assert sum(n for n, _ in census.values()) == 272
    with pytest.raises(ValueError):
        O.block_format_row_bytes(O.GGUF_TYPE_Q4_K, 576)


def _fp16(x):
    return np.array([x], "<f2").view(np.uint8)


# ---- Q5_0 -------------------------------------------------------------------

def pack_q5_0(d, codes):
    """codes: 32 ints in [0, 32) -> 22 bytes."""
    out = np.zeros(22, np.uint8)
    out[0:2] = _fp16(d)
    qh = 0
    for j, c in enumerate(codes):
        qh |= ((c >> 4) & 1) << j
        if j < 16:
            out[6 + j] |= c & 15
        else:
            out[6 + j - 16] |= (c & 15) << 4
    out[2:6] = np.frombuffer(int(qh).to_bytes(4, "little"), np.uint8)
    return out


@pytest.mark.parametrize("d,codes", [
    (1.0, [j for j in range(16)] + [15 - j for j in range(16)]),        # nibble order, interleave j / j + 16
    (2.0, [16 if j in (5, 20) else 0 for j in range(32)]),             # fifth bit of weights 5 and 20 only
    (0.333251953125, [(7 * j + 3) % 32 for j in range(32)]),           # every code, a non-trivial fp16 d
])
def test_q5_0_block_layout(d, codes):
    blob = pack_q5_0(d, codes)[None, :]
    w = O.dequantize_q5_0(blob, 1, 32)[0]
    np.testing.assert_array_equal(w, [d * (c - 16) for c in codes])


def test_q5_0_rows_and_blocks_in_order():
    a = pack_q5_0(1.0, [17] * 32)       # all +1
    b = pack_q5_0(0.5, [0] * 32)        # all -8
    blob = np.stack([np.concatenate([a, b]), np.concatenate([b, a])])
    w = O.dequantize_q5_0(blob, 2, 64)
    np.testing.assert_array_equal(w[0], [1.0] * 32 + [-8.0] * 32)
    np.testing.assert_array_equal(w[1], [-8.0] * 32 + [1.0] * 32)


# ---- Q4_K -------------------------------------------------------------------

def pack_q4_k(d, dmin, sc, mn, codes):
    """sc, mn: 8 six-bit ints; codes: [8][32] ints in [0, 16) -> 144 bytes."""
    out = np.zeros(144, np.uint8)
    out[0:2] = _fp16(d)
    out[2:4] = _fp16(dmin)
    s = np.zeros(12, np.int64)
    for j in range(4):
        s[j] |= sc[j] & 63
        s[j + 4] |= mn[j] & 63
    for j in range(4, 8):
        s[j + 4] |= (sc[j] & 15) | ((mn[j] & 15) << 4)
        s[j - 4] |= (sc[j] >> 4) << 6
        s[j] |= (mn[j] >> 4) << 6
    out[4:16] = s.astype(np.uint8)
    for c in range(4):
        for l in range(32):
            out[16 + 32 * c + l] = codes[2 * c][l] | (codes[2 * c + 1][l] << 4)
    return out


def test_q4_k_block_layout():
    sc = [1, 2, 3, 4, 17, 33, 50, 63]          # sub-blocks 4..7 use the top two bits
    mn = [0, 5, 10, 63, 16, 32, 48, 1]
    codes = [[(l + 3 * s) % 16 for l in range(32)] for s in range(8)]
    d, dmin = 0.5, 0.25
    blob = pack_q4_k(d, dmin, sc, mn, codes)[None, :]
    w = O.dequantize_q4_k(blob, 1, 256)[0]
    want = [d * sc[s] * codes[s][l] - dmin * mn[s] for s in range(8) for l in range(32)]
    np.testing.assert_array_equal(w, want)
    scaled, offset = O.dequantize_q4_k(blob, 1, 256, parts=True)
    np.testing.assert_array_equal(scaled[0] - offset[0], want)
    np.testing.assert_array_equal(offset[0], np.repeat([dmin * m for m in mn], 32))


def test_q4_k_scale_unpacking_is_the_inverse_of_packing():
    rng = np.random.default_rng(3)
    for _ in range(50):
        sc, mn = rng.integers(0, 64, 8), rng.integers(0, 64, 8)
        blob = pack_q4_k(1.0, 1.0, sc, mn, [[0] * 32] * 8)
        got_sc, got_mn = O.q4_k_scales_mins(blob[4:16][None, :])
        np.testing.assert_array_equal(got_sc[0], sc)
        np.testing.assert_array_equal(got_mn[0], mn)


# ---- Q6_K -------------------------------------------------------------------

def pack_q6_k(d, scales, codes):
    """scales: 16 int8; codes: 256 ints in [0, 64) -> 210 bytes."""
    out = np.zeros(210, np.uint8)
    for h in range(2):
        for g in range(4):
            for l in range(32):
                c = codes[128 * h + 32 * g + l]
                i = 64 * h + l + 32 * (g % 2)
                out[i] |= (c & 15) if g < 2 else (c & 15) << 4
                out[128 + 32 * h + l] |= (c >> 4) << (2 * g)
    out[192:208] = np.array(scales, np.int8).view(np.uint8)
    out[208:210] = _fp16(d)
    return out


def test_q6_k_block_layout():
    codes = [(7 * t + 5) % 64 for t in range(256)]
    scales = [s - 8 for s in range(16)]         # negative scales: int8, not uint8
    d = 0.25
    blob = pack_q6_k(d, scales, codes)[None, :]
    w = O.dequantize_q6_k(blob, 1, 256)[0]
    np.testing.assert_array_equal(w, [d * scales[t // 16] * (codes[t] - 32) for t in range(256)])


def test_block_format_dispatch_and_q8_0():
    w32 = (np.arange(64, dtype=np.float32) - 31.5).reshape(1, 64) / 8
    blob = O.quantize_q8_0(w32)
    np.testing.assert_array_equal(O.dequantize_block_format(O.GGUF_TYPE_Q8_0, blob, 1, 64),
                                  O.dequantize_q8_0(blob, 1, 64).astype(np.float64))
    q6 = pack_q6_k(1.0, [1] * 16, [32] * 256)[None, :]
    np.testing.assert_array_equal(O.dequantize_block_format(O.GGUF_TYPE_Q6_K, q6, 1, 256), np.zeros((1, 256)))
