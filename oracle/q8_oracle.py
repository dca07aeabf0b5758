"""CPU oracle for one forward pass of a Q8_0-quantised Llama.

TEST INFRASTRUCTURE ONLY. The only code that may import or run this module is
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl
reference`` legs of ``bench.py``. The product (the CUDA library under
``q8_quantized_llama_gb300/`` and its ctypes binding) never imports it, and it
imports nothing from the product. Inputs come from the seeded generators in
``q8_quantized_llama_gb300/synth.py`` (which hold none of this arithmetic) or
from test fixtures.

Arithmetic: numpy, float64 for every reduction, matmul, norm, rotation and
softmax, float32 storage between ops (the model on the pages keeps the
embedding, every activation and the KV cache in f32). Q8_0 quantisation runs
in the precision the format fixes: f32 scale and f32 division, fp16 storage.

Sources, all candle 0.11.0 documentation pages:
  [QL] "量化 llama 的一次前向" (candle / 07-models / quantized-llama)
  [OT] "生成一个 token" (candle / 01-overview / one-token)
  [SP] "速度" (pytorch-to-candle / 09-deploy / speed)

Readings where the pages are silent:
  R1 Q8_0 block: the pages give only byte counts ([OT] "实验程序" file size,
     [OT] "读 GGUF" data offset, [SP] "CPU GGUF" 136.3 MiB). Blocks of 32
     along the input dim; d = max|w| / 127 in f32; q = round(w / d) with an
     f32 IEEE division and round-half-away-from-zero, clamped to +-127; d == 0
     gives q == 0; d stored as IEEE fp16 (round to nearest even) followed by
     the 32 int8 codes: 34 bytes per block.
  R2 RMSNorm: y = x * g / sqrt(mean(x^2) + eps), eps = 1e-5, mean over the
     hidden dim.
  R3 RoPE (rope_i, pairs 2i / 2i+1): angle = p * theta^(-2i/hd), theta 1e4,
     evaluated exactly (f64); rotation (a, b) -> (a c - b s, a s + b c).
  R4 GQA: query head h reads KV head h // (n_head / n_head_kv) (repeat_kv
     copies each KV head into a contiguous group).
  R5 Attention scale 1 / sqrt(head_dim), applied as a division in f64.
  R6 Activations are never quantised: Q8_0 weights times f32 activations.
  R7 Greedy argmax returns the lowest index among equal maxima.
  R13 Q5_0 / Q4_K / Q6_K blocks: the pages give their names, their timings
     and the byte census of a Q4_K_M file ([SP] "CPU GGUF"), not their
     layouts; those follow the published GGUF block definitions, and their
     byte sizes reproduce the census.

Parity pins (tests/test_oracle_pins.py): every public function here is pinned
against byte counts printed on the pages, hand-computed fixtures under
tests/golden/, closed forms or invariants stated on the pages. No function is
left "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np

QK8_0 = 32            # weights per Q8_0 block
Q8_0_BLOCK_BYTES = 34  # fp16 scale + 32 int8 codes
MAX_SEQ_LEN = 4096     # [QL] "from_gguf": fixed size of the cos/sin table


# --------------------------------------------------------------------------
# Q8_0 format (reading R1)
# --------------------------------------------------------------------------

def _round_half_away_from_zero(r32: np.ndarray) -> np.ndarray:
    """Round f32 values to integers, ties away from zero, exactly (via f64)."""
    r = r32.astype(np.float64)
    return np.where(r >= 0.0, np.floor(r + 0.5), -np.floor(-r + 0.5))


def quantize_q8_0(w: np.ndarray) -> np.ndarray:
    """Quantise an f32 matrix [rows, k] (k % 32 == 0) to Q8_0 blocks.

    Returns uint8 [rows, k / 32 * 34]: per block the fp16 scale
    (little-endian) then the 32 int8 codes. Reading R1; the block size and
    34-byte stride are fixed by the byte counts on [OT] and [SP].
    """
    w = np.ascontiguousarray(w, dtype=np.float32)
    if w.ndim != 2 or w.shape[1] % QK8_0 != 0:
        raise ValueError(f"quantize_q8_0 needs [rows, k] with k % 32 == 0, got {w.shape}")
    rows, k = w.shape
    nb = k // QK8_0
    blocks = w.reshape(rows, nb, QK8_0)
    amax = np.max(np.abs(blocks), axis=2)                  # f32
    d = (amax / np.float32(127.0)).astype(np.float32)      # f32 division
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = (blocks / d[..., None]).astype(np.float32)  # f32 IEEE division
    q = _round_half_away_from_zero(ratio)
    q = np.where(d[..., None] == 0.0, 0.0, q)
    q = np.clip(q, -127.0, 127.0).astype(np.int8)
    dh = d.astype("<f2")                                   # round to nearest even
    out = np.empty((rows, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    out[..., 0:2] = dh.view(np.uint8).reshape(rows, nb, 2)
    out[..., 2:] = q.view(np.uint8)
    return out.reshape(rows, nb * Q8_0_BLOCK_BYTES)


def q8_0_row_bytes(k: int) -> int:
    """Bytes one Q8_0 row of k weights occupies (reading R1)."""
    if k % QK8_0:
        raise ValueError("k must be a multiple of 32")
    return k // QK8_0 * Q8_0_BLOCK_BYTES


def q8_0_scales_and_codes(blob: np.ndarray, rows: int, k: int):
    """Split a Q8_0 blob into (fp16 scales [rows, k/32], int8 codes [rows, k])."""
    b = np.ascontiguousarray(blob, dtype=np.uint8).reshape(rows, k // QK8_0, Q8_0_BLOCK_BYTES)
    dh = np.ascontiguousarray(b[..., 0:2]).view("<f2")[..., 0]
    q = np.ascontiguousarray(b[..., 2:]).view(np.int8).reshape(rows, k)
    return dh, q


def dequantize_q8_0(blob: np.ndarray, rows: int, k: int) -> np.ndarray:
    """Q8_0 blob -> f32 [rows, k]; w = (f32) d * (f32) q, exact in f32."""
    dh, q = q8_0_scales_and_codes(blob, rows, k)
    w = dh.astype(np.float32)[..., None] * q.reshape(rows, k // QK8_0, QK8_0).astype(np.float32)
    return w.reshape(rows, k)


# --------------------------------------------------------------------------
# Other GGUF block formats (reading R13): Q5_0, Q4_K, Q6_K
# --------------------------------------------------------------------------
# [SP] "CPU GGUF：decode 快，prefill 慢" times QMatMul in Q5_0, Q4K and Q6K and
# lists the tensor census of the 135M Q4_K_M file (Q4K 16 tensors 7.6 MiB,
# Q5_0 166 tensors 51.2 MiB, Q6K 14 tensors 9.7 MiB, Q8_0 15 tensors 30.3 MiB);
# it notes that K-quant blocks hold 256 weights, so rows of 576 fall back to
# Q5_0. The pages do not print the layouts inside a block; they are read from
# the published GGUF block definitions, and the byte sizes below reproduce the
# census exactly (tests/test_oracle_pins.py).
GGUF_TYPE_Q5_0, GGUF_TYPE_Q8_0, GGUF_TYPE_Q4_K, GGUF_TYPE_Q6_K = 6, 8, 12, 14
# type -> (weights per block, bytes per block)
BLOCK_FORMATS = {GGUF_TYPE_Q5_0: (32, 22), GGUF_TYPE_Q8_0: (32, 34), GGUF_TYPE_Q4_K: (256, 144),
                 GGUF_TYPE_Q6_K: (256, 210)}


def block_format_row_bytes(gguf_type: int, k: int) -> int:
    """Bytes one row of k weights occupies in a block format."""
    qk, nbytes = BLOCK_FORMATS[gguf_type]
    if k % qk:
        raise ValueError(f"row length {k} is not a multiple of the block size {qk}")
    return k // qk * nbytes


def _blocks(blob, rows, k, gguf_type):
    qk, nbytes = BLOCK_FORMATS[gguf_type]
    return np.ascontiguousarray(blob, dtype=np.uint8).reshape(rows, k // qk, nbytes)


def _f16(b2: np.ndarray) -> np.ndarray:
    """Little-endian fp16 in the last axis (2 bytes) -> f64."""
    return np.ascontiguousarray(b2).view("<f2")[..., 0].astype(np.float64)


def dequantize_q5_0(blob: np.ndarray, rows: int, k: int) -> np.ndarray:
    """Q5_0 -> f64 [rows, k]. Block of 32 weights, 22 bytes: fp16 scale d, a
    32-bit little-endian word qh whose bit j is the fifth bit of weight j, and
    16 bytes qs whose byte j holds the low four bits of weight j (low nibble)
    and of weight j + 16 (high nibble). w_j = d * (code_j - 16)."""
    b = _blocks(blob, rows, k, GGUF_TYPE_Q5_0)
    d = _f16(b[..., 0:2])
    qh = np.ascontiguousarray(b[..., 2:6]).view("<u4")[..., 0].astype(np.int64)
    qs = b[..., 6:22].astype(np.int64)
    low = np.concatenate([qs & 0x0F, qs >> 4], axis=-1)                   # weights 0..15, 16..31
    high = (qh[..., None] >> np.arange(32)) & 1
    q = (low | (high << 4)) - 16
    return (d[..., None] * q).reshape(rows, k)


def q4_k_scales_mins(sc12: np.ndarray):
    """The eight 6-bit (scale, min) pairs packed into a Q4_K block's 12 bytes:
    sub-blocks 0-3 take the low six bits of bytes j (scale) and j + 4 (min);
    sub-blocks 4-7 take the low / high nibble of byte j + 4 for the low four
    bits and the top two bits of bytes j - 4 (scale) and j (min)."""
    b = sc12.astype(np.int64)
    sc = np.empty(b.shape[:-1] + (8,), np.int64)
    mn = np.empty_like(sc)
    for j in range(4):
        sc[..., j] = b[..., j] & 63
        mn[..., j] = b[..., j + 4] & 63
    for j in range(4, 8):
        sc[..., j] = (b[..., j + 4] & 0x0F) | ((b[..., j - 4] >> 6) << 4)
        mn[..., j] = (b[..., j + 4] >> 4) | ((b[..., j] >> 6) << 4)
    return sc, mn


def dequantize_q4_k(blob: np.ndarray, rows: int, k: int, parts: bool = False):
    """Q4_K -> f64 [rows, k]. Block of 256 weights, 144 bytes: fp16 d, fp16
    dmin, 12 bytes of packed 6-bit (scale, min) pairs for eight sub-blocks of
    32, then 128 bytes of 4-bit codes: bytes [32c, 32c + 32) hold sub-block 2c
    in their low nibbles and sub-block 2c + 1 in their high nibbles.
    w = d * scale_s * q - dmin * min_s. parts=True returns the two terms
    (d * scale * q, dmin * min) separately."""
    b = _blocks(blob, rows, k, GGUF_TYPE_Q4_K)
    d = _f16(b[..., 0:2])
    dmin = _f16(b[..., 2:4])
    sc, mn = q4_k_scales_mins(b[..., 4:16])
    qs = b[..., 16:144].astype(np.int64).reshape(rows, k // 256, 4, 32)
    q = np.stack([qs & 0x0F, qs >> 4], axis=3).reshape(rows, k // 256, 8, 32)   # [.., sub-block, 32]
    scaled = d[..., None, None] * sc[..., None] * q
    offset = np.broadcast_to((dmin[..., None] * mn)[..., None], scaled.shape)
    if parts:
        return scaled.reshape(rows, k), np.ascontiguousarray(offset).reshape(rows, k)
    return (scaled - offset).reshape(rows, k)


def dequantize_q6_k(blob: np.ndarray, rows: int, k: int) -> np.ndarray:
    """Q6_K -> f64 [rows, k]. Block of 256 weights, 210 bytes: 128 bytes ql
    (low four bits), 64 bytes qh (top two bits), 16 int8 scales (one per 16
    weights), fp16 d. Each half h of 128 weights uses ql[64h, 64h + 64) and
    qh[32h, 32h + 32): for l < 32, weights 128h + 32g + l (g = 0..3) take the
    low (g even) or high (g odd) nibble of ql[64h + l + 32 (g % 2)] and bits
    2g, 2g + 1 of qh[32h + l]. w_t = d * scale[t // 16] * (code_t - 32)."""
    b = _blocks(blob, rows, k, GGUF_TYPE_Q6_K)
    nb = k // 256
    ql = b[..., 0:128].astype(np.int64).reshape(rows, nb, 2, 64)
    qh = b[..., 128:192].astype(np.int64).reshape(rows, nb, 2, 32)
    scales = np.ascontiguousarray(b[..., 192:208]).view(np.int8).astype(np.int64)
    d = _f16(b[..., 208:210])
    codes = np.empty((rows, nb, 2, 4, 32), np.int64)
    for g in range(4):
        nib = ql[..., 32 * (g % 2): 32 * (g % 2) + 32]
        low = (nib & 0x0F) if g < 2 else (nib >> 4)
        codes[..., g, :] = low | (((qh >> (2 * g)) & 3) << 4)
    q = codes.reshape(rows, nb, 256) - 32
    w = d[..., None] * np.repeat(scales, 16, axis=-1) * q
    return w.reshape(rows, k)


def dequantize_block_format(gguf_type: int, blob: np.ndarray, rows: int, k: int) -> np.ndarray:
    """Any of the block formats above (and Q8_0) -> f64 [rows, k]."""
    if gguf_type == GGUF_TYPE_Q8_0:
        return dequantize_q8_0(blob, rows, k).astype(np.float64)
    return {GGUF_TYPE_Q5_0: dequantize_q5_0, GGUF_TYPE_Q4_K: dequantize_q4_k,
            GGUF_TYPE_Q6_K: dequantize_q6_k}[gguf_type](blob, rows, k)


# --------------------------------------------------------------------------
# Layer operations
# --------------------------------------------------------------------------

def rms_norm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RmsNorm over the last dim (reading R2): x * g / sqrt(mean(x^2) + eps).

    [QL] "forward：mask 什么时候建": attention_norm, ffn_norm and the final norm.
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    ms = np.mean(x64 * x64, axis=-1, keepdims=True)
    y = x64 / np.sqrt(ms + float(eps)) * np.asarray(g, dtype=np.float32).astype(np.float64)
    return y.astype(np.float32)


def linear(x: np.ndarray, w: np.ndarray) -> np.ndarray:
    """y = x W^T with W already dequantised (QMatMul forward); f64 products."""
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    w64 = w if w.dtype == np.float64 else w.astype(np.float64)
    return (x64 @ w64.T).astype(np.float32)


def rope_freqs(head_dim: int, theta: float) -> np.ndarray:
    """theta^(-2i/hd) for i < hd/2 (reading R3)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_table(head_dim: int, theta: float, max_seq: int = MAX_SEQ_LEN):
    """cos/sin table of shape [max_seq, head_dim/2] ([QL] "from_gguf").

    Positions past max_seq are out of range: the pages report a narrow error
    for index_pos 4096 with a [4096, 32] table.
    """
    ang = np.arange(max_seq, dtype=np.float64)[:, None] * rope_freqs(head_dim, theta)[None, :]
    return np.cos(ang), np.sin(ang)


def rope_i(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """Interleaved RoPE (the Llama convention): dims 2i and 2i+1 form a pair.

    x: [T, heads, hd] f32; positions: [T] absolute positions.
    [QL] "RoPE：两种约定，按架构名选".
    """
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    hd = x64.shape[-1]
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_freqs(hd, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a = x64[..., 0::2]
    b = x64[..., 1::2]
    out = np.empty_like(x64)
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = a * s + b * c
    return out.astype(np.float32)


def rope_neox(x: np.ndarray, positions: np.ndarray, theta: float) -> np.ndarray:
    """NEOX RoPE: dim i pairs with dim i + hd/2 (the other convention on
    [QL] "RoPE：两种约定，按架构名选"; not on the Llama path, kept for the
    pairing pin)."""
    x64 = np.asarray(x, dtype=np.float32).astype(np.float64)
    hd = x64.shape[-1]
    half = hd // 2
    ang = np.asarray(positions, dtype=np.float64)[:, None] * rope_freqs(hd, theta)[None, :]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    a = x64[..., :half]
    b = x64[..., half:]
    out = np.empty_like(x64)
    out[..., :half] = a * c - b * s
    out[..., half:] = a * s + b * c
    return out.astype(np.float32)


def build_causal_mask(seq_len: int, index_pos: int) -> np.ndarray:
    """uint8 mask [seq_len, index_pos + seq_len]; 1 = may not attend.

    [QL] "forward：mask 什么时候建": kv_len = index_pos + seq_len, the first
    index_pos columns (the cached prefix) are visible, the last seq_len
    columns form a causal triangle.
    """
    kv_len = index_pos + seq_len
    i = np.arange(seq_len)[:, None]
    j = np.arange(kv_len)[None, :]
    return (j > index_pos + i).astype(np.uint8)


def repeat_kv(x: np.ndarray, n_rep: int) -> np.ndarray:
    """[kv_len, n_kv_head, hd] -> [kv_len, n_kv_head * n_rep, hd] (reading R4)."""
    return np.repeat(x, n_rep, axis=1)


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, mask: np.ndarray | None) -> np.ndarray:
    """softmax(q k^T / sqrt(hd) + mask) v with repeat_kv materialised.

    q: [T, n_head, hd]; k, v: [kv_len, n_kv_head, hd] (the whole cache);
    mask: uint8 [T, mask_kv] or None. A mask whose width differs from the
    cache length is an error, as the broadcast failure on [QL]
    "index_pos 传错" shows. [QL] "forward_attn：自己拼 KV"; [OT] "prefill 和
    decode：同一个 forward，不同的路".
    """
    T, n_head, hd = q.shape
    kv_len, n_kv, _ = k.shape
    n_rep = n_head // n_kv
    kr = repeat_kv(np.asarray(k, np.float32), n_rep).astype(np.float64)
    vr = repeat_kv(np.asarray(v, np.float32), n_rep).astype(np.float64)
    q64 = np.asarray(q, np.float32).astype(np.float64)
    # scores[h, t, j] = q[t, h] . k[j, h] / sqrt(hd): one f64 matrix product per head
    att = np.matmul(q64.transpose(1, 0, 2), kr.transpose(1, 2, 0)) / math.sqrt(hd)
    if mask is not None:
        if mask.shape != (T, kv_len):
            raise ValueError(
                f"cannot broadcast {list(mask.shape)} to {[1, n_head, T, kv_len]}")
        att = np.where(mask[None, :, :] != 0, -np.inf, att)
    m = np.max(att, axis=-1, keepdims=True)
    e = np.exp(att - m)
    p = e / np.sum(e, axis=-1, keepdims=True)
    # o[t, h] = sum_j p[h, t, j] v[j, h]
    o = np.matmul(p, vr.transpose(1, 0, 2)).transpose(1, 0, 2)
    return o.astype(np.float32)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)), f64."""
    z64 = np.asarray(z, dtype=np.float64)
    return z64 / (1.0 + np.exp(-z64))


def argmax_lowest(logits: np.ndarray) -> int:
    """Greedy token: the lowest index among the maxima (reading R7)."""
    return int(np.argmax(np.asarray(logits)))   # numpy returns the first maximum


# --------------------------------------------------------------------------
# Model
# --------------------------------------------------------------------------

LAYER_MATRICES = ("attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up", "ffn_down")


def layer_matrix_shape(cfg: dict, name: str):
    h, hd = cfg["n_embd"], cfg["head_dim"]
    return {
        "attn_q": (cfg["n_head"] * hd, h),
        "attn_k": (cfg["n_head_kv"] * hd, h),
        "attn_v": (cfg["n_head_kv"] * hd, h),
        "attn_output": (h, cfg["n_head"] * hd),
        "ffn_gate": (cfg["n_ff"], h),
        "ffn_up": (cfg["n_ff"], h),
        "ffn_down": (h, cfg["n_ff"]),
    }[name]


class ModelWeights:
    """Q8_0 Llama with a growing per-layer KV cache, step by step as the
    pages describe ``ModelWeights::forward`` / ``forward_attn``
    ([QL] "forward：mask 什么时候建", "forward_attn：自己拼 KV",
    "换 prompt 要不要 clear_kv_cache"; [OT] "建模型：按名字取张量").

    ``tensors`` maps GGUF names to arrays: Q8_0 blobs (uint8 [rows, k/32*34])
    for ``token_embd.weight``, ``output.weight`` (optional; absent means the
    head shares the Q8_0 embedding) and ``blk.{i}.{attn_q,...}.weight``;
    f32 vectors for ``blk.{i}.attn_norm.weight``, ``blk.{i}.ffn_norm.weight``
    and ``output_norm.weight``.

    ``weight_cache``: "f64" keeps dequantised matrices in f64, "f32" in f32
    (same values, half the memory), "none" dequantises at every use.
    """

    def __init__(self, cfg: dict, tensors: dict, weight_cache: str = "f64"):
        self.cfg = dict(cfg)
        self.t = tensors
        self.weight_cache = weight_cache
        self._deq: dict = {}
        h, V = cfg["n_embd"], cfg["n_vocab"]
        if tensors["token_embd.weight"].shape != (V, q8_0_row_bytes(h)):
            raise ValueError("token_embd.weight has the wrong shape")
        # The embedding is dequantised to f32 once ([OT] "建模型").
        self.tok_embeddings = dequantize_q8_0(tensors["token_embd.weight"], V, h)
        self.tied = "output.weight" not in tensors
        self.max_seq = int(cfg.get("max_seq", MAX_SEQ_LEN))
        self.counters = {"qmatmul": 0, "rms_norm": 0, "rope": 0}
        self.clear_kv_cache()

    # -- weights ----------------------------------------------------------
    def _matrix(self, name: str, rows: int, k: int) -> np.ndarray:
        if name in self._deq:
            return self._deq[name]
        if name == "token_embd.weight":
            w = self.tok_embeddings           # same values as the Q8_0 head
        else:
            w = dequantize_q8_0(self.t[name], rows, k)
        if self.weight_cache == "f64":
            w = w.astype(np.float64)
            self._deq[name] = w
        elif self.weight_cache == "f32":
            self._deq[name] = w
        return w

    def _qmatmul(self, x: np.ndarray, name: str, rows: int, k: int) -> np.ndarray:
        self.counters["qmatmul"] += 1
        return linear(x, self._matrix(name, rows, k))

    def _norm(self, x, name):
        self.counters["rms_norm"] += 1
        return rms_norm(x, self.t[name], self.cfg["rms_eps"])

    def _rope(self, x, positions):
        """rope_i, or NEOX when cfg["rope_style"] == 1 (the loader's choice by
        architecture name, [QL] "RoPE：两种约定，按架构名选")."""
        self.counters["rope"] += 1
        rope = rope_neox if int(self.cfg.get("rope_style", 0)) == 1 else rope_i
        return rope(x, positions, self.cfg["rope_theta"])

    # -- state ------------------------------------------------------------
    def clear_kv_cache(self):
        """Drop every layer's cache ([QL] "换 prompt 要不要 clear_kv_cache")."""
        self.kv_cache = [None] * self.cfg["n_layer"]

    def cache_len(self) -> int:
        c = self.kv_cache[0]
        return 0 if c is None else int(c[0].shape[0])

    # -- forward ----------------------------------------------------------
    def forward(self, ids, index_pos: int) -> np.ndarray:
        """Logits (f32 [n_vocab]) for the last of the T input positions."""
        cfg = self.cfg
        ids = np.asarray(ids, dtype=np.int64).reshape(-1)
        T = int(ids.shape[0])
        if T < 1:
            raise ValueError("empty input")
        if index_pos < 0 or index_pos + T > self.max_seq:
            # The rotary table holds max_seq rows; narrowing past it fails.
            raise ValueError(
                f"narrow invalid args start + len > dim_len: [{self.max_seq}, "
                f"{cfg['head_dim'] // 2}], dim: 0, start: {index_pos}, len:{T}")
        if np.any(ids < 0) or np.any(ids >= cfg["n_vocab"]):
            raise ValueError("token id out of range")
        h, hd = cfg["n_embd"], cfg["head_dim"]
        nh, nkv, nff = cfg["n_head"], cfg["n_head_kv"], cfg["n_ff"]
        mask = None if T == 1 else build_causal_mask(T, index_pos)
        positions = np.arange(index_pos, index_pos + T)
        x = self.tok_embeddings[ids].astype(np.float32)          # [T, h]
        for li in range(cfg["n_layer"]):
            p = f"blk.{li}."
            residual = x
            y = self._norm(x, p + "attn_norm.weight")
            q = self._qmatmul(y, p + "attn_q.weight", nh * hd, h).reshape(T, nh, hd)
            k = self._qmatmul(y, p + "attn_k.weight", nkv * hd, h).reshape(T, nkv, hd)
            v = self._qmatmul(y, p + "attn_v.weight", nkv * hd, h).reshape(T, nkv, hd)
            q = self._rope(q, positions)
            k = self._rope(k, positions)
            prev = self.kv_cache[li]
            if index_pos == 0 or prev is None:
                kc, vc = k, v                                      # drop the old cache
            else:
                kc = np.concatenate([prev[0], k], axis=0)          # cat on the seq dim
                vc = np.concatenate([prev[1], v], axis=0)
            attn = attention(q, kc, vc, mask).reshape(T, nh * hd)
            self.kv_cache[li] = (kc, vc)
            x = (residual.astype(np.float64)
                 + self._qmatmul(attn, p + "attn_output.weight", h, nh * hd)).astype(np.float32)
            residual = x
            y = self._norm(x, p + "ffn_norm.weight")
            g = self._qmatmul(y, p + "ffn_gate.weight", nff, h)
            u = self._qmatmul(y, p + "ffn_up.weight", nff, h)
            a = (silu(g) * u.astype(np.float64)).astype(np.float32)
            x = (residual.astype(np.float64)
                 + self._qmatmul(a, p + "ffn_down.weight", h, nff)).astype(np.float32)
        y = self._norm(x[T - 1:T], "output_norm.weight")              # last position only
        head = "token_embd.weight" if self.tied else "output.weight"
        logits = self._qmatmul(y, head, cfg["n_vocab"], h)
        return logits[0]

    def generate(self, prompt, n_new: int):
        """Greedy loop of [OT] "实验程序": prefill at 0, then one token per step
        at pos = tokens processed so far. Returns (new_ids, per-step logits)."""
        ids = list(int(t) for t in prompt)
        logits = self.forward(ids, 0)
        out, all_logits = [], [logits]
        nxt = argmax_lowest(logits)
        out.append(nxt)
        pos = len(ids)
        for _ in range(n_new):
            logits = self.forward([nxt], pos)
            pos += 1
            all_logits.append(logits)
            nxt = argmax_lowest(logits)
            out.append(nxt)
        return out, all_logits
