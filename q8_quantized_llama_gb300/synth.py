"""Seeded synthetic inputs: model weights, prompts and activations.

This module draws random numbers and nothing else. It holds no Q8_0, norm,
rotation, attention or matmul arithmetic, so that both the CUDA path and the
CPU oracle can take their inputs from it without sharing any of the method.

Workload shapes follow the Q8_0 Llama the candle pages time ("生成一个 token",
"实验程序": SmolLM2-135M, 30 layers, hidden 576, 9 query / 3 KV heads of 64,
FFN 1536, vocabulary 49152) and a Llama-7B-shaped model. The pages use trained
weights and real prompts; here matrices are N(0, 0.02) drawn in f32, norm
weights 1 + N(0, 0.02), and prompts are uniform random token ids.

Every tensor is drawn from its own numpy PCG64 stream seeded by
(seed, tensor index, row chunk), so a tensor's values do not depend on which
other tensors are drawn or on the number of threads drawing them.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os

import numpy as np

MODEL_135M = dict(n_layer=30, n_embd=576, n_head=9, n_head_kv=3, head_dim=64, n_ff=1536,
                  n_vocab=49152, max_seq=4096, rms_eps=1e-5, rope_theta=10000.0, tied_output=1)
MODEL_7B = dict(n_layer=32, n_embd=4096, n_head=32, n_head_kv=8, head_dim=128, n_ff=14336,
                n_vocab=32000, max_seq=4096, rms_eps=1e-5, rope_theta=10000.0, tied_output=0)

WEIGHT_STD = 0.02
_ROW_CHUNK = 256

_LAYER_TENSORS = ("attn_norm", "attn_q", "attn_k", "attn_v", "attn_output",
                  "ffn_norm", "ffn_gate", "ffn_up", "ffn_down")


def model_tensor_specs(cfg: dict):
    """[(gguf name, shape, kind)] in file order; kind is "matrix" or "norm".

    30 layers x 9 tensors + token_embd + output_norm = 272 for the 135M shape
    (plus output.weight when the head is not tied).
    """
    h, hd, nff = cfg["n_embd"], cfg["head_dim"], cfg["n_ff"]
    qd, kvd = cfg["n_head"] * hd, cfg["n_head_kv"] * hd
    shapes = {"attn_norm": (h,), "ffn_norm": (h,), "attn_q": (qd, h), "attn_k": (kvd, h),
              "attn_v": (kvd, h), "attn_output": (h, qd), "ffn_gate": (nff, h),
              "ffn_up": (nff, h), "ffn_down": (h, nff)}
    specs = [("token_embd.weight", (cfg["n_vocab"], h), "matrix")]
    for i in range(cfg["n_layer"]):
        for t in _LAYER_TENSORS:
            specs.append((f"blk.{i}.{t}.weight", shapes[t], "norm" if t.endswith("norm") else "matrix"))
    specs.append(("output_norm.weight", (h,), "norm"))
    if not cfg.get("tied_output", 1):
        specs.append(("output.weight", (cfg["n_vocab"], h), "matrix"))
    return specs


def _fill_normal(out: np.ndarray, seed_words) -> None:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(seed_words))))
    rng.standard_normal(out=out, dtype=np.float32)


def _draw_tensor(shape, kind: str, seed: int, index: int, pool=None) -> np.ndarray:
    out = np.empty(shape, dtype=np.float32)
    if len(shape) == 1:
        _fill_normal(out, (seed, index, 0))
    else:
        rows = shape[0]
        chunks = [(r, min(r + _ROW_CHUNK, rows)) for r in range(0, rows, _ROW_CHUNK)]
        jobs = [(out[a:b], (seed, index, ci)) for ci, (a, b) in enumerate(chunks)]
        if pool is None:
            for view, words in jobs:
                _fill_normal(view, words)
        else:
            list(pool.map(lambda j: _fill_normal(*j), jobs))
    out *= np.float32(WEIGHT_STD)
    if kind == "norm":
        out += np.float32(1.0)
    return out


def iter_model_weights_f32(cfg: dict, seed: int, threads: int | None = None):
    """Yield (name, f32 array, kind) for every tensor of the model, in order."""
    threads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(max_workers=threads) as pool:
        for idx, (name, shape, kind) in enumerate(model_tensor_specs(cfg)):
            yield name, _draw_tensor(shape, kind, seed, idx, pool), kind


def model_weights_f32(cfg: dict, seed: int, threads: int | None = None) -> dict:
    """All tensors of the model as f32 arrays, keyed by GGUF name."""
    return {name: w for name, w, _ in iter_model_weights_f32(cfg, seed, threads)}


def prompt_ids(n: int, n_vocab: int, seed: int) -> np.ndarray:
    """n token ids uniform in [0, n_vocab), int32 (no special tokens)."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0x1D5, n])))
    return rng.integers(0, n_vocab, size=n, dtype=np.int64).astype(np.int32)


def normal_f32(shape, seed: int, stream: int = 0, std: float = 1.0) -> np.ndarray:
    """N(0, std) f32 array, e.g. activations or q/k/v for kernel workloads."""
    out = np.empty(shape, dtype=np.float32)
    _fill_normal(out.reshape(-1), (seed, 0xAC7, stream))
    if std != 1.0:
        out *= np.float32(std)
    return out


def weight_matrix_f32(rows: int, k: int, seed: int, stream: int = 0) -> np.ndarray:
    """One N(0, 0.02) f32 weight matrix [rows, k] for the isolated linear sweep."""
    return normal_f32((rows, k), seed, 0x3000 + stream, WEIGHT_STD)


# Other GGUF block formats: (weights per block, bytes per block, byte offsets of
# the fp16 scale fields). Random blocks are random bytes with those fields
# replaced by finite fp16 values of a typical magnitude.
_BLOCK_FORMATS = {6: (32, 22, (0,)), 12: (256, 144, (0, 2)), 14: (256, 210, (208,))}


def random_blocks(gguf_type: int, rows: int, k: int, seed: int, stream: int = 0) -> np.ndarray:
    """uint8 [rows, k / block * block bytes] of random Q5_0 (6), Q4_K (12) or
    Q6_K (14) blocks: every code, scale and min byte uniform, fp16 scales
    |N(0, 1)| * 2^-7 (so weights stay of order 0.1)."""
    qk, nbytes, f16_at = _BLOCK_FORMATS[gguf_type]
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xB10C, gguf_type, stream])))
    blocks = rng.integers(0, 256, size=(rows, k // qk, nbytes), dtype=np.uint8)
    for off in f16_at:
        scale = (np.abs(rng.standard_normal((rows, k // qk))) * 2.0 ** -7).astype("<f2")
        blocks[..., off:off + 2] = scale.view(np.uint8).reshape(rows, k // qk, 2)
    return blocks.reshape(rows, k // qk * nbytes)
