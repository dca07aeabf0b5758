"""Shared helpers for the GPU tests: device buffers come from torch, every
computation from the library's C ABI (through the ctypes binding)."""
import functools

import numpy as np
import pytest

try:
    import torch
except Exception:  # pragma: no cover
    torch = None


def gpu_available() -> bool:
    return torch is not None and torch.cuda.is_available()


def require_gpu():
    if not gpu_available():
        pytest.skip("no CUDA device")


@functools.lru_cache(maxsize=None)
def built_lib():
    from q8_quantized_llama_gb300 import build
    return build.build()


def binding():
    built_lib()
    from q8_quantized_llama_gb300 import binding as B
    B.lib()
    return B


def to_dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_quantize(w: np.ndarray):
    """Q8_0 blocks of an f32 host matrix, quantised by the library on the GPU.
    Returns a uint8 device tensor [rows, k/32*34]."""
    B = binding()
    rows, k = w.shape
    dw = to_dev(w.astype(np.float32))
    out = torch.empty((rows, k // 32 * 34), dtype=torch.uint8, device="cuda")
    B.llama_q8_quantize(dw, rows, k, out)
    torch.cuda.synchronize()
    del dw
    return out


def gpu_model_tensors(cfg, seed, host_f32=None):
    """GGUF-named device tensors for the library: matrices quantised on the
    GPU, norms copied. host_f32: optional dict of the f32 weights."""
    from q8_quantized_llama_gb300 import synth
    t = {}
    it = host_f32.items() if host_f32 is not None else (
        (n, w) for n, w, _ in synth.iter_model_weights_f32(cfg, seed))
    for name, w in it:
        t[name] = gpu_quantize(w) if w.ndim == 2 else to_dev(w)
    return t


def oracle_model_tensors(cfg, seed, host_f32=None):
    from oracle import q8_oracle as O
    from q8_quantized_llama_gb300 import synth
    t = {}
    it = host_f32.items() if host_f32 is not None else (
        (n, w) for n, w, _ in synth.iter_model_weights_f32(cfg, seed))
    for name, w in it:
        t[name] = O.quantize_q8_0(w) if w.ndim == 2 else w
    return t


def logits_close(got, ref, rel=2e-3):
    """max |got - ref| <= rel * max |ref| (the logits tolerance of the build)."""
    err = float(np.max(np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))))
    bound = rel * float(np.max(np.abs(ref)))
    return err <= bound, err, bound
