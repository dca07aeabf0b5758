"""The C-ABI library builds, loads and exports every symbol include/llama_q8.h
declares; argument checks that need no GPU return their status codes."""
import ctypes as C
import os
import re

import pytest

from tests.conftest import ROOT
from tests.gpu_helpers import built_lib


@pytest.fixture(scope="module")
def B():
    built_lib()
    from q8_quantized_llama_gb300 import binding
    binding.lib()
    return binding


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "llama_q8.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(llama_q8_[a-z0-9_]+)\s*\(", text)))


def test_header_lists_the_binding_exports(B):
    assert sorted(B.EXPORTS) == _declared_symbols()


def test_library_exports_every_declared_symbol(B):
    lib = C.CDLL(B.LIB_PATH)
    for name in _declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(B):
    for s in range(9):
        assert B.status_str(s)
    assert B.status_str(0) == "ok"


def test_null_arguments_rejected_without_a_gpu(B):
    L = B.lib()
    out = C.c_void_p()
    assert L.llama_q8_load(None, None, 0, C.byref(out)) == B.LQ8_ERR_ARG
    assert L.llama_q8_forward(None, None, 1, 0, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_forward_argmax(None, None, 1, 0, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_generate(None, None, 1, 1, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_reset(None) == B.LQ8_ERR_ARG
    assert L.llama_q8_free(None) == B.LQ8_OK
    assert L.llama_q8_quantize(None, 1, 32, None, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_matmul(None, 1, 32, None, 1, None, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_matmul_ex(None, 1, 32, None, 1, None, 0, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_selftest_wait_timeout(None) == B.LQ8_ERR_ARG
    assert L.llama_q8_attention(None, None, None, 1, 0, 9, 3, 64, 4096, None, None, 0, None) == B.LQ8_ERR_ARG


def test_config_validation_without_a_gpu(B):
    import numpy as np
    from q8_quantized_llama_gb300 import synth
    cfg = dict(synth.MODEL_135M, n_layer=1)
    dummy = np.zeros(64, np.uint8)
    t = {n: dummy for n, _, _ in synth.model_tensor_specs(cfg)}
    for bad, status in [(dict(head_dim=96), B.LQ8_ERR_UNSUPPORTED), (dict(n_embd=500), B.LQ8_ERR_UNSUPPORTED),
                        (dict(n_head_kv=4), B.LQ8_ERR_ARG), (dict(n_layer=0), B.LQ8_ERR_ARG),
                        (dict(tied_output=0), B.LQ8_ERR_ARG), (dict(decode_kernel=6), B.LQ8_ERR_ARG),
                        (dict(decode_kernel=-1), B.LQ8_ERR_ARG), (dict(rope_style=2), B.LQ8_ERR_ARG),
                        (dict(rope_style=-1), B.LQ8_ERR_ARG),
                        # the one-cluster whole-step and per-layer forms are not built
                        (dict(decode_kernel=2), B.LQ8_ERR_UNSUPPORTED), (dict(decode_kernel=5), B.LQ8_ERR_UNSUPPORTED),
                        # split-K lm_head: 2..8 CTAs, no more than n_embd / 32
                        (dict(head_splits=1), B.LQ8_ERR_ARG), (dict(head_splits=9), B.LQ8_ERR_ARG),
                        (dict(head_splits=-1), B.LQ8_ERR_ARG)]:
        c = B.make_config(dict(cfg, **bad))
        w, keep = B.make_weights(cfg, t, on_device=False)
        out = C.c_void_p()
        assert B.lib().llama_q8_load(C.byref(c), C.byref(w), 0, C.byref(out)) == status, bad


def test_size_queries(B):
    assert B.llama_q8_packed_bytes(576, 576) == 576 * 576 + 576 * 18 * 2
    assert B.llama_q8_packed_bytes(1, 32) == 32 * 32 + (256 - 32 * 32 % 256) % 256 + 32 * 2
    assert B.llama_q8_packed_bytes(10, 31) == 0
    assert B.llama_q8_attention_workspace_bytes(9, 3, 64, 4096) > 0
    assert B.llama_q8_attention_workspace_bytes(9, 4, 64, 4096) == 0


def test_rope_style_by_architecture_name(B):
    """The loader's choice of rotary convention by general.architecture: NEOX
    for the names the pages print from its list, rope_i for llama and any
    other name ("量化 llama 的一次前向", RoPE：两种约定，按架构名选)."""
    for arch in ("qwen", "qwen2", "falcon", "phi3", "stablelm"):
        assert B.rope_style_for_arch(arch) == 1, arch
    for arch in ("llama", "Qwen2", "qwen3moe", "", "mistral"):
        assert B.rope_style_for_arch(arch) == 0, arch
    assert B.rope_style_for_arch(None) == -1


def test_matmul_argument_checks_without_a_gpu(B):
    """llama_q8_matmul_ex refuses bad arguments on the host, before any CUDA
    call: the pointers below are never dereferenced (16-byte aligned stand-in
    addresses, or misaligned ones where the check is the alignment)."""
    L = B.lib()
    p, x, y = C.c_void_p(1 << 20), C.c_void_p(1 << 21), C.c_void_p(1 << 22)
    tc, cc = B.LQ8_MATMUL_TENSOR_CORES, B.LQ8_MATMUL_CUDA_CORES
    assert L.llama_q8_matmul_ex(p, 64, 33, x, 20, y, 0, None) == B.LQ8_ERR_ARG       # k % 32
    assert L.llama_q8_matmul_ex(p, 0, 64, x, 20, y, 0, None) == B.LQ8_ERR_ARG        # rows
    assert L.llama_q8_matmul_ex(p, 64, 64, x, 0, y, 0, None) == B.LQ8_ERR_ARG        # m
    assert L.llama_q8_matmul_ex(p, 64, 64, x, 20, y, 8, None) == B.LQ8_ERR_ARG       # unknown flag bit
    assert L.llama_q8_matmul_ex(p, 64, 64, x, 20, y, tc | cc, None) == B.LQ8_ERR_ARG  # both kernels forced
    assert L.llama_q8_matmul_ex(C.c_void_p((1 << 20) + 4), 64, 64, x, 20, y, 0, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_matmul_ex(p, 64, 64, C.c_void_p((1 << 21) + 8), 20, y, 0, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_matmul_ex(p, (1 << 30) + 1, 64, x, 20, y, 0, None) == B.LQ8_ERR_UNSUPPORTED


@pytest.mark.parametrize("entry", ["llama_q8_attention_decode", "llama_q8_attention_decode_noalloc"])
def test_decode_attention_argument_checks_without_a_gpu(B, entry):
    """The decode attention entries refuse bad shapes and misaligned buffers on
    the host, before any CUDA call (stand-in addresses, never dereferenced)."""
    f = getattr(B.lib(), entry)
    q, k, v, o = (C.c_void_p(a << 20) for a in (1, 2, 3, 4))
    assert f(q, k, v, 0, 9, 3, 64, 4096, o, None) == B.LQ8_ERR_ARG           # kv_len
    assert f(q, k, v, 100, 9, 4, 64, 4096, o, None) == B.LQ8_ERR_ARG         # heads not grouped evenly
    assert f(q, k, v, 4097, 9, 3, 64, 4096, o, None) == B.LQ8_ERR_CTX        # past the cache
    assert f(q, k, v, 100, 9, 3, 96, 4096, o, None) == B.LQ8_ERR_UNSUPPORTED  # head_dim
    assert f(q, k, v, 100, 18, 1, 64, 4096, o, None) == B.LQ8_ERR_UNSUPPORTED  # group of 18 > 8
    for bad in range(4):
        ptrs = [q, k, v, o]
        ptrs[bad] = C.c_void_p(((bad + 1) << 20) + 4)                        # misaligned buffer
        assert f(ptrs[0], ptrs[1], ptrs[2], 100, 9, 3, 64, 4096, ptrs[3], None) == B.LQ8_ERR_ARG, bad


def test_prefill_attention_argument_checks_without_a_gpu(B):
    """llama_q8_attention (T > 1) refuses bad shapes, a prompt past the cache
    and misaligned buffers on the host, before any CUDA call."""
    f = B.lib().llama_q8_attention
    q, k, v, o = (C.c_void_p(a << 20) for a in (1, 2, 3, 4))
    assert f(q, k, v, 0, 0, 9, 3, 64, 4096, o, None, 0, None) == B.LQ8_ERR_ARG            # T
    assert f(q, k, v, 8, -1, 9, 3, 64, 4096, o, None, 0, None) == B.LQ8_ERR_ARG           # index_pos
    assert f(q, k, v, 8, 0, 9, 2, 64, 4096, o, None, 0, None) == B.LQ8_ERR_ARG            # 9 heads over 2
    assert f(q, k, v, 8, 4090, 9, 3, 64, 4096, o, None, 0, None) == B.LQ8_ERR_CTX         # index_pos + T > 4096
    assert f(q, k, v, 8, 0, 9, 3, 32, 4096, o, None, 0, None) == B.LQ8_ERR_UNSUPPORTED    # head_dim
    assert f(q, k, v, 8, 0, 32, 2, 64, 4096, o, None, 0, None) == B.LQ8_ERR_UNSUPPORTED   # group of 16
    assert f(q, k, C.c_void_p((3 << 20) + 8), 8, 0, 9, 3, 64, 4096, o, None, 0, None) == B.LQ8_ERR_ARG


def test_block_format_matvec_argument_checks_without_a_gpu(B):
    """llama_q8_matvec_fmt refuses unsupported types, k off the block size,
    unknown flags and misaligned buffers on the host; the packed size query
    is 0 for those shapes."""
    L = B.lib()
    p, x, y = C.c_void_p(1 << 20), C.c_void_p(1 << 21), C.c_void_p(1 << 22)
    q4_k, q5_0 = 12, 6
    assert L.llama_q8_matvec_fmt(q4_k, p, 64, 128, x, y, 0, None) == B.LQ8_ERR_ARG         # k % 256
    assert L.llama_q8_matvec_fmt(q5_0, p, 64, 48, x, y, 0, None) == B.LQ8_ERR_ARG          # k % 32
    assert L.llama_q8_matvec_fmt(2, p, 64, 256, x, y, 0, None) == B.LQ8_ERR_UNSUPPORTED    # Q4_0: not built
    assert L.llama_q8_matvec_fmt(q4_k, p, 64, 256, x, y, 4, None) == B.LQ8_ERR_ARG         # unknown flag
    assert L.llama_q8_matvec_fmt(q4_k, C.c_void_p((1 << 20) + 4), 64, 256, x, y, 0, None) == B.LQ8_ERR_ARG
    assert L.llama_q8_packed_bytes_fmt(q4_k, 64, 128) == 0
    assert L.llama_q8_packed_bytes_fmt(2, 64, 256) == 0
    assert L.llama_q8_packed_bytes_fmt(q4_k, 64, 256) > 0
