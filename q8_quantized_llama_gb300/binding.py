"""ctypes binding to libllama_q8.so (declared in include/llama_q8.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels. Functions keep the C names; ``Model`` is a small owner of a
``llama_q8_ctx``. Arrays can be numpy arrays (host memory) or objects with a
``data_ptr()`` method such as torch CUDA tensors (device memory).

If the library has not been built, importing this module raises: there is no
fallback path.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libllama_q8.so")

STATUS = {0: "LQ8_OK", 1: "LQ8_ERR_ARG", 2: "LQ8_ERR_POS", 3: "LQ8_ERR_CTX", 4: "LQ8_ERR_TOKEN",
          5: "LQ8_ERR_CUDA", 6: "LQ8_ERR_OOM", 7: "LQ8_ERR_STATE", 8: "LQ8_ERR_UNSUPPORTED"}
LQ8_OK, LQ8_ERR_ARG, LQ8_ERR_POS, LQ8_ERR_CTX, LQ8_ERR_TOKEN = 0, 1, 2, 3, 4
LQ8_ERR_CUDA, LQ8_ERR_OOM, LQ8_ERR_STATE, LQ8_ERR_UNSUPPORTED, LQ8_ERR_FORMAT = 5, 6, 7, 8, 9

# Every symbol include/llama_q8.h declares.
EXPORTS = ("llama_q8_load", "llama_q8_forward", "llama_q8_forward_argmax", "llama_q8_generate",
           "llama_q8_prefill_async", "llama_q8_decode_async", "llama_q8_sync", "llama_q8_reset",
           "llama_q8_free", "llama_q8_cache_len", "llama_q8_read_kv", "llama_q8_stream",
           "llama_q8_decode_kernel_count", "llama_q8_status_str", "llama_q8_quantize",
           "llama_q8_packed_bytes", "llama_q8_pack", "llama_q8_matmul", "llama_q8_matmul_ex",
           "llama_q8_attention_workspace_bytes", "llama_q8_attention", "llama_q8_launch_count",
           "llama_q8_profile_decode", "llama_q8_attention_decode_noalloc", "llama_q8_attention_decode",
           "llama_q8_selftest_wait_timeout", "llama_q8_rope_style_for_arch", "llama_q8_gguf_config",
           "llama_q8_load_gguf", "llama_q8_packed_bytes_fmt", "llama_q8_pack_fmt", "llama_q8_matvec_fmt")
GGUF_Q5_0, GGUF_Q8_0, GGUF_Q4_K, GGUF_Q6_K = 6, 8, 12, 14


class Q8Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class llama_q8_kernel_stat(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("launches", C.c_int32), ("ms", C.c_double), ("span_ms", C.c_double),
                ("bytes", C.c_double)]


class llama_q8_config(C.Structure):
    _fields_ = [("n_layer", C.c_int32), ("n_embd", C.c_int32), ("n_head", C.c_int32),
                ("n_head_kv", C.c_int32), ("head_dim", C.c_int32), ("n_ff", C.c_int32),
                ("n_vocab", C.c_int32), ("max_seq", C.c_int32), ("rms_eps", C.c_float),
                ("rope_theta", C.c_float), ("tied_output", C.c_int32), ("decode_kernel", C.c_int32),
                ("rope_style", C.c_int32), ("head_splits", C.c_int32)]


class llama_q8_layer_weights(C.Structure):
    _fields_ = [("attn_norm", C.c_void_p), ("ffn_norm", C.c_void_p), ("attn_q", C.c_void_p),
                ("attn_k", C.c_void_p), ("attn_v", C.c_void_p), ("attn_output", C.c_void_p),
                ("ffn_gate", C.c_void_p), ("ffn_up", C.c_void_p), ("ffn_down", C.c_void_p)]


class llama_q8_weights(C.Structure):
    _fields_ = [("token_embd", C.c_void_p), ("output_norm", C.c_void_p), ("output", C.c_void_p),
                ("layers", C.POINTER(llama_q8_layer_weights)), ("on_device", C.c_int32)]


_lib = None


def lib() -> C.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with q8_quantized_llama_gb300.build.build()")
    L = C.CDLL(LIB_PATH)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    sig = {
        "llama_q8_load": (i32, [C.POINTER(llama_q8_config), C.POINTER(llama_q8_weights), i32, C.POINTER(vp)]),
        "llama_q8_forward": (i32, [vp, vp, i32, i32, vp]),
        "llama_q8_forward_argmax": (i32, [vp, vp, i32, i32, vp]),
        "llama_q8_generate": (i32, [vp, vp, i32, i32, vp]),
        "llama_q8_prefill_async": (i32, [vp, vp, i32, i32, vp]),
        "llama_q8_decode_async": (i32, [vp, i32, vp]),
        "llama_q8_sync": (i32, [vp]),
        "llama_q8_reset": (i32, [vp]),
        "llama_q8_free": (i32, [vp]),
        "llama_q8_cache_len": (i32, [vp, C.POINTER(i32)]),
        "llama_q8_read_kv": (i32, [vp, i32, i32, i32, vp, vp]),
        "llama_q8_stream": (vp, [vp]),
        "llama_q8_decode_kernel_count": (i32, [vp]),
        "llama_q8_status_str": (C.c_char_p, [i32]),
        "llama_q8_rope_style_for_arch": (i32, [C.c_char_p]),
        "llama_q8_gguf_config": (i32, [C.c_char_p, vp, vp, vp]),
        "llama_q8_load_gguf": (i32, [C.c_char_p, i32, i32, vp]),
        "llama_q8_quantize": (i32, [vp, i64, i64, vp, vp]),
        "llama_q8_packed_bytes": (sz, [i64, i64]),
        "llama_q8_pack": (i32, [vp, i64, i64, vp, vp]),
        "llama_q8_matmul": (i32, [vp, i64, i64, vp, i64, vp, vp]),
        "llama_q8_matmul_ex": (i32, [vp, i64, i64, vp, i64, vp, i32, vp]),
        "llama_q8_attention_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "llama_q8_attention": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, sz, vp]),
        "llama_q8_launch_count": (i64, [vp]),
        "llama_q8_attention_decode_noalloc": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]),
        "llama_q8_attention_decode": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp]),
        "llama_q8_profile_decode": (i32, [vp, i32, C.POINTER(llama_q8_kernel_stat), i32, C.POINTER(i32)]),
        "llama_q8_selftest_wait_timeout": (i32, [C.POINTER(i32)]),
        "llama_q8_packed_bytes_fmt": (sz, [i32, i64, i64]),
        "llama_q8_pack_fmt": (i32, [i32, vp, i64, i64, vp, vp]),
        "llama_q8_matvec_fmt": (i32, [i32, vp, i64, i64, vp, vp, i32, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def ptr(a) -> int | None:
    """Address of a numpy array or of an object with data_ptr() (None for None)."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        return int(a.data_ptr())
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return int(a.ctypes.data)
    if isinstance(a, int):
        return a
    raise TypeError(f"cannot take the address of {type(a)}")


def check(status: int, where: str) -> None:
    if status != LQ8_OK:
        raise Q8Error(status, where)


def rope_style_for_arch(arch: str | None) -> int:
    """0 (rope_i) or 1 (NEOX) for a general.architecture name; -1 for None."""
    return int(lib().llama_q8_rope_style_for_arch(None if arch is None else arch.encode()))


def gguf_config_status(path: str):
    """(status, config dict or None, tensor count, data offset) of llama_q8_gguf_config."""
    c = llama_q8_config()
    n = C.c_int64(0)
    off = C.c_int64(0)
    st = lib().llama_q8_gguf_config(path.encode(), C.byref(c), C.byref(n), C.byref(off))
    cfg = {f: getattr(c, f) for f, _ in llama_q8_config._fields_} if st == LQ8_OK else None
    return st, cfg, n.value, off.value


def gguf_config(path: str):
    """(config dict, tensor count, data offset) of a GGUF file; raises Q8Error."""
    st, cfg, n, off = gguf_config_status(path)
    check(st, "llama_q8_gguf_config")
    return cfg, n, off


def make_config(cfg: dict) -> llama_q8_config:
    return llama_q8_config(cfg["n_layer"], cfg["n_embd"], cfg["n_head"], cfg["n_head_kv"], cfg["head_dim"],
                           cfg["n_ff"], cfg["n_vocab"], cfg.get("max_seq", 4096), cfg.get("rms_eps", 1e-5),
                           cfg.get("rope_theta", 10000.0), int(cfg.get("tied_output", 1)),
                           int(cfg.get("decode_kernel", 0)), int(cfg.get("rope_style", 0)),
                           int(cfg.get("head_splits", 0)))


_LAYER_KEYS = ("attn_norm", "ffn_norm", "attn_q", "attn_k", "attn_v", "attn_output", "ffn_gate", "ffn_up",
               "ffn_down")


def make_weights(cfg: dict, tensors: dict, on_device: bool):
    """Build the llama_q8_weights struct from GGUF-named tensors (Q8_0 blobs
    for matrices, f32 vectors for norms). Returns (struct, keep-alive list)."""
    layers = (llama_q8_layer_weights * cfg["n_layer"])()
    for i in range(cfg["n_layer"]):
        for k in _LAYER_KEYS:
            setattr(layers[i], k, ptr(tensors[f"blk.{i}.{k}.weight"]))
    w = llama_q8_weights(ptr(tensors["token_embd.weight"]), ptr(tensors["output_norm.weight"]),
                         ptr(tensors.get("output.weight")), layers, 1 if on_device else 0)
    return w, [layers]


class Model:
    """Owner of a llama_q8_ctx; methods map one-to-one onto the C calls."""

    def __init__(self, cfg: dict, tensors: dict, device: int = 0, on_device: bool = False):
        L = lib()
        self.cfg = dict(cfg)
        c = make_config(cfg)
        w, keep = make_weights(cfg, tensors, on_device)
        out = C.c_void_p()
        check(L.llama_q8_load(C.byref(c), C.byref(w), device, C.byref(out)), "llama_q8_load")
        self.ctx = out
        del keep

    @classmethod
    def from_gguf(cls, path: str, device: int = 0, decode_kernel: int = 0) -> "Model":
        """llama_q8_load_gguf: the model of a GGUF file (config from its llama.* keys)."""
        cfg = gguf_config(path)[0]
        out = C.c_void_p()
        check(lib().llama_q8_load_gguf(path.encode(), device, decode_kernel, C.byref(out)), "llama_q8_load_gguf")
        self = cls.__new__(cls)
        self.cfg = dict(cfg, decode_kernel=decode_kernel)
        self.ctx = out
        return self

    def close(self):
        if getattr(self, "ctx", None):
            lib().llama_q8_free(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, ids, index_pos: int) -> np.ndarray:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        logits = np.empty(self.cfg["n_vocab"], dtype=np.float32)
        check(lib().llama_q8_forward(self.ctx, ptr(ids), ids.size, index_pos, ptr(logits)), "llama_q8_forward")
        return logits

    def forward_status(self, ids, index_pos: int) -> int:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        logits = np.empty(self.cfg["n_vocab"], dtype=np.float32)
        return lib().llama_q8_forward(self.ctx, ptr(ids) if ids.size else ptr(np.zeros(1, np.int32)),
                                      ids.size, index_pos, ptr(logits))

    def forward_argmax(self, ids, index_pos: int) -> int:
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        nxt = np.zeros(1, dtype=np.int32)
        check(lib().llama_q8_forward_argmax(self.ctx, ptr(ids), ids.size, index_pos, ptr(nxt)),
              "llama_q8_forward_argmax")
        return int(nxt[0])

    def generate(self, prompt, n_decode: int) -> np.ndarray:
        prompt = np.ascontiguousarray(prompt, dtype=np.int32)
        out = np.empty(n_decode + 1, dtype=np.int32)
        check(lib().llama_q8_generate(self.ctx, ptr(prompt), prompt.size, n_decode, ptr(out)), "llama_q8_generate")
        return out

    def prefill_async(self, d_ids, T: int, index_pos: int, d_next) -> None:
        check(lib().llama_q8_prefill_async(self.ctx, ptr(d_ids), T, index_pos, ptr(d_next)), "llama_q8_prefill_async")

    def decode_async(self, n_steps: int, d_out) -> None:
        check(lib().llama_q8_decode_async(self.ctx, n_steps, ptr(d_out)), "llama_q8_decode_async")

    def sync(self) -> None:
        check(lib().llama_q8_sync(self.ctx), "llama_q8_sync")

    def reset(self) -> None:
        check(lib().llama_q8_reset(self.ctx), "llama_q8_reset")

    def cache_len(self) -> int:
        n = C.c_int32()
        check(lib().llama_q8_cache_len(self.ctx, C.byref(n)), "llama_q8_cache_len")
        return n.value

    def read_kv(self, layer: int, pos0: int, n: int):
        kvh, hd = self.cfg["n_head_kv"], self.cfg["head_dim"]
        k = np.empty((kvh, n, hd), np.float32)
        v = np.empty((kvh, n, hd), np.float32)
        check(lib().llama_q8_read_kv(self.ctx, layer, pos0, n, ptr(k), ptr(v)), "llama_q8_read_kv")
        return k, v

    def stream(self) -> int:
        return lib().llama_q8_stream(self.ctx) or 0

    def decode_kernel_count(self) -> int:
        return lib().llama_q8_decode_kernel_count(self.ctx)

    def launch_count(self) -> int:
        return int(lib().llama_q8_launch_count(self.ctx))

    def profile_decode(self, n_steps: int):
        """Per-kernel-family timeline of n_steps decode steps of the instrumented
        graph: {name: (launches, exclusive ms, span ms, bytes)}."""
        stats = (llama_q8_kernel_stat * 16)()
        n = C.c_int32()
        check(lib().llama_q8_profile_decode(self.ctx, n_steps, stats, 16, C.byref(n)), "llama_q8_profile_decode")
        return {stats[i].name.decode(): (stats[i].launches, stats[i].ms, stats[i].span_ms, stats[i].bytes)
                for i in range(n.value)}


# ---- device-level entry points ------------------------------------------------

def llama_q8_quantize(w, rows: int, k: int, out, stream=0) -> None:
    check(lib().llama_q8_quantize(ptr(w), rows, k, ptr(out), stream or None), "llama_q8_quantize")


def llama_q8_packed_bytes(rows: int, k: int) -> int:
    return int(lib().llama_q8_packed_bytes(rows, k))


def llama_q8_pack(q8, rows: int, k: int, packed, stream=0) -> None:
    check(lib().llama_q8_pack(ptr(q8), rows, k, ptr(packed), stream or None), "llama_q8_pack")


def llama_q8_matmul(packed, rows: int, k: int, x, m: int, y, stream=0) -> None:
    check(lib().llama_q8_matmul(ptr(packed), rows, k, ptr(x), m, ptr(y), stream or None), "llama_q8_matmul")


LQ8_MATMUL_EARLY_WEIGHTS = 1
LQ8_MATMUL_TENSOR_CORES = 2
LQ8_MATMUL_CUDA_CORES = 4


def llama_q8_selftest_wait_timeout() -> int:
    """Code recorded by a kernel whose bounded wait ran out (see the header)."""
    code = C.c_int32(0)
    check(lib().llama_q8_selftest_wait_timeout(C.byref(code)), "llama_q8_selftest_wait_timeout")
    return int(code.value)


def llama_q8_matmul_ex(packed, rows: int, k: int, x, m: int, y, flags: int, stream=0) -> None:
    check(lib().llama_q8_matmul_ex(ptr(packed), rows, k, ptr(x), m, ptr(y), flags, stream or None),
          "llama_q8_matmul_ex")


def llama_q8_packed_bytes_fmt(gguf_type: int, rows: int, k: int) -> int:
    return int(lib().llama_q8_packed_bytes_fmt(gguf_type, rows, k))


def llama_q8_pack_fmt(gguf_type: int, blocks, rows: int, k: int, packed, stream=0) -> None:
    check(lib().llama_q8_pack_fmt(gguf_type, ptr(blocks), rows, k, ptr(packed), stream or None), "llama_q8_pack_fmt")


def llama_q8_matvec_fmt(gguf_type: int, packed, rows: int, k: int, x, y, flags: int = 0, stream=0) -> None:
    check(lib().llama_q8_matvec_fmt(gguf_type, ptr(packed), rows, k, ptr(x), ptr(y), flags, stream or None),
          "llama_q8_matvec_fmt")


def llama_q8_attention_workspace_bytes(n_head: int, n_head_kv: int, head_dim: int, cache_stride: int) -> int:
    return int(lib().llama_q8_attention_workspace_bytes(n_head, n_head_kv, head_dim, cache_stride))


def llama_q8_attention(q, k_cache, v_cache, T: int, index_pos: int, n_head: int, n_head_kv: int, head_dim: int,
                       cache_stride: int, out, workspace, workspace_bytes: int, stream=0) -> None:
    check(lib().llama_q8_attention(ptr(q), ptr(k_cache), ptr(v_cache), T, index_pos, n_head, n_head_kv, head_dim,
                                   cache_stride, ptr(out), ptr(workspace), workspace_bytes, stream or None),
          "llama_q8_attention")


def llama_q8_attention_decode(q, k_cache, v_cache, kv_len: int, n_head: int, n_head_kv: int, head_dim: int,
                              cache_stride: int, out, stream=0) -> None:
    """Single-token attention with the decode step's cluster kernel."""
    check(lib().llama_q8_attention_decode(ptr(q), ptr(k_cache), ptr(v_cache), kv_len, n_head, n_head_kv, head_dim,
                                          cache_stride, ptr(out), stream or None), "llama_q8_attention_decode")


def llama_q8_attention_decode_noalloc(q, k_cache, v_cache, kv_len: int, n_head: int, n_head_kv: int,
                                      head_dim: int, cache_stride: int, out, stream=0) -> None:
    """Single-token attention with the library's fixed scratch array (no allocation)."""
    check(lib().llama_q8_attention_decode_noalloc(ptr(q), ptr(k_cache), ptr(v_cache), kv_len, n_head, n_head_kv,
                                                  head_dim, cache_stride, ptr(out), stream or None),
          "llama_q8_attention_decode_noalloc")


def status_str(s: int) -> str:
    return lib().llama_q8_status_str(s).decode()
