"""Minimal GGUF writer for the tests (version 3 of the published GGUF layout):
"GGUF", u32 version, u64 tensor count, u64 key/value count, the key/values
(string key, u32 type, value; arrays as u32 element type + u64 count +
elements), the tensor directory (string name, u32 rank, u64 extents innermost
first, u32 element type, u64 offset into the data region), padding to the
alignment, then the data region. Test infrastructure only: it writes bytes
given to it and holds no model arithmetic."""
from __future__ import annotations

import struct

T_U32, T_I32, T_F32, T_BOOL, T_STRING, T_ARRAY, T_U64, T_F64 = 4, 5, 6, 7, 8, 9, 10, 12
TENSOR_F32, TENSOR_Q5_0, TENSOR_Q8_0 = 0, 6, 8


def _str(s: str) -> bytes:
    b = s.encode()
    return struct.pack("<Q", len(b)) + b


def _value(t: int, v) -> bytes:
    if t == T_U32:
        return struct.pack("<I", v)
    if t == T_I32:
        return struct.pack("<i", v)
    if t == T_U64:
        return struct.pack("<Q", v)
    if t == T_F32:
        return struct.pack("<f", v)
    if t == T_F64:
        return struct.pack("<d", v)
    if t == T_BOOL:
        return struct.pack("<B", 1 if v else 0)
    if t == T_STRING:
        return _str(v)
    if t == T_ARRAY:
        et, items = v
        return struct.pack("<IQ", et, len(items)) + b"".join(_value(et, x) for x in items)
    raise ValueError(t)


def header_bytes(kv, tensors, alignment: int = 32, version: int = 3, magic: bytes = b"GGUF"):
    """(header bytes incl. padding, data region bytes) for kv = [(key, type,
    value)] and tensors = [(name, type, dims innermost first, data bytes)]."""
    out = bytearray(magic + struct.pack("<IQQ", version, len(tensors), len(kv)))
    for key, t, v in kv:
        out += _str(key) + struct.pack("<I", t) + _value(t, v)
    data = bytearray()
    for name, t, dims, blob in tensors:
        pad = (-len(data)) % alignment
        data += b"\0" * pad
        out += _str(name) + struct.pack("<I", len(dims)) + b"".join(struct.pack("<Q", d) for d in dims)
        out += struct.pack("<IQ", t, len(data))
        data += blob
    out += b"\0" * ((-len(out)) % alignment)
    return bytes(out), bytes(data)


def write_gguf(path, kv, tensors, alignment: int = 32, version: int = 3, magic: bytes = b"GGUF") -> int:
    """Write the file; returns the offset where the data region starts."""
    head, data = header_bytes(kv, tensors, alignment, version, magic)
    with open(path, "wb") as f:
        f.write(head)
        f.write(data)
    return len(head)


def llama_kv(cfg: dict, arch: str = "llama", eps: bool = True, theta: bool = True, kv_heads: bool = True):
    """The llama.* metadata of a model config (the keys the pages' loader reads)."""
    kv = [("general.architecture", T_STRING, arch),
          ("llama.block_count", T_U32, cfg["n_layer"]),
          ("llama.embedding_length", T_U32, cfg["n_embd"]),
          ("llama.feed_forward_length", T_U32, cfg["n_ff"]),
          ("llama.attention.head_count", T_U32, cfg["n_head"])]
    if kv_heads:
        kv.append(("llama.attention.head_count_kv", T_U32, cfg["n_head_kv"]))
    if eps:
        kv.append(("llama.attention.layer_norm_rms_epsilon", T_F32, cfg.get("rms_eps", 1e-5)))
    if theta:
        kv.append(("llama.rope.freq_base", T_F32, cfg.get("rope_theta", 10000.0)))
    return kv


def model_tensors(cfg: dict, blobs: dict, untied: bool = False):
    """Directory entries for GGUF-named tensors: blobs maps names to uint8 Q8_0
    arrays [rows, k/32*34] or f32 vectors; extents are (k, rows) / (n,)."""
    out = []
    for name, b in blobs.items():
        if name == "output.weight" and not untied:
            continue
        if b.dtype.kind == "u":
            rows, rb = b.shape
            out.append((name, TENSOR_Q8_0, (rb // 34 * 32, rows), b.tobytes()))
        else:
            out.append((name, TENSOR_F32, (b.shape[0],), b.astype("<f4").tobytes()))
    return out
