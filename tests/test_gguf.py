"""GGUF loading ("量化 llama 的一次前向", from_gguf：键名写死了 llama.;
"生成一个 token", 读 GGUF / 建模型：按名字取张量): files written by the test
writer from the published GGUF layout.

- The 135M tensor set (272 tensors, no output.weight) has a data region of
  exactly the size the pages print (file 144,811,360 bytes, tensor data from
  1,785,952: 143,025,408 bytes), and the reader finds the 135M hyperparameters
  and the tied head in it.
- Keys and defaults, the rotary convention by architecture, alignment, and
  the errors (bad magic or version, truncation, a missing key or tensor, a
  wrong extent, a non-Q8_0 matrix) without a GPU.
- On the GPU, a model loaded from a file gives the same logits, bit for bit,
  as the same tensors passed as arrays, and the oracle's tokens.
"""
import numpy as np
import pytest

from q8_quantized_llama_gb300 import synth
from tests import gguf_writer as G

PAGE_FILE_BYTES = 144_811_360
PAGE_DATA_OFFSET = 1_785_952


@pytest.fixture(scope="module")
def B():
    from q8_quantized_llama_gb300 import binding
    binding.lib()
    return binding


def zero_blobs(cfg):
    out = {}
    for name, shape, kind in synth.model_tensor_specs(cfg):
        if kind == "matrix":
            out[name] = np.zeros((shape[0], shape[1] // 32 * 34), np.uint8)
        else:
            out[name] = np.zeros(shape[0], np.float32)
    return out


TINY = dict(synth.MODEL_135M, n_layer=2, n_vocab=320)


def test_135m_tensor_set_matches_page_byte_counts(B, tmp_path):
    cfg = dict(synth.MODEL_135M)
    blobs = zero_blobs(cfg)
    tensors = G.model_tensors(cfg, blobs)
    assert len(tensors) == 272                      # 30 layers x 9 + token_embd + output_norm
    path = tmp_path / "m135.gguf"
    data_offset = G.write_gguf(path, G.llama_kv(cfg), tensors)
    region = path.stat().st_size - data_offset
    assert region == PAGE_FILE_BYTES - PAGE_DATA_OFFSET
    got, n, off = B.gguf_config(str(path))
    assert (n, off) == (272, data_offset)
    for key in ("n_layer", "n_embd", "n_head", "n_head_kv", "head_dim", "n_ff", "n_vocab", "max_seq"):
        assert got[key] == cfg[key], key
    assert got["tied_output"] == 1 and got["rope_style"] == 0 and got["decode_kernel"] == 0
    assert abs(got["rms_eps"] - 1e-5) < 1e-12 and got["rope_theta"] == 10000.0


def _tiny_file(path, arch="llama", untied=False, kv=None, alignment=32, drop=(), retype=None, reshape=None,
               cfg=TINY):
    blobs = zero_blobs(dict(cfg, tied_output=0))
    tensors = [t for t in G.model_tensors(cfg, blobs, untied=untied) if t[0] not in drop]
    if retype:
        tensors = [(n, retype[1] if n == retype[0] else t, d, b) for n, t, d, b in tensors]
    if reshape:
        tensors = [(n, t, reshape[1] if n == reshape[0] else d, b) for n, t, d, b in tensors]
    return G.write_gguf(path, kv if kv is not None else G.llama_kv(TINY, arch), tensors, alignment)


def test_keys_defaults_tied_head_and_architecture(B, tmp_path):
    p = tmp_path / "a.gguf"
    mha = dict(TINY, n_head_kv=TINY["n_head"])
    _tiny_file(p, kv=G.llama_kv(mha, eps=False, theta=False, kv_heads=False), cfg=mha)
    cfg = B.gguf_config(str(p))[0]
    assert cfg["rms_eps"] == np.float32(1e-5) and cfg["rope_theta"] == 10000.0
    assert cfg["n_head_kv"] == cfg["n_head"]        # head_count_kv absent: plain multi-head
    assert cfg["tied_output"] == 1 and cfg["n_vocab"] == TINY["n_vocab"]
    # the same file with the GQA tensors but no head_count_kv key: K/V extents do not match
    p1 = tmp_path / "a1.gguf"
    _tiny_file(p1, kv=G.llama_kv(TINY, kv_heads=False))
    assert B.gguf_config_status(str(p1))[0] == B.LQ8_ERR_FORMAT
    p2 = tmp_path / "b.gguf"
    _tiny_file(p2, arch="qwen2", untied=True, kv=G.llama_kv(dict(TINY, rms_eps=1e-6, rope_theta=5e5), "qwen2"))
    cfg = B.gguf_config(str(p2))[0]
    assert cfg["tied_output"] == 0 and cfg["rope_style"] == 1
    assert cfg["rms_eps"] == np.float32(1e-6) and cfg["rope_theta"] == 5e5
    assert cfg["n_head_kv"] == TINY["n_head_kv"] and cfg["head_dim"] == 64


def test_alignment_key(B, tmp_path):
    p = tmp_path / "c.gguf"
    off = _tiny_file(p, kv=G.llama_kv(TINY) + [("general.alignment", G.T_U32, 256)], alignment=256)
    cfg, n, got_off = B.gguf_config(str(p))
    assert got_off == off and off % 256 == 0 and n == 2 * 9 + 2


def test_bad_alignment_and_integer_keys_are_rejected(B, tmp_path):
    """general.alignment must be an integer power of two up to 64 KiB, and the
    integer hyperparameters finite integers within +-2^53; anything else is a
    format error, never an undefined conversion or a wrapped data offset."""
    def status(kv):
        p = tmp_path / "al.gguf"
        _tiny_file(p, kv=kv)
        return B.gguf_config_status(str(p))[0]

    base = G.llama_kv(TINY)
    for bad in ((G.T_U32, 0), (G.T_U32, 48), (G.T_U32, 1 << 17), (G.T_U64, 2**64 - 1),
                (G.T_F32, 32.5), (G.T_F32, float("inf")), (G.T_F32, float("nan")), (G.T_F64, 2.0**63)):
        assert status(base + [("general.alignment", bad[0], bad[1])]) == B.LQ8_ERR_FORMAT, bad
    assert status(base + [("general.alignment", G.T_STRING, "32")]) == B.LQ8_ERR_FORMAT

    def with_key(key, t, v):
        return [x for x in base if x[0] != key] + [(key, t, v)]

    for key in ("llama.block_count", "llama.embedding_length", "llama.attention.head_count_kv"):
        for t, v in ((G.T_F32, float("nan")), (G.T_F32, float("inf")), (G.T_F32, 2.5), (G.T_F64, 1e300),
                     (G.T_F64, -1e300)):
            assert status(with_key(key, t, v)) == B.LQ8_ERR_FORMAT, (key, t, v)
    # an integral value given as a float is still an integer
    assert status(with_key("llama.block_count", G.T_F32, 2.0)) == B.LQ8_OK


def test_extra_metadata_arrays_are_skipped(B, tmp_path):
    kv = G.llama_kv(TINY) + [("tokenizer.ggml.tokens", G.T_ARRAY, (G.T_STRING, ["a", "bb", "<s>"] * 50)),
                             ("tokenizer.ggml.token_type", G.T_ARRAY, (G.T_I32, list(range(150)))),
                             ("general.name", G.T_STRING, "synthetic")]
    p = tmp_path / "d.gguf"
    _tiny_file(p, kv=kv)
    assert B.gguf_config(str(p))[0]["n_layer"] == 2


def test_errors(B, tmp_path):
    def status(**kw):
        p = tmp_path / "e.gguf"
        _tiny_file(p, **kw)
        return B.gguf_config_status(str(p))[0]

    assert B.gguf_config_status(str(tmp_path / "missing.gguf"))[0] == B.LQ8_ERR_FORMAT
    kv = [x for x in G.llama_kv(TINY) if x[0] != "llama.block_count"]
    assert status(kv=kv) == B.LQ8_ERR_FORMAT                     # "cannot find ... in metadata"
    assert status(drop=("blk.1.ffn_up.weight",)) == B.LQ8_ERR_FORMAT
    assert status(drop=("token_embd.weight",)) == B.LQ8_ERR_FORMAT
    assert status(retype=("blk.0.attn_q.weight", G.TENSOR_Q5_0)) == B.LQ8_ERR_UNSUPPORTED
    assert status(retype=("blk.0.attn_norm.weight", G.TENSOR_Q8_0)) == B.LQ8_ERR_UNSUPPORTED
    assert status(reshape=("blk.0.attn_k.weight", (576, 128))) == B.LQ8_ERR_FORMAT
    # bad magic, unknown version, a file cut inside the tensor data
    p = tmp_path / "f.gguf"
    _tiny_file(p)
    raw = p.read_bytes()
    for bad in (b"GGUX" + raw[4:], raw[:4] + (1).to_bytes(4, "little") + raw[8:], raw[:-100]):
        p.write_bytes(bad)
        assert B.gguf_config_status(str(p))[0] == B.LQ8_ERR_FORMAT
    p.write_bytes(raw[:200])                                     # cut inside the key/values
    assert B.gguf_config_status(str(p))[0] == B.LQ8_ERR_FORMAT


def test_truncated_and_corrupted_files_fail_cleanly(B, tmp_path):
    """Every truncation of a small file and seeded byte corruptions of its
    header give a status (never a crash or an out-of-file read); a corrupted
    tensor offset near 2^64 is rejected rather than wrapping the bounds check."""
    p = tmp_path / "g.gguf"
    off = _tiny_file(p)
    raw = p.read_bytes()
    ok = B.gguf_config_status(str(p))[0]
    assert ok == B.LQ8_OK
    for cut in list(range(0, off, 97)) + [off - 1, off + 1, len(raw) - 1]:
        p.write_bytes(raw[:cut])
        assert B.gguf_config_status(str(p))[0] in (B.LQ8_ERR_FORMAT, B.LQ8_ERR_UNSUPPORTED), cut
    rng = np.random.default_rng(12)
    for _ in range(200):
        bad = bytearray(raw)
        for _ in range(int(rng.integers(1, 4))):
            i = int(rng.integers(4, off))
            bad[i] = int(rng.integers(0, 256))
        p.write_bytes(bytes(bad))
        assert B.gguf_config_status(str(p))[0] in (B.LQ8_OK, B.LQ8_ERR_FORMAT, B.LQ8_ERR_UNSUPPORTED)
    # the last tensor's offset field (the 8 bytes before the header padding) set near 2^64
    tensors = G.model_tensors(TINY, zero_blobs(dict(TINY, tied_output=0)))
    huge = bytearray(raw)
    name = tensors[-1][0].encode()
    pos = raw.rfind(name)
    assert pos > 0
    rank_at = pos + len(name)
    rank = int.from_bytes(raw[rank_at:rank_at + 4], "little")
    off_at = rank_at + 4 + 8 * rank + 4
    huge[off_at:off_at + 8] = (2**64 - 64).to_bytes(8, "little")
    p.write_bytes(bytes(huge))
    assert B.gguf_config_status(str(p))[0] == B.LQ8_ERR_FORMAT


@pytest.mark.gpu
def test_model_from_file_equals_model_from_arrays(B, tmp_path):
    from oracle import q8_oracle as O
    from tests.gpu_helpers import logits_close, oracle_model_tensors, require_gpu
    require_gpu()
    cfg = dict(synth.MODEL_135M, n_layer=3)
    host = synth.model_weights_f32(cfg, 21)
    ora_t = oracle_model_tensors(cfg, 21, host)
    path = tmp_path / "m.gguf"
    G.write_gguf(path, G.llama_kv(cfg), G.model_tensors(cfg, ora_t))
    from_file = B.Model.from_gguf(str(path))
    from_arrays = B.Model(cfg, ora_t)
    try:
        assert from_file.cfg["n_layer"] == 3 and from_file.cfg["tied_output"] == 1
        prompt = synth.prompt_ids(21, cfg["n_vocab"], 8)
        a = from_file.forward(prompt, 0)
        b = from_arrays.forward(prompt, 0)
        np.testing.assert_array_equal(a, b)
        oracle = O.ModelWeights(cfg, ora_t)
        ids, logits = oracle.generate(prompt, 4)
        ok, err, bound = logits_close(a, logits[0])
        assert ok, (err, bound)
        np.testing.assert_array_equal(from_file.generate(prompt, 4), ids)
    finally:
        from_file.close()
        from_arrays.close()
