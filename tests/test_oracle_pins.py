"""Pins for the CPU oracle: every check here compares the oracle with something
other than itself — numbers printed on the candle pages, hand-worked fixtures
under tests/golden/, closed forms, or invariants the pages state."""
import math

import numpy as np
import pytest

from oracle import q8_oracle as O
from q8_quantized_llama_gb300 import synth
from tests.conftest import golden_path

TINY = dict(n_layer=2, n_embd=288, n_head=9, n_head_kv=3, head_dim=32, n_ff=96,
            n_vocab=160, max_seq=4096, rms_eps=1e-5, rope_theta=10000.0, tied_output=1)


def _read_kv(name):
    out = {}
    for line in open(golden_path(name)):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split()[:2]
            out[k] = float(v)
    return out


def quantized_tensors(cfg, seed):
    t = {}
    for name, w, kind in synth.iter_model_weights_f32(cfg, seed):
        t[name] = O.quantize_q8_0(w) if kind == "matrix" else w
    return t


@pytest.fixture(scope="module")
def tiny_tensors():
    return quantized_tensors(TINY, 7)


# ---------------------------------------------------------------- Q8_0 format

def test_q8_0_layout_matches_page_byte_counts():
    """34 bytes per 32 weights + f32 norms reproduce the GGUF data region exactly."""
    pc = _read_kv("pages_counts.txt")
    cfg = synth.MODEL_135M
    specs = synth.model_tensor_specs(cfg)
    assert len(specs) == pc["gguf_tensor_count"]
    q8 = sum(r * O.q8_0_row_bytes(k) for _, (r, k), kind in
             [(n, s, kd) for n, s, kd in specs if kd == "matrix"])
    norms = sum(s[0] * 4 for _, s, kd in specs if kd == "norm")
    assert q8 + norms == pc["gguf_file_bytes"] - pc["gguf_data_offset"]
    assert round(q8 / 2**20, 1) == pc["q8_weights_mib"]
    n_w = sum(int(np.prod(s)) for _, s, _ in specs)
    assert round(n_w * 4 / 2**20) == pc["f32_weights_mib"]
    # the quantiser's own output has that row size
    assert O.quantize_q8_0(np.ones((3, 576), np.float32)).shape == (3, 612)


def _hand_blocks():
    cases, cur = [], {}
    for line in open(golden_path("q8_0_hand_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rest = line.split(None, 1)
        if key == "case":
            cur = {"name": rest}
            cases.append(cur)
        elif key == "w":
            cur["w"] = np.array([float(v) for v in rest.split()], np.float32)
        elif key == "bytes":
            cur["bytes"] = np.array([int(v, 16) for v in rest.split()], np.uint8)
    return cases


@pytest.mark.parametrize("case", _hand_blocks(), ids=lambda c: c["name"])
def test_q8_0_hand_blocks(case):
    out = O.quantize_q8_0(case["w"][None, :])
    assert out.shape == (1, 34)
    np.testing.assert_array_equal(out[0], case["bytes"])


def test_q8_0_hand_blocks_dequantise():
    cases = {c["name"]: c for c in _hand_blocks()}
    w = O.dequantize_q8_0(cases["A"]["bytes"][None, :], 1, 32)[0]
    expect = [127, 3, -3, 1, -1, 2, -2, 64, -127] + [0] * 23
    np.testing.assert_array_equal(w, np.array(expect, np.float32))
    w = O.dequantize_q8_0(cases["C"]["bytes"][None, :], 1, 32)[0]
    d = 0.00787353515625
    np.testing.assert_array_equal(w[:5], np.array([127 * d, -64 * d, 32 * d, 95 * d, -16 * d], np.float32))


def test_q8_0_round_trip_bound_and_extremes():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((64, 256)) * rng.uniform(1e-3, 10, (64, 1))).astype(np.float32)
    w[3, 32:64] = 0.0                       # an all-zero block
    blob = O.quantize_q8_0(w)
    dh, q = O.q8_0_scales_and_codes(blob, 64, 256)
    deq = O.dequantize_q8_0(blob, 64, 256).reshape(64, 8, 32)
    wb = w.reshape(64, 8, 32).astype(np.float64)
    d = (np.max(np.abs(w.reshape(64, 8, 32)), axis=2) / np.float32(127)).astype(np.float64)
    bound = d / 2 + 127 * np.abs(d - dh.astype(np.float64)) + 1e-6 * d
    assert np.all(np.abs(wb - deq) <= bound[..., None])
    qb = q.reshape(64, 8, 32).astype(np.int64)
    am = np.argmax(np.abs(wb), axis=2)
    for r in range(64):
        for b in range(8):
            if d[r, b] > 0:
                assert abs(qb[r, b, am[r, b]]) == 127
    assert np.all(qb[3, 1] == 0) and dh[3, 1] == 0
    assert qb.max() <= 127 and qb.min() >= -127


# ---------------------------------------------------------------- small ops

def test_rms_norm_closed_form():
    y = O.rms_norm(np.array([[3.0, 4.0]], np.float32), np.array([2.0, 0.5], np.float32), 0.0)
    r = math.sqrt(12.5)
    np.testing.assert_allclose(y[0], [2 * 3 / r, 0.5 * 4 / r], rtol=1e-7)
    y = O.rms_norm(np.zeros((1, 8), np.float32), np.ones(8, np.float32), 1e-5)
    assert np.all(y == 0)
    # eps sits inside the square root: x = [1] -> 1 / sqrt(1 + eps)
    y = O.rms_norm(np.array([[1.0]], np.float32), np.array([1.0], np.float32), 0.25)
    np.testing.assert_allclose(y[0, 0], 1 / math.sqrt(1.25), rtol=1e-7)


def test_silu_closed_form():
    np.testing.assert_allclose(O.silu(np.array([0.0, math.log(3.0), -math.log(3.0)])),
                               [0.0, 0.75 * math.log(3.0), -0.25 * math.log(3.0)], rtol=1e-15)


def _rope_fixture():
    f = {}
    for line in open(golden_path("rope_hand_example.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, *v = line.split()
            f[k] = [float(t) for t in v]
    return f


def test_rope_pairing_hand_example():
    f = _rope_fixture()
    x = np.array(f["x"], np.float32).reshape(1, 1, 4)
    pos = np.array([int(f["position"][0])])
    np.testing.assert_allclose(O.rope_i(x, pos, f["theta"][0])[0, 0], f["rope_i"], rtol=1e-6)
    np.testing.assert_allclose(O.rope_neox(x, pos, f["theta"][0])[0, 0], f["neox"], rtol=1e-6)


def test_rope_position_zero_and_relative_invariance():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((1, 2, 64)).astype(np.float32)
    np.testing.assert_array_equal(O.rope_i(x, np.array([0]), 1e4), x)
    q = rng.standard_normal((1, 1, 64)).astype(np.float32)
    k = rng.standard_normal((1, 1, 64)).astype(np.float32)
    dots = []
    for m, n in [(5, 2), (103, 100), (4000, 3997)]:
        a = O.rope_i(q, np.array([m]), 1e4).astype(np.float64)
        b = O.rope_i(k, np.array([n]), 1e4).astype(np.float64)
        dots.append(float(np.sum(a * b)))
    np.testing.assert_allclose(dots, dots[0], rtol=2e-5)
    # norms are preserved by the rotation
    r = O.rope_i(q, np.array([777]), 1e4)
    np.testing.assert_allclose(np.linalg.norm(r), np.linalg.norm(q), rtol=1e-6)


def test_rope_table_shape_and_limit(tiny_tensors):
    pc = _read_kv("pages_counts.txt")
    c, s = O.rope_table(64, 1e4)
    assert c.shape == s.shape == (pc["rope_table_rows"], pc["rope_table_cols"])
    model = O.ModelWeights(TINY, tiny_tensors)
    with pytest.raises(ValueError, match="start: 4096"):
        model.forward([1], 4096)
    model.forward([1], 4095)       # the last row of the table is usable


def test_causal_mask_shape_and_prefix():
    m = O.build_causal_mask(5, 5)
    assert m.shape == (5, 10)
    assert np.all(m[:, :5] == 0)
    np.testing.assert_array_equal(m[:, 5:], np.triu(np.ones((5, 5), np.uint8), 1))
    assert O.build_causal_mask(13, 33).shape == (13, 46)
    assert O.build_causal_mask(1, 0).shape == (1, 1) and O.build_causal_mask(1, 0)[0, 0] == 0


def test_attention_two_token_closed_form():
    # hd = 4 -> scale 1/2; q . k1 / 2 = ln 3, q . k0 = 0 -> softmax = (1/4, 3/4)
    q = np.array([[[2.0, 0, 0, 0]]], np.float32)
    k = np.array([[[0.0, 0, 0, 0]], [[math.log(3.0), 0, 0, 0]]], np.float32)
    v = np.array([[[1.0, 2, 3, 4]], [[5.0, 6, 7, 8]]], np.float32)
    o = O.attention(q, k, v, None)
    np.testing.assert_allclose(o[0, 0], 0.25 * v[0, 0] + 0.75 * v[1, 0], rtol=1e-6)
    # causal prefill of the same two positions: query 0 sees only key 0
    q2 = np.concatenate([q, q], axis=0)
    o2 = O.attention(q2, k, v, O.build_causal_mask(2, 0))
    np.testing.assert_array_equal(o2[0, 0], v[0, 0])
    np.testing.assert_allclose(o2[1, 0], o[0, 0], rtol=1e-7)
    # one cached key: the output is v itself
    o1 = O.attention(q, k[:1] + 3.0, v[:1], None)
    np.testing.assert_array_equal(o1[0, 0], v[0, 0])


def test_gqa_group_mapping_reduces_to_mha():
    rng = np.random.default_rng(5)
    T, L, hd = 3, 7, 8
    q = rng.standard_normal((T, 6, hd)).astype(np.float32)
    k = rng.standard_normal((L, 2, hd)).astype(np.float32)
    v = rng.standard_normal((L, 2, hd)).astype(np.float32)
    mask = O.build_causal_mask(T, L - T)
    o = O.attention(q, k, v, mask)
    # explicit MHA with head h reading KV head h // 3 (contiguous groups)
    idx = [0, 0, 0, 1, 1, 1]
    o_mha = O.attention(q, k[:, idx], v[:, idx], mask)
    np.testing.assert_array_equal(o, o_mha)
    # identical queries inside a group give identical outputs
    q[:, 4] = q[:, 3]
    o = O.attention(q, k, v, mask)
    np.testing.assert_array_equal(o[:, 4], o[:, 3])
    assert not np.allclose(o[:, 2], o[:, 3])


def test_argmax_lowest_index_on_ties():
    assert O.argmax_lowest(np.array([1.0, 3.0, 3.0, 2.0], np.float32)) == 1


# ---------------------------------------------------------------- model-level

def test_structural_counts_per_forward():
    pc = _read_kv("pages_counts.txt")
    cfg = dict(TINY, n_layer=30, n_embd=32, n_head=2, n_head_kv=1, head_dim=16, n_ff=32, n_vocab=40)
    t = quantized_tensors(cfg, 1)
    assert len(t) == pc["gguf_tensor_count"]
    model = O.ModelWeights(cfg, t)
    model.forward([1, 2, 3], 0)
    assert model.counters == {"qmatmul": pc["qmatmul_per_forward"],
                              "rms_norm": pc["rms_norm_per_forward"],
                              "rope": pc["rope_calls_per_forward"]}


def test_decode_after_prefill_equals_full_sequence(tiny_tensors):
    ids = synth.prompt_ids(13, TINY["n_vocab"], 0)
    full = O.ModelWeights(TINY, tiny_tensors).forward(ids, 0)
    m = O.ModelWeights(TINY, tiny_tensors)
    m.forward(ids[:12], 0)
    dec = m.forward(ids[12:], 12)
    np.testing.assert_allclose(dec, full, rtol=0, atol=1e-6 * np.max(np.abs(full)))
    m = O.ModelWeights(TINY, tiny_tensors)
    m.forward(ids[:8], 0)
    chunked = m.forward(ids[8:], 8)           # chunk 2 at index_pos 8 is accepted
    np.testing.assert_allclose(chunked, full, rtol=0, atol=1e-6 * np.max(np.abs(full)))


def test_index_pos_misuse_matches_pages(tiny_tensors):
    ids = synth.prompt_ids(13, TINY["n_vocab"], 0)
    m = O.ModelWeights(TINY, tiny_tensors)
    m.forward(ids[:8], 0)
    with pytest.raises(ValueError, match=r"cannot broadcast \[5, 10\] to \[1, 9, 5, 13\]"):
        m.forward(ids[8:], 5)
    m = O.ModelWeights(TINY, tiny_tensors)
    m.forward(ids, 0)
    m.forward(ids[:7], 13)                    # continue at 13 -> cache 20
    m.clear_kv_cache()
    with pytest.raises(ValueError, match=r"cannot broadcast \[13, 46\] to \[1, 9, 13, 13\]"):
        m.forward(ids, 33)


def test_index_pos_zero_equals_fresh_model(tiny_tensors):
    ids = synth.prompt_ids(13, TINY["n_vocab"], 0)
    other = synth.prompt_ids(9, TINY["n_vocab"], 4)
    fresh = O.ModelWeights(TINY, tiny_tensors).forward(ids, 0)
    m = O.ModelWeights(TINY, tiny_tensors)
    m.forward(other, 0)
    m.forward(other[:3], 9)
    np.testing.assert_array_equal(m.forward(ids, 0), fresh)


def test_single_token_after_clear_equals_position_zero(tiny_tensors):
    m = O.ModelWeights(TINY, tiny_tensors)
    at0 = m.forward([17], 0)
    m.forward(synth.prompt_ids(5, TINY["n_vocab"], 2), 0)
    m.clear_kv_cache()
    np.testing.assert_array_equal(m.forward([17], 33), at0)


def test_tied_head_uses_the_q8_embedding(tiny_tensors):
    ids = synth.prompt_ids(6, TINY["n_vocab"], 1)
    tied = O.ModelWeights(TINY, tiny_tensors).forward(ids, 0)
    t2 = dict(tiny_tensors)
    t2["output.weight"] = tiny_tensors["token_embd.weight"]
    untied = O.ModelWeights(dict(TINY, tied_output=0), t2).forward(ids, 0)
    np.testing.assert_array_equal(tied, untied)


def _zero_layer_tensors(cfg, seed):
    t = quantized_tensors(cfg, seed)
    for li in range(cfg["n_layer"]):
        for mname in O.LAYER_MATRICES:
            rows, k = O.layer_matrix_shape(cfg, mname)
            t[f"blk.{li}.{mname}.weight"] = O.quantize_q8_0(np.zeros((rows, k), np.float32))
    return t


def test_zero_projections_pass_the_embedding_through(tiny_tensors):
    t = _zero_layer_tensors(TINY, 3)
    ids = [5, 77, 131]
    logits = O.ModelWeights(TINY, t).forward(ids, 0)
    E = O.dequantize_q8_0(t["token_embd.weight"], TINY["n_vocab"], TINY["n_embd"]).astype(np.float64)
    x = E[131]
    g = t["output_norm.weight"].astype(np.float64)
    y = x / math.sqrt(np.mean(x * x) + TINY["rms_eps"]) * g
    np.testing.assert_allclose(logits, E @ y, rtol=1e-5, atol=1e-6)


def _one_layer_cfg():
    return dict(TINY, n_layer=1, n_embd=32, n_head=2, n_head_kv=1, head_dim=16, n_ff=32, n_vocab=8)


def _single_entry(rows, k, r, c, val):
    w = np.zeros((rows, k), np.float32)
    w[r, c] = val
    blob = O.quantize_q8_0(w)
    return blob, float(O.dequantize_q8_0(blob, rows, k)[r, c])


def test_mlp_closed_form_single_entries():
    cfg = _one_layer_cfg()
    t = _zero_layer_tensors(cfg, 4)
    t["blk.0.ffn_gate.weight"], cg = _single_entry(32, 32, 0, 0, 0.8)
    t["blk.0.ffn_up.weight"], cu = _single_entry(32, 32, 0, 0, -0.3)
    t["blk.0.ffn_down.weight"], cd = _single_entry(32, 32, 0, 0, 0.6)
    m = O.ModelWeights(cfg, t)
    m.forward([3], 0)
    # read the hidden state through a second model whose head is the identity
    # on dim 0: logits[v] = E[v] . final_norm(x); compare the whole vector instead
    E = O.dequantize_q8_0(t["token_embd.weight"], 8, 32).astype(np.float64)
    x0 = E[3].copy()
    y = x0 / math.sqrt(np.mean(x0 * x0) + cfg["rms_eps"]) * t["blk.0.ffn_norm.weight"].astype(np.float64)
    z = cg * y[0]
    x1 = x0.copy()
    x1[0] += cd * (z / (1 + math.exp(-z))) * (cu * y[0])
    g = t["output_norm.weight"].astype(np.float64)
    yo = x1 / math.sqrt(np.mean(x1 * x1) + cfg["rms_eps"]) * g
    np.testing.assert_allclose(O.ModelWeights(cfg, t).forward([3], 0), E @ yo, rtol=1e-5, atol=1e-7)


def test_attention_value_path_closed_form():
    cfg = _one_layer_cfg()
    t = _zero_layer_tensors(cfg, 5)
    t["blk.0.attn_v.weight"], a = _single_entry(16, 32, 2, 1, 0.7)     # v[2] = a * y[1]
    t["blk.0.attn_output.weight"], b = _single_entry(32, 32, 5, 2, -0.9)  # x[5] += b * o[2]
    t["blk.0.attn_q.weight"], _ = _single_entry(32, 32, 0, 0, 0.5)     # q, k do not matter for
    t["blk.0.attn_k.weight"], _ = _single_entry(16, 32, 1, 3, 0.4)     # a single cached key
    E = O.dequantize_q8_0(t["token_embd.weight"], 8, 32).astype(np.float64)
    x0 = E[6].copy()
    y = x0 / math.sqrt(np.mean(x0 * x0) + cfg["rms_eps"]) * t["blk.0.attn_norm.weight"].astype(np.float64)
    x1 = x0.copy()
    x1[5] += b * a * y[1]           # o for head 0 = v of the only position, dims 0..15
    g = t["output_norm.weight"].astype(np.float64)
    yo = x1 / math.sqrt(np.mean(x1 * x1) + cfg["rms_eps"]) * g
    for pos in (0, 200):            # at any position a lone token attends to itself
        m = O.ModelWeights(cfg, t)
        np.testing.assert_allclose(m.forward([6], pos), E @ yo, rtol=1e-5, atol=1e-7)


def test_generate_loop_positions(tiny_tensors):
    m = O.ModelWeights(TINY, tiny_tensors)
    ids = synth.prompt_ids(5, TINY["n_vocab"], 9)
    out, logits = m.generate(ids, 4)
    assert len(out) == 5 and len(logits) == 5
    assert m.cache_len() == 5 + 4
    assert out[0] == O.argmax_lowest(logits[0])


def test_neox_forward_equals_rope_i_with_interleaved_rows(tiny_tensors):
    """NEOX RoPE pairs dim i with dim i + hd/2 at the angle rope_i gives pair
    (2i, 2i+1) ([QL] "RoPE：两种约定，按架构名选"), and attention scores are
    sums over dims: so the NEOX model must equal the rope_i model whose Q and K
    rows are reordered within each head to (0, hd/2, 1, hd/2 + 1, ...). A
    wrong pairing, angle or sign in either rotation breaks this."""
    cfg = dict(TINY, rope_style=1)
    hd = cfg["head_dim"]
    perm = np.empty(hd, np.int64)
    perm[0::2] = np.arange(hd // 2)
    perm[1::2] = np.arange(hd // 2) + hd // 2
    t2 = dict(tiny_tensors)
    for li in range(cfg["n_layer"]):
        for name, heads in (("attn_q", cfg["n_head"]), ("attn_k", cfg["n_head_kv"])):
            blob = tiny_tensors[f"blk.{li}.{name}.weight"]
            rows = np.concatenate([hh * hd + perm for hh in range(heads)])
            t2[f"blk.{li}.{name}.weight"] = blob[rows]
    ids = synth.prompt_ids(11, cfg["n_vocab"], 3)
    neox = O.ModelWeights(cfg, tiny_tensors)
    inter = O.ModelWeights(TINY, t2)
    a, b = neox.forward(ids, 0), inter.forward(ids, 0)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-5 * float(np.max(np.abs(a))))
    a, b = neox.forward([5], 11), inter.forward([5], 11)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-5 * float(np.max(np.abs(a))))
    # and the conventions do differ on this model
    plain = O.ModelWeights(TINY, tiny_tensors).forward(ids, 0)
    assert float(np.max(np.abs(plain - neox.forward(ids, 0)))) > 1e-3 * float(np.max(np.abs(plain)))
