"""The seeded input generator: deterministic, thread-count independent, right shapes."""
import numpy as np

from q8_quantized_llama_gb300 import synth


def test_specs_135m():
    specs = synth.model_tensor_specs(synth.MODEL_135M)
    assert len(specs) == 272
    assert specs[0] == ("token_embd.weight", (49152, 576), "matrix")
    assert ("blk.29.ffn_down.weight", (576, 1536), "matrix") in specs
    assert not any(n == "output.weight" for n, _, _ in specs)
    specs7 = synth.model_tensor_specs(synth.MODEL_7B)
    assert len(specs7) == 32 * 9 + 3 and specs7[-1] == ("output.weight", (32000, 4096), "matrix")


def test_weights_deterministic_and_thread_independent():
    cfg = dict(synth.MODEL_135M, n_layer=1, n_vocab=600)
    a = synth.model_weights_f32(cfg, 0, threads=1)
    b = synth.model_weights_f32(cfg, 0, threads=4)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])
    c = synth.model_weights_f32(cfg, 1, threads=2)
    assert not np.array_equal(a["blk.0.attn_q.weight"], c["blk.0.attn_q.weight"])
    w = a["blk.0.ffn_up.weight"]
    assert w.dtype == np.float32 and abs(float(w.std()) - 0.02) < 1e-3
    g = a["blk.0.attn_norm.weight"]
    assert abs(float(g.mean()) - 1.0) < 5e-3


def test_prompt_ids_range_and_determinism():
    ids = synth.prompt_ids(203, 49152, 0)
    assert ids.dtype == np.int32 and ids.shape == (203,)
    assert ids.min() >= 0 and ids.max() < 49152
    np.testing.assert_array_equal(ids, synth.prompt_ids(203, 49152, 0))
