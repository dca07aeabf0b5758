"""The 135M-shaped model with NEOX RoPE (rope_style 1: dim i pairs with dim
i + head_dim/2, the convention the pages' loader picks for the architectures it
lists, "量化 llama 的一次前向", RoPE：两种约定，按架构名选) against the oracle's
NEOX forward: identical greedy tokens and logits within tolerance for the
two-, three- and five-kernel decode layers, the tensor-core prefill, and the
K/V cache in natural dim order."""
import numpy as np
import pytest

from oracle import q8_oracle as O
from q8_quantized_llama_gb300 import synth
from tests.gpu_helpers import binding, gpu_model_tensors, logits_close, oracle_model_tensors, require_gpu, torch

pytestmark = pytest.mark.gpu

CFG = dict(synth.MODEL_135M, n_layer=4, rope_style=1)
V = CFG["n_vocab"]


@pytest.fixture(scope="module")
def neox():
    require_gpu()
    B = binding()
    host = synth.model_weights_f32(CFG, 11)
    dev_t = gpu_model_tensors(CFG, 11, host)
    ora_t = oracle_model_tensors(CFG, 11, host)
    models = {
        "auto": B.Model(CFG, dev_t, on_device=True),
        "layered": B.Model(dict(CFG, decode_kernel=1), dev_t, on_device=True),
        "three": B.Model(dict(CFG, decode_kernel=4), dev_t, on_device=True),
    }
    del dev_t
    torch.cuda.empty_cache()
    yield models, ora_t
    for m in models.values():
        m.close()


@pytest.mark.parametrize("form", ["auto", "three", "layered"])
def test_neox_generation_matches_oracle(neox, form):
    models, ora_t = neox
    model = models[form]
    oracle = O.ModelWeights(CFG, ora_t)
    prompt = synth.prompt_ids(13, V, 4)
    ora_ids, ora_logits = oracle.generate(prompt, 8)
    logits = model.forward(prompt, 0)
    ok, err, bound = logits_close(logits, ora_logits[0])
    assert ok, ("prefill", err, bound)
    got = [int(np.argmax(logits))]
    pos = len(prompt)
    for step in range(1, 9):
        logits = model.forward([got[-1]], pos)
        pos += 1
        ok, err, bound = logits_close(logits, ora_logits[step])
        assert ok, (step, err, bound)
        got.append(int(np.argmax(logits)))
    assert got == ora_ids


def test_neox_tensor_core_prefill_and_cache(neox):
    models, ora_t = neox
    model = models["auto"]
    oracle = O.ModelWeights(CFG, ora_t)
    prompt = synth.prompt_ids(40, V, 5)                 # > 16 rows: tensor-core products
    ref = oracle.forward(prompt, 0)
    got = model.forward(prompt, 0)
    ok, err, bound = logits_close(got, ref)
    assert ok, (err, bound)
    assert int(np.argmax(got)) == int(np.argmax(ref))
    for layer in (0, 3):
        k, v = model.read_kv(layer, 0, 40)               # natural dim order
        kc, vc = oracle.kv_cache[layer]
        for a, b in ((k, np.transpose(kc, (1, 0, 2))), (v, np.transpose(vc, (1, 0, 2)))):
            e = float(np.max(np.abs(a.astype(np.float64) - b)))
            assert e <= 1e-4 * float(np.max(np.abs(b))), (layer, e)


def test_neox_differs_from_rope_i(neox):
    """The same weights under the Llama convention give other logits (the
    convention is not silently ignored)."""
    models, ora_t = neox
    B = binding()
    prompt = synth.prompt_ids(13, V, 4)
    a = models["auto"].forward(prompt, 0)
    host = synth.model_weights_f32(CFG, 11)
    plain = B.Model(dict(CFG, rope_style=0), gpu_model_tensors(CFG, 11, host), on_device=True)
    try:
        b = plain.forward(prompt, 0)
    finally:
        plain.close()
    assert float(np.max(np.abs(a - b))) > 1e-3 * float(np.max(np.abs(a)))
