"""End-to-end parity of the 135M-shaped Q8_0 Llama through the C ABI against
the CPU oracle: the 13 + 20 generation run, the 203 + 128 run, the KV cache
after RoPE, the index_pos rules of the boundary, and the device-resident API."""
import numpy as np
import pytest

from oracle import q8_oracle as O
from q8_quantized_llama_gb300 import synth
from tests.gpu_helpers import (binding, gpu_model_tensors, logits_close, oracle_model_tensors, require_gpu,
                               torch)

pytestmark = pytest.mark.gpu

CFG = dict(synth.MODEL_135M)
V = CFG["n_vocab"]


@pytest.fixture(scope="module")
def m135():
    require_gpu()
    B = binding()
    host = synth.model_weights_f32(CFG, 0)
    dev_t = gpu_model_tensors(CFG, 0, host)
    ora_t = oracle_model_tensors(CFG, 0, host)
    for name, t in dev_t.items():     # the GPU quantiser matches the oracle's bytes
        if ora_t[name].dtype == np.uint8:
            np.testing.assert_array_equal(t.cpu().numpy(), ora_t[name], err_msg=name)
    models = {
        "front": B.Model(CFG, dev_t, on_device=True),                          # automatic: two kernels per layer
        "three": B.Model(dict(CFG, decode_kernel=4), dev_t, on_device=True),   # front, gate/up, down
        "four": B.Model(dict(CFG, decode_kernel=3), dev_t, on_device=True),    # attention applies W_o
        "layered": B.Model(dict(CFG, decode_kernel=1), dev_t, on_device=True), # five kernels per layer
        "splitk": B.Model(dict(CFG, head_splits=2), dev_t, on_device=True),    # split-K lm_head
    }
    del dev_t
    torch.cuda.empty_cache()
    models["oracle"] = O.ModelWeights(CFG, ora_t, weight_cache="f64")
    yield models
    for name, m in models.items():
        if name != "oracle":
            m.close()


@pytest.fixture(params=["front", "three", "four", "layered", "splitk"])
def either(request, m135):
    return m135[request.param], m135["oracle"]


def _check_run(model, oracle, prompt, n_decode):
    """Greedy run step by step on both sides: identical tokens, logits within tol."""
    ora_ids, ora_logits = oracle.generate(prompt, n_decode)
    logits = model.forward(prompt, 0)
    ok, err, bound = logits_close(logits, ora_logits[0])
    assert ok, ("prefill", err, bound)
    got = [int(np.argmax(logits))]
    pos = len(prompt)
    for step in range(1, n_decode + 1):
        logits = model.forward([got[-1]], pos)
        pos += 1
        ok, err, bound = logits_close(logits, ora_logits[step])
        assert ok, (step, err, bound)
        got.append(int(np.argmax(logits)))
    assert got == ora_ids
    return ora_ids


def test_generation_13_prompt_20_decode(either):
    model, oracle = either
    prompt = synth.prompt_ids(13, V, 0)
    ids = _check_run(model, oracle, prompt, 20)
    # the graph-replay generation loop gives the same tokens
    np.testing.assert_array_equal(model.generate(prompt, 20), ids)
    assert model.cache_len() == 33


def test_generation_203_prompt_128_decode(either):
    model, oracle = either
    prompt = synth.prompt_ids(203, V, 0)
    ids = _check_run(model, oracle, prompt, 128)
    for _ in range(2):  # fresh cache each repetition, same tokens
        np.testing.assert_array_equal(model.generate(prompt, 128), ids)


def test_kv_cache_after_rope_matches_oracle(either):
    model, oracle = either
    prompt = synth.prompt_ids(13, V, 5)
    oracle.forward(prompt, 0)
    model.forward(prompt, 0)
    oracle.forward([7], 13)
    model.forward([7], 13)
    for layer in (0, 29):
        k, v = model.read_kv(layer, 0, 14)
        kc, vc = oracle.kv_cache[layer]
        kr = np.transpose(kc, (1, 0, 2))
        vr = np.transpose(vc, (1, 0, 2))
        for got, ref in ((k, kr), (v, vr)):
            err = float(np.max(np.abs(got.astype(np.float64) - ref)))
            assert err <= 1e-4 * float(np.max(np.abs(ref))), (layer, err)


def test_index_pos_rules(m135):
    model = m135["front"]
    B = binding()
    prompt = synth.prompt_ids(13, V, 1)
    full = model.forward(prompt, 0)
    assert model.cache_len() == 13
    # page transcript: a second chunk at the wrong index_pos is rejected ...
    model.forward(prompt[:8], 0)
    assert model.forward_status(prompt[8:], 5) == B.LQ8_ERR_POS
    assert model.cache_len() == 8                      # state unchanged
    # ... and at the right one it equals the single prefill
    chunked = model.forward(prompt[8:], 8)
    ok, err, bound = logits_close(chunked, full)
    assert ok and int(np.argmax(chunked)) == int(np.argmax(full))
    # decode with a wrong index_pos (silent on the pages) is an error here
    assert model.forward_status([3], 20) == B.LQ8_ERR_POS
    assert model.forward_status([3], 12) == B.LQ8_ERR_POS
    # T == 0 and bad ids
    assert model.forward_status(np.zeros(0, np.int32), 13) == B.LQ8_ERR_ARG
    assert model.forward_status([V], 13) == B.LQ8_ERR_TOKEN
    assert model.forward_status([-1], 13) == B.LQ8_ERR_TOKEN
    assert model.cache_len() == 13
    # reset: counter back to 0; continuing at the old position is an error
    model.reset()
    assert model.cache_len() == 0
    assert model.forward_status(prompt, 33) == B.LQ8_ERR_POS
    # index_pos 0 after use equals a fresh run, bit for bit
    again = model.forward(prompt, 0)
    np.testing.assert_array_equal(again, full)


def test_context_limit(m135):
    model = m135["front"]
    B = binding()
    prompt = synth.prompt_ids(64, V, 2)
    assert model.forward_status(np.zeros(4097, np.int32), 0) == B.LQ8_ERR_CTX
    model.forward(prompt, 0)
    assert model.forward_status([1], 4095) == B.LQ8_ERR_POS
    assert model.cache_len() == 64
    big = synth.prompt_ids(4032, V, 3)
    model.forward(big, 64)                              # fills the cache to 4096
    assert model.cache_len() == 4096
    assert model.forward_status([1], 4096) == B.LQ8_ERR_CTX
    assert model.cache_len() == 4096


def test_prefill_and_decode_paths_agree(either):
    model, oracle = either
    seq = synth.prompt_ids(40, V, 4)
    whole = model.forward(seq, 0)                       # matrix-matrix path
    model.forward(seq[:39], 0)
    last = model.forward(seq[39:], 39)                  # CUDA-graph decode step
    ref = oracle.forward(seq, 0)
    for got in (whole, last):
        ok, err, bound = logits_close(got, ref)
        assert ok, (err, bound)


def test_device_resident_api(m135):
    model, layered = m135["front"], m135["layered"]
    prompt = synth.prompt_ids(203, V, 0)
    ref = model.generate(prompt, 16)
    d_ids = torch.from_numpy(prompt).cuda()
    d_next = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_out = torch.zeros(16, dtype=torch.int32, device="cuda")
    model.prefill_async(d_ids, 203, 0, d_next)
    model.decode_async(16, d_out)
    model.sync()
    got = np.concatenate([d_next.cpu().numpy(), d_out.cpu().numpy()])
    np.testing.assert_array_equal(got, ref)
    assert model.cache_len() == 203 + 16
    assert model.decode_kernel_count() == 1 + 2 * CFG["n_layer"] + 1   # layer front + MLP
    assert m135["three"].decode_kernel_count() == 1 + 3 * CFG["n_layer"] + 1
    assert m135["four"].decode_kernel_count() == 1 + 4 * CFG["n_layer"] + 1
    assert layered.decode_kernel_count() == 1 + 5 * CFG["n_layer"] + 1


LONG_PROMPT = 3900


@pytest.fixture(scope="module")
def long_run(m135):
    """The oracle's greedy run from a 3900-token prompt to the end of the
    4096-position cache: prefill, then decode steps at positions 3900..4095."""
    prompt = synth.prompt_ids(LONG_PROMPT, V, 6)
    ids, logits = m135["oracle"].generate(prompt, CFG["max_seq"] - LONG_PROMPT)
    return prompt, ids, logits


def test_long_context_decode_matches_oracle(either, long_run):
    """Decode steps near the 4096-position limit ([QL] from_gguf: the rotary
    table and the cache end at 4096) against the oracle, every step: logits
    within tolerance and identical greedy tokens, up to the last position."""
    model, _ = either
    prompt, ref_ids, ref_logits = long_run
    logits = model.forward(prompt, 0)
    ok, err, bound = logits_close(logits, ref_logits[0])
    assert ok, ("prefill", err, bound)
    got = [int(np.argmax(logits))]
    pos = LONG_PROMPT
    for step in range(1, len(ref_logits)):
        logits = model.forward([got[-1]], pos)
        pos += 1
        ok, err, bound = logits_close(logits, ref_logits[step])
        assert ok, (pos - 1, err, bound)
        got.append(int(np.argmax(logits)))
        assert got[-1] == ref_ids[step], (pos - 1, got[-1], ref_ids[step])
    assert model.cache_len() == CFG["max_seq"]
    assert got == ref_ids


@pytest.mark.parametrize("variant", ["front", "layered"])
def test_decode_timeline_profile(m135, variant):
    """The instrumented copy of the decode graph (timeline stamps on every
    launch) computes the same greedy tokens as the product graph, and reports
    every launch of every step: exclusive times that add up to the step and
    spans that contain them."""
    model = m135[variant]
    prompt = synth.prompt_ids(203, V, 0)
    ref = model.generate(prompt, 17)
    assert model.forward_argmax(prompt, 0) == ref[0]
    prof = model.profile_decode(16)                       # decode steps 1..16, instrumented
    assert model.cache_len() == 203 + 16
    d_out = torch.zeros(1, dtype=torch.int32, device="cuda")
    model.decode_async(1, d_out)                          # step 17 on the product graph
    model.sync()
    assert int(d_out.cpu()[0]) == ref[17]
    launches = sum(v[0] for v in prof.values())
    assert launches == 16 * model.decode_kernel_count()
    for name, (n, ms, span_ms, nbytes) in prof.items():
        if n:
            assert 0.0 < ms <= span_ms and nbytes > 0, name
    assert prof["embed"][0] == 16 and prof["gemv_head_argmax"][0] == 16
