"""The Llama-7B-shaped Q8_0 model (32 layers, hidden 4096, 32/8 heads of 128,
FFN 14336, vocab 32000, untied head, seed 1) at full size.

- Every weight tensor: GPU quantiser bytes == oracle quantiser bytes.
- The full 512-token prefill + 256 greedy decode run on the GPU; the oracle
  (f64) reproduces the prefill and the first decode steps, one by one:
  identical tokens, logits within 2e-3 of the largest reference logit.
- At the end of the run (768 cached positions) the CUDA-graph decode step and
  a full 768-token prefill agree on the last position (a property that holds
  at any size), and a call with index_pos + T = 4097 is rejected with the
  cache intact.
"""
import concurrent.futures as cf

import numpy as np
import pytest

from oracle import q8_oracle as O
from q8_quantized_llama_gb300 import synth
from tests.gpu_helpers import binding, gpu_quantize, logits_close, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu

CFG = dict(synth.MODEL_7B)
SEED = 1
N_ORACLE_DECODE = 3


def _oracle_quantize(w, pool):
    rows = w.shape[0]
    step = 512
    parts = list(pool.map(lambda a: O.quantize_q8_0(w[a:a + step]), range(0, rows, step)))
    return np.concatenate(parts, axis=0)


def _oracle_dequantize_f64(blob, rows, k, pool):
    step = 512
    out = np.empty((rows, k), np.float64)

    def one(a):
        out[a:a + step] = O.dequantize_q8_0(blob[a:a + step], min(step, rows - a), k)

    list(pool.map(one, range(0, rows, step)))
    return out


@pytest.fixture(scope="module")
def m7b():
    require_gpu()
    B = binding()
    dev, ora = {}, {}
    with cf.ThreadPoolExecutor(max_workers=16) as pool:
        for name, w, kind in synth.iter_model_weights_f32(CFG, SEED):
            if kind == "matrix":
                q = gpu_quantize(w)
                ora[name] = _oracle_quantize(w, pool)
                np.testing.assert_array_equal(q.cpu().numpy(), ora[name], err_msg=name)
                dev[name] = q
            else:
                dev[name] = to_dev(w)
                ora[name] = w
        model = B.Model(CFG, dev, on_device=True)
        del dev
        torch.cuda.empty_cache()
        oracle = O.ModelWeights(CFG, ora, weight_cache="f64")
        # fill the oracle's dequantised-weight cache in parallel (same function, row chunks)
        for name, blob in ora.items():
            if blob.dtype == np.uint8:
                rows = blob.shape[0]
                k = blob.shape[1] // 34 * 32
                if name == "token_embd.weight":
                    continue  # the oracle dequantises the embedding itself
                oracle._deq[name] = _oracle_dequantize_f64(blob, rows, k, pool)
    yield model, oracle
    model.close()


def test_7b_prefill_512_decode_256(m7b):
    model, oracle = m7b
    B = binding()
    prompt = synth.prompt_ids(512, CFG["n_vocab"], SEED)
    ids = model.generate(prompt, 255)               # 256 tokens: prefill's + 255 decode steps
    assert model.cache_len() == 512 + 255

    # oracle, step by step, on the first decode steps
    ref_logits = oracle.forward(prompt, 0)
    ref = [O.argmax_lowest(ref_logits)]
    gpu_logits = model.forward(prompt, 0)
    ok, err, bound = logits_close(gpu_logits, ref_logits)
    assert ok, ("prefill", err, bound)
    pos = 512
    for step in range(N_ORACLE_DECODE):
        ref_logits = oracle.forward([ref[-1]], pos)
        gpu_logits = model.forward([ref[-1]], pos)
        pos += 1
        ok, err, bound = logits_close(gpu_logits, ref_logits)
        assert ok, (step, err, bound)
        ref.append(O.argmax_lowest(ref_logits))
    assert list(ids[:N_ORACLE_DECODE + 1]) == ref

    # full-size property: decode step at position 767 == prefill of 768 tokens
    ids = model.generate(prompt, 255)
    seq = np.concatenate([prompt, ids]).astype(np.int32)   # 768 tokens, the last not yet consumed
    dec = model.forward(seq[767:], 767)
    assert model.cache_len() == 768
    # index_pos + T = 4097 is rejected and leaves the cache as it was
    too_long = np.zeros(4097 - 768, np.int32)
    assert model.forward_status(too_long, 768) == B.LQ8_ERR_CTX
    assert model.cache_len() == 768
    pre = model.forward(seq, 0)
    ok, err, bound = logits_close(dec, pre)
    assert ok, ("decode vs prefill at 767", err, bound)
    assert int(np.argmax(dec)) == int(np.argmax(pre))
