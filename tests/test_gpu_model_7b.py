"""The Llama-7B-shaped Q8_0 model (32 layers, hidden 4096, 32/8 heads of 128,
FFN 14336, vocab 32000, untied head, seed 1) at full size: the generation run
of "生成一个 token" (实验程序) with a 512-token prompt and 256 greedy decode
steps, the cache reaching 768 positions.

- Every weight tensor: GPU quantiser bytes == oracle quantiser bytes.
- The oracle (f64) runs the prefill and all 256 decode steps one by one; at
  every step the GPU's logits lie within 2e-3 of the largest reference logit
  and the greedy tokens are identical, both for the host API step by step and
  for the device-fed generation loop. Steps whose oracle top-2 gap is below
  that tolerance are reported as ambiguous (they must still agree).
- A call with index_pos + T = 4097 is rejected with the cache intact, and the
  CUDA-graph decode step at position 767 agrees with a 768-token prefill.
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
N_DECODE = 256


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
    ids = model.generate(prompt, N_DECODE)           # the prefill's token + one per decode step
    assert len(ids) == N_DECODE + 1 and model.cache_len() == 512 + N_DECODE

    # oracle and the host API, step by step over the whole run
    ref_logits = oracle.forward(prompt, 0)
    ref = [O.argmax_lowest(ref_logits)]
    gpu_logits = model.forward(prompt, 0)
    ok, err, bound = logits_close(gpu_logits, ref_logits)
    assert ok, ("prefill", err, bound)
    got = [int(np.argmax(gpu_logits))]
    ambiguous, worst = [], err / bound

    def note_gap(step, lg):
        top2 = np.sort(lg)[-2:]
        if top2[1] - top2[0] <= 2e-3 * float(np.max(np.abs(lg))):
            ambiguous.append(step)

    note_gap(0, ref_logits)
    pos = 512
    for step in range(1, N_DECODE + 1):
        ref_logits = oracle.forward([ref[-1]], pos)
        note_gap(step, ref_logits)
        gpu_logits = model.forward([got[-1]], pos)
        pos += 1
        ok, err, bound = logits_close(gpu_logits, ref_logits)
        assert ok, (step, err, bound)
        worst = max(worst, err / bound)
        ref.append(O.argmax_lowest(ref_logits))
        got.append(int(np.argmax(gpu_logits)))
        assert got[-1] == ref[-1], (step, got[-1], ref[-1])
    print(f"7B run: {N_DECODE} decode steps, worst logit error {worst:.3f} of the bound, "
          f"ambiguous steps (oracle top-2 gap within tolerance): {ambiguous}")
    assert got == ref
    assert list(ids) == ref                           # the device-fed loop gives the same tokens
    assert model.cache_len() == 768

    # index_pos + T = 4097 is rejected and leaves the cache as it was
    too_long = np.zeros(4097 - 768, np.int32)
    assert model.forward_status(too_long, 768) == B.LQ8_ERR_CTX
    assert model.cache_len() == 768

    # full-size property: the decode step at position 767 == a prefill of the 768 tokens
    seq = np.concatenate([prompt, ids[:-1]]).astype(np.int32)   # 768 tokens
    model.forward(seq[:767], 0)
    dec = model.forward(seq[767:], 767)
    pre = model.forward(seq, 0)
    ok, err, bound = logits_close(dec, pre)
    assert ok, ("decode vs prefill at 767", err, bound)
    assert int(np.argmax(dec)) == int(np.argmax(pre))
