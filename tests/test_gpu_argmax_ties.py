"""Greedy argmax ties on the GPU: the lowest index among equal maxima (reading
R7 of the build; "生成一个 token", prefill 和 decode: argmax then to_scalar).

The output head is built from a few distinct rows repeated with a period, so
every logit value occurs at many indices spread over the whole vocabulary
(and so over many CTAs of the lm_head kernel). The duplicated rows must give
bit-identical logits, and the greedy token must be the lowest index holding
the maximum — for the prefill, the CUDA-graph decode step and the device-fed
generation loop, with the head untied (output.weight) and tied (token_embd),
row-parallel and split-K over a 2-CTA cluster.
"""
import numpy as np
import pytest

from oracle import q8_oracle as O
from q8_quantized_llama_gb300 import synth
from tests.gpu_helpers import binding, gpu_model_tensors, logits_close, oracle_model_tensors, require_gpu, torch

pytestmark = pytest.mark.gpu

PERIOD = 97
BASE = dict(n_layer=1, n_embd=128, n_head=4, n_head_kv=2, head_dim=64, n_ff=256, n_vocab=49152,
            max_seq=4096, rms_eps=1e-5, rope_theta=10000.0)


def _periodic(w):
    rows = w.shape[0]
    return np.ascontiguousarray(w[np.arange(rows) % PERIOD])


@pytest.mark.parametrize("tied,head_splits", [(0, 0), (1, 0), (0, 2)])
def test_argmax_returns_lowest_index_among_equal_maxima(tied, head_splits):
    require_gpu()
    B = binding()
    cfg = dict(BASE, tied_output=tied, head_splits=head_splits)
    host = synth.model_weights_f32(cfg, 7)
    head = "token_embd.weight" if tied else "output.weight"
    host[head] = _periodic(host[head])
    dev_t = gpu_model_tensors(cfg, 7, host)
    ora_t = oracle_model_tensors(cfg, 7, host)
    model = B.Model(cfg, dev_t, on_device=True)
    oracle = O.ModelWeights(cfg, ora_t)
    try:
        prompt = synth.prompt_ids(9, cfg["n_vocab"], 7)
        ref_ids, ref_logits = oracle.generate(prompt, 4)
        pos = len(prompt)
        toks = []
        for step in range(5):
            ids = prompt if step == 0 else [toks[-1]]
            logits = model.forward(ids, 0 if step == 0 else pos)
            if step:
                pos += 1
            ok, err, bound = logits_close(logits, ref_logits[step])
            assert ok, (step, err, bound)
            mx = logits.max()
            at = np.flatnonzero(logits == mx)
            assert at.size >= cfg["n_vocab"] // PERIOD, at.size     # a tie across the vocabulary
            # duplicated rows give bit-identical logits on the GPU
            lg = logits[: (cfg["n_vocab"] // PERIOD) * PERIOD].reshape(-1, PERIOD)
            assert np.all(lg == lg[0:1]), step
            toks.append(int(at[0]))
            assert toks[-1] < PERIOD and toks[-1] == ref_ids[step]
        # the same tokens from the greedy calls that return the token only
        nxt = model.forward_argmax(prompt, 0)
        assert nxt == toks[0]
        pos = len(prompt)
        for step in range(1, 5):
            nxt = model.forward_argmax([nxt], pos)
            pos += 1
            assert nxt == toks[step], step
        np.testing.assert_array_equal(model.generate(prompt, 4), toks)
    finally:
        model.close()
        torch.cuda.empty_cache()
