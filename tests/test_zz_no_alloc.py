"""The allocation-free attention entry point against the regular one.

Some callers cannot allocate device memory: hosts that give all GPU memory to
their own pool and accept only the buffers they pass in, real-time loops that
cannot take cudaMalloc's implicit synchronisation, plugins that must not
create allocations they cannot account for. llama_q8_attention_decode_noalloc
serves them with the library's fixed scratch array. This file is collected
last on purpose, and must pass both alone in a fresh process and after the
rest of the suite (the array keeps the contents of earlier calls).
"""
import numpy as np
import pytest

from q8_quantized_llama_gb300 import synth
from tests.gpu_helpers import binding, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu


def _run_both(B, nh, nkv, hd, stride, kv_len, seed):
    q = to_dev(synth.normal_f32((1, nh, hd), seed, 11))
    kc = to_dev(synth.normal_f32((nkv, stride, hd), seed, 12))
    vc_host = synth.normal_f32((nkv, stride, hd), seed, 13)
    vc = to_dev(vc_host)
    ws_bytes = B.llama_q8_attention_workspace_bytes(nh, nkv, hd, stride)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty((1, nh, hd), dtype=torch.float32, device="cuda")
    B.llama_q8_attention(q, kc, vc, 1, kv_len - 1, nh, nkv, hd, stride, ref, ws, ws_bytes)
    out = torch.full((1, nh, hd), float("nan"), dtype=torch.float32, device="cuda")
    B.llama_q8_attention_decode_noalloc(q, kc, vc, kv_len, nh, nkv, hd, stride, out)
    torch.cuda.synchronize()
    got, want = out.cpu().numpy(), ref.cpu().numpy()
    # same tolerance as the attention parity tests: 2e-4 * max|v| over the visible rows
    tol = 2e-4 * float(np.max(np.abs(vc_host[:, :kv_len])))
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(got.astype(np.float64) - want))) <= tol


def test_noalloc_attention_matches_regular_entry_point_twice():
    require_gpu()
    B = binding()
    # two calls in a row: the second must not see the first call's leftovers
    _run_both(B, 9, 3, 64, 4096, 331, seed=21)
    _run_both(B, 32, 8, 128, 4096, 1500, seed=22)


def test_noalloc_rejects_oversized_scratch():
    require_gpu()
    B = binding()
    q = torch.zeros(16 * 128, dtype=torch.float32, device="cuda")
    kv = torch.zeros(16, dtype=torch.float32, device="cuda")
    out = torch.zeros(16 * 128, dtype=torch.float32, device="cuda")
    with pytest.raises(B.Q8Error) as e:
        # 64 KV heads x 64 chunks x group 8 x 130 floats is far above the fixed 2 MiB
        B.llama_q8_attention_decode_noalloc(q, kv, kv, 10, 512, 64, 128, 4096, out)
    assert e.value.status == B.LQ8_ERR_UNSUPPORTED
