"""The allocation-free attention entry point, checked against the CPU oracle's
attention and against the regular entry point.

Some callers cannot allocate device memory: hosts that give all GPU memory to
their own pool and accept only the buffers they pass in, real-time loops that
cannot take cudaMalloc's implicit synchronisation, plugins that must not
create allocations they cannot account for. llama_q8_attention_decode_noalloc
serves them with the library's fixed scratch array. This file is collected
last on purpose, and must pass both alone in a fresh process and after the
rest of the suite (the array keeps the contents of earlier calls).

kv_len 1 and 64 take the kernel's single-split path (one 64-position chunk
per KV head, the output written directly); 65 and above take the multi-split
path whose partial results are merged through the scratch array.
"""
import numpy as np
import pytest

from oracle import q8_oracle as O
from q8_quantized_llama_gb300 import synth
from tests.gpu_helpers import binding, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu


def _check(B, nh, nkv, hd, stride, kv_len, seed):
    q_host = synth.normal_f32((1, nh, hd), seed, 11)
    k_host = synth.normal_f32((nkv, stride, hd), seed, 12)
    v_host = synth.normal_f32((nkv, stride, hd), seed, 13)
    q, kc, vc = to_dev(q_host), to_dev(k_host), to_dev(v_host)
    ws_bytes = B.llama_q8_attention_workspace_bytes(nh, nkv, hd, stride)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    ref = torch.empty((1, nh, hd), dtype=torch.float32, device="cuda")
    B.llama_q8_attention(q, kc, vc, 1, kv_len - 1, nh, nkv, hd, stride, ref, ws, ws_bytes)
    out = torch.full((1, nh, hd), float("nan"), dtype=torch.float32, device="cuda")
    B.llama_q8_attention_decode_noalloc(q, kc, vc, kv_len, nh, nkv, hd, stride, out)
    torch.cuda.synchronize()
    got, regular = out.cpu().numpy(), ref.cpu().numpy()
    # the oracle: cache positions [0, kv_len) as [kv_len, n_head_kv, head_dim], no mask (T == 1)
    k_seq = np.ascontiguousarray(k_host[:, :kv_len].transpose(1, 0, 2))
    v_seq = np.ascontiguousarray(v_host[:, :kv_len].transpose(1, 0, 2))
    want = O.attention(q_host, k_seq, v_seq, None)
    # the attention tolerance of the suite: 2e-4 * max|v| over the visible rows
    tol = 2e-4 * float(np.max(np.abs(v_host[:, :kv_len])))
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got.astype(np.float64) - want)))
    assert err <= tol, (nh, nkv, hd, kv_len, err, tol)
    err_regular = float(np.max(np.abs(got.astype(np.float64) - regular)))
    assert err_regular <= tol, (nh, nkv, hd, kv_len, err_regular, tol)


@pytest.mark.parametrize("kv_lens", [(1, 64, 65, 331, 4096)])
def test_noalloc_attention_matches_oracle_on_consecutive_calls(kv_lens):
    require_gpu()
    B = binding()
    # calls in a row on the shared array: each must not see the previous call's leftovers
    for i, kv_len in enumerate(kv_lens):
        _check(B, 9, 3, 64, 4096, kv_len, seed=21 + i)
    for i, kv_len in enumerate((1, 64, 65, 1500)):
        _check(B, 32, 8, 128, 4096, kv_len, seed=31 + i)


def test_noalloc_rejects_oversized_scratch_and_misaligned_buffers():
    require_gpu()
    B = binding()
    q = torch.zeros(16 * 128, dtype=torch.float32, device="cuda")
    kv = torch.zeros(16, dtype=torch.float32, device="cuda")
    out = torch.zeros(16 * 128, dtype=torch.float32, device="cuda")
    with pytest.raises(B.Q8Error) as e:
        # 64 KV heads x 64 chunks x group 8 x 130 floats is far above the fixed 2 MiB
        B.llama_q8_attention_decode_noalloc(q, kv, kv, 10, 512, 64, 128, 4096, out)
    assert e.value.status == B.LQ8_ERR_UNSUPPORTED
    # a buffer 4 bytes past a 16-byte boundary is refused on the host, before any launch
    nh, nkv, hd, stride = 9, 3, 64, 128
    qb = torch.zeros(nh * hd + 4, dtype=torch.float32, device="cuda")
    kb = torch.zeros(nkv * stride * hd + 4, dtype=torch.float32, device="cuda")
    ob = torch.zeros(nh * hd + 4, dtype=torch.float32, device="cuda")
    aligned = (qb[:nh * hd], kb[:nkv * stride * hd], kb[:nkv * stride * hd], ob[:nh * hd])
    for which in range(4):
        args = list(aligned)
        base = (qb, kb, kb, ob)[which]
        n = args[which].numel()
        args[which] = base[1:1 + n]
        assert args[which].data_ptr() % 16 == 4
        with pytest.raises(B.Q8Error) as e:
            B.llama_q8_attention_decode_noalloc(args[0], args[1], args[2], 10, nh, nkv, hd, stride, args[3])
        assert e.value.status == B.LQ8_ERR_ARG
    torch.cuda.synchronize()
    assert float(ob.abs().sum()) == 0.0   # nothing was written
