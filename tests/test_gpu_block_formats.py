"""The matrix-vector product in Q5_0, Q4_K and Q6_K ("速度", CPU GGUF：decode
快，prefill 慢) through the C ABI against the oracle's dequantisation times x
in f64, element by element.

Shapes: the pages' QMatMul shape [1,1536]x[1536,576] (the down projection,
whose rows of 1536 fit the 256-weight K-quant block); ragged row counts (a
partial last tile); one block per row; few tiles (the block range split over
a cluster); many tiles (persistent CTAs looping over tiles); the 7B down
projection's row length 14336; and the chained-launch flag.

Bound per output: |y - ref| <= (n + 12) 2^-24 sum_i (|a_i| + |b_i|) |x_i|,
where w_i = a_i - b_i splits each weight into its scaled code and (Q4_K) its
subtracted minimum, and n = 16 + k / 256 + 8 is the longest f32 summation
chain of the kernel (16 pairwise steps in a 32-weight unit, the units of one
warp, eight warp partials); 12 more roundings cover the scale products and
the cluster sum.
"""
import numpy as np
import pytest

from oracle import q8_oracle as O
from q8_quantized_llama_gb300 import synth
from tests.gpu_helpers import binding, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu

TYPES = {"Q5_0": 6, "Q4_K": 12, "Q6_K": 14}


def _run(B, t, rows, k, seed, flags=0):
    blob = synth.random_blocks(t, rows, k, seed)
    x = synth.normal_f32((k,), seed, 5)
    nbytes = B.llama_q8_packed_bytes_fmt(t, rows, k)
    assert nbytes == ((rows + 31) // 32 * 32) * O.block_format_row_bytes(t, k)
    packed = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    B.llama_q8_pack_fmt(t, to_dev(blob), rows, k, packed)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    B.llama_q8_matvec_fmt(t, packed, rows, k, to_dev(x), y, flags)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    if t == O.GGUF_TYPE_Q4_K:
        a, b = O.dequantize_q4_k(blob, rows, k, parts=True)
        w = a - b
        mag = np.abs(a) + np.abs(b)
    else:
        w = O.dequantize_block_format(t, blob, rows, k)
        mag = np.abs(w)
    x64 = x.astype(np.float64)
    ref = w @ x64
    bound = (16 + k / 256 + 8 + 12) * 2.0 ** -24 * (mag @ np.abs(x64))
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= bound), (rows, k, float(np.max(err / bound)))
    return got


@pytest.mark.parametrize("fmt", list(TYPES))
@pytest.mark.parametrize("rows,k", [(576, 1536), (200, 1536), (33, 256), (96, 14336), (4096, 1024),
                                    (14336 // 4, 4096)])
def test_matvec_block_formats_against_oracle(fmt, rows, k):
    require_gpu()
    B = binding()
    t = TYPES[fmt]
    _run(B, t, rows, k, seed=rows + k)


@pytest.mark.parametrize("fmt", list(TYPES))
def test_matvec_block_formats_q5_0_row_lengths_and_chained_flag(fmt):
    require_gpu()
    B = binding()
    t = TYPES[fmt]
    if t == O.GGUF_TYPE_Q5_0:
        for rows, k in ((576, 576), (1536, 576), (31, 32), (64, 96)):   # the Q4_K_M file's Q5_0 shapes
            _run(B, t, rows, k, seed=7 + rows)
    a = _run(B, t, 576, 1536, seed=3)
    b = _run(B, t, 576, 1536, seed=3, flags=B.LQ8_MATMUL_EARLY_WEIGHTS)
    np.testing.assert_array_equal(a, b)


def test_matvec_block_formats_argument_checks():
    require_gpu()
    B = binding()
    buf = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    x = torch.zeros(4096, dtype=torch.float32, device="cuda")
    y = torch.zeros(64, dtype=torch.float32, device="cuda")
    for t, k in ((12, 576), (14, 300), (6, 48)):                        # k not a multiple of the block
        assert B.llama_q8_packed_bytes_fmt(t, 64, k) == 0
        with pytest.raises(B.Q8Error) as e:
            B.llama_q8_matvec_fmt(t, buf, 64, k, x, y)
        assert e.value.status == B.LQ8_ERR_ARG
    with pytest.raises(B.Q8Error) as e:
        B.llama_q8_matvec_fmt(2, buf, 64, 256, x, y)                    # Q4_0: not built
    assert e.value.status == B.LQ8_ERR_UNSUPPORTED
    with pytest.raises(B.Q8Error) as e:
        B.llama_q8_matvec_fmt(12, buf[4:], 64, 256, x, y)               # unaligned packed matrix
    assert e.value.status == B.LQ8_ERR_ARG
