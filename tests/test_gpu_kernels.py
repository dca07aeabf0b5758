"""Kernel parity through the C ABI against the CPU oracle: Q8_0 quantiser
(bit-exact), Q8_0 matmul (the linear sweep shapes of the 135M model plus the
7B GEMV shapes), GQA attention (decode and causal prefill)."""
import math

import numpy as np
import pytest

from oracle import q8_oracle as O
from q8_quantized_llama_gb300 import synth
from tests.gpu_helpers import binding, gpu_quantize, require_gpu, to_dev, torch

pytestmark = pytest.mark.gpu

U = 2.0 ** -24  # f32 unit roundoff


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


# ------------------------------------------------------------------ quantiser

def _golden_blocks():
    from tests.test_oracle_pins import _hand_blocks
    return _hand_blocks()


def test_quantize_hand_blocks_bit_exact():
    cases = _golden_blocks()
    w = np.stack([c["w"] for c in cases])
    got = gpu_quantize(w).cpu().numpy()
    for i, c in enumerate(cases):
        np.testing.assert_array_equal(got[i], c["bytes"], err_msg=c["name"])


@pytest.mark.parametrize("rows,k,scale", [(576, 576, 0.02), (1536, 576, 0.02), (576, 1536, 0.02),
                                          (49152, 576, 0.02), (7, 32, 3.0), (33, 96, 1e-3),
                                          (64, 4096, 0.02)])
def test_quantize_bit_exact_vs_oracle(rows, k, scale):
    w = synth.normal_f32((rows, k), 42, rows * 7 + k, std=scale)
    w[0, :32] = 0.0                          # an all-zero block
    w[min(1, rows - 1), 32 - 1] = 1e-30      # tiny values
    np.testing.assert_array_equal(gpu_quantize(w).cpu().numpy(), O.quantize_q8_0(w))


def test_quantize_ties_and_extremes():
    rng = np.random.default_rng(0)
    # exact half-way ratios: w = (j + 0.5) * d for d = amax/127 with amax a power of two
    amax = np.float32(1.0)
    d = np.float32(amax / np.float32(127))
    blocks = []
    for j in range(0, 126, 4):
        b = np.zeros(32, np.float32)
        b[0] = amax
        b[1:5] = np.float32((np.arange(j, j + 4) + 0.5) * np.float64(d))
        b[5:9] = -b[1:5]
        b[9:] = rng.uniform(-1, 1, 23).astype(np.float32)
        blocks.append(b)
    w = np.stack(blocks)
    np.testing.assert_array_equal(gpu_quantize(w).cpu().numpy(), O.quantize_q8_0(w))


# ------------------------------------------------------------------ matmul

def _packed(wq_dev, rows, k):
    B = binding()
    packed = torch.empty(B.llama_q8_packed_bytes(rows, k), dtype=torch.uint8, device="cuda")
    B.llama_q8_pack(wq_dev, rows, k, packed)
    return packed


def _on_tensor_cores(rows, k, m, path):
    """The library's choice for m > 1 rows (llama_q8.h, LQ8_MATMUL_*)."""
    if path != "auto":
        return path == "tc"
    return m > 16


def _matmul_case(rows, k, m, seed, path="auto"):
    B = binding()
    flags = {"auto": 0, "tc": B.LQ8_MATMUL_TENSOR_CORES, "cc": B.LQ8_MATMUL_CUDA_CORES}[path]
    w = synth.weight_matrix_f32(rows, k, seed, stream=rows + k)
    x = synth.normal_f32((m, k), seed, stream=m * 131 + k)
    wq = gpu_quantize(w)
    np.testing.assert_array_equal(wq.cpu().numpy(), O.quantize_q8_0(w))
    packed = _packed(wq, rows, k)
    dx = to_dev(x)
    dy = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    B.llama_q8_matmul_ex(packed, rows, k, dx, m, dy, flags)
    torch.cuda.synchronize()
    got = dy.cpu().numpy().astype(np.float64)
    wd = O.dequantize_q8_0(O.quantize_q8_0(w), rows, k).astype(np.float64)
    ref = x.astype(np.float64) @ wd.T
    mag = np.abs(x.astype(np.float64)) @ np.abs(wd).T
    # f32 accumulation: the matrix-vector kernel sums 32-code blocks, then at
    # most k/256 blocks per warp, then 8 warp partials; the matrix-matrix
    # kernel sums the k products in one chain. Bound = (chain + 8) u sum|w x|.
    # On the tensor cores (codes times x scaled per token row by a power of two
    # and split into f16 hi and lo, block sums scaled by d) each product
    # carries at most 2^-22 relative error (and 2^-39 of its row's largest
    # |x|) on top of the f32 accumulation.
    chain = (k // 256 + 40) if m == 1 else (k + 8)
    split = 2.0 ** -19 if (m > 1 and _on_tensor_cores(rows, k, m, path)) else 0.0
    tol = ((chain + 8) * U + split) * mag + 1e-30
    assert np.all(np.isfinite(got))
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} elements off; max err {np.max(np.abs(got - ref))}"


@pytest.mark.parametrize("rows,k", [(576, 576), (192, 576), (1536, 576), (576, 1536), (49152, 576)])
@pytest.mark.parametrize("m", [1, 8, 203])
def test_matmul_linear_sweep_135m(rows, k, m):
    _matmul_case(rows, k, m, seed=2)


@pytest.mark.parametrize("rows,k", [(4096, 4096), (14336, 4096), (4096, 14336)])
def test_matvec_7b_shapes(rows, k):
    _matmul_case(rows, k, 1, seed=3)


@pytest.mark.parametrize("rows,k,m", [(1, 32, 1), (33, 64, 1), (7, 32, 3), (100, 96, 65), (31, 4096, 2),
                                      (16, 32, 17), (130, 64, 128), (96, 4096, 129), (256, 2048, 300)])
def test_matmul_ragged_edges(rows, k, m):
    _matmul_case(rows, k, m, seed=4)


@pytest.mark.parametrize("rows,k,m", [(576, 1536, 13), (960, 576, 16), (33, 96, 5), (4096, 14336, 16),
                                      (14336, 4096, 8), (49152, 576, 2)])
def test_matmul_few_rows(rows, k, m):
    """2..16 token rows: every weight tile streamed once for all rows, the block
    range split over a cluster when the rows' slices of x need it (k = 14336)."""
    _matmul_case(rows, k, m, seed=6)


@pytest.mark.parametrize("rows,k,m", [(960, 576, 203), (3072, 576, 203), (576, 1536, 203), (576, 576, 17),
                                      (100, 96, 65), (4096, 4096, 40), (33, 14336, 31)])
@pytest.mark.parametrize("path", ["cc", "tc"])
def test_matmul_both_kernels_many_rows(rows, k, m, path):
    """More than 16 token rows through each kernel, forced by flag: the
    CUDA-core kernel in chunks of 16 rows (a ragged last chunk everywhere
    here; 14336-wide rows split over a cluster) and the tensor cores, at the
    135M prefill shapes of a 203-token prompt and ragged small shapes."""
    _matmul_case(rows, k, m, seed=8, path=path)


def test_matmul_path_flags_rejected_together():
    B = binding()
    rows, k, m = 64, 64, 20
    packed = _packed(gpu_quantize(synth.weight_matrix_f32(rows, k, 9)), rows, k)
    dx = torch.zeros((m, k), dtype=torch.float32, device="cuda")
    dy = torch.zeros((m, rows), dtype=torch.float32, device="cuda")
    with pytest.raises(B.Q8Error) as e:
        B.llama_q8_matmul_ex(packed, rows, k, dx, m, dy, B.LQ8_MATMUL_TENSOR_CORES | B.LQ8_MATMUL_CUDA_CORES)
    assert e.value.status == B.LQ8_ERR_ARG
    rows, k = 64, 16928  # above the CUDA-core kernel's 16896 for chunks of 16 rows
    packed = _packed(gpu_quantize(synth.weight_matrix_f32(rows, k, 9)), rows, k)
    dx = torch.zeros((m, k), dtype=torch.float32, device="cuda")
    with pytest.raises(B.Q8Error) as e:
        B.llama_q8_matmul_ex(packed, rows, k, dx, m, dy, B.LQ8_MATMUL_CUDA_CORES)
    assert e.value.status == B.LQ8_ERR_UNSUPPORTED


def test_matmul_early_weights_chain_equals_serial_calls():
    """A chain of matrix-vector calls whose weight streams start before the
    previous call ends (each call reading the previous call's output) gives
    the same bytes as the same calls made one at a time."""
    B = binding()
    rows = k = 1024
    mats = []
    for i in range(3):
        w = synth.weight_matrix_f32(rows, k, 6, stream=i)
        mats.append(_packed(gpu_quantize(w), rows, k))
    x0 = to_dev(synth.normal_f32((1, k), 6, 9))
    ys = [torch.empty((1, rows), dtype=torch.float32, device="cuda") for _ in range(6)]

    def run(flags):
        src = x0
        for i in range(6):
            B.llama_q8_matmul_ex(mats[i % 3], rows, k, src, 1, ys[i], flags)
            src = ys[i]
        torch.cuda.synchronize()
        return [y.cpu().numpy().copy() for y in ys]

    serial = run(0)
    chained = run(B.LQ8_MATMUL_EARLY_WEIGHTS)
    for a, b in zip(serial, chained):
        np.testing.assert_array_equal(a, b)
    with pytest.raises(B.Q8Error):
        B.llama_q8_matmul_ex(mats[0], rows, k, x0, 1, ys[0], 8)  # an unknown flag bit


@pytest.mark.parametrize("rows,k", [(4096, 4096), (6144, 4096), (4096, 14336)])
def test_matmul_tensor_core_7b_prefill_shapes(rows, k):
    assert _on_tensor_cores(rows, k, 512, "auto")
    _matmul_case(rows, k, 512, seed=5)


@pytest.mark.parametrize("rows,k,m", [(256, 512, 40), (4096, 256, 300)])
def test_matmul_tensor_core_split_precision_one_hot(rows, k, m):
    """Weight rows with a single nonzero: every output is one product w * x
    with no accumulation error, so the tensor-core bound of a single product
    must hold element by element: 2^-22 relative for the f16 hi + lo split of
    the activation scaled by its row's power of two (taken here as 2^-21, for
    the one f32 rounding of the product), plus 2^-39 of the row's largest |x|
    times |w| where the lo part falls below the f16 normal range. A split
    whose lo part were dropped or misplaced, a row scale not undone, or a
    block scale applied to the wrong row or block would leave errors near
    2^-11 or worse."""
    B = binding()
    cols = (np.arange(rows) * 37 + 5) % k
    w = np.zeros((rows, k), np.float32)
    w[np.arange(rows), cols] = synth.normal_f32((rows,), 7, 1)
    x = synth.normal_f32((m, k), 7, 2)
    wq = gpu_quantize(w)
    np.testing.assert_array_equal(wq.cpu().numpy(), O.quantize_q8_0(w))
    packed = _packed(wq, rows, k)
    dy = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    B.llama_q8_matmul_ex(packed, rows, k, to_dev(x), m, dy, B.LQ8_MATMUL_TENSOR_CORES)
    torch.cuda.synchronize()
    got = dy.cpu().numpy().astype(np.float64)
    wd = O.dequantize_q8_0(O.quantize_q8_0(w), rows, k).astype(np.float64)
    wcol = wd[np.arange(rows), cols][None, :]
    ref = x.astype(np.float64)[:, cols] * wcol
    rmax = np.abs(x.astype(np.float64)).max(axis=1, keepdims=True)  # each token row's largest |x|
    err = np.abs(got - ref)
    bound = 2.0 ** -21 * np.abs(ref) + 2.0 ** -39 * np.abs(wcol) * rmax
    assert np.all(err <= bound), float(np.max(err / np.maximum(np.abs(ref), 1e-30)))
    assert np.mean(err <= 2.0 ** -21 * np.abs(ref)) > 0.999  # the bulk to 2^-21 relative


def test_matmul_tensor_core_row_scales():
    """Token rows whose magnitudes span 1e-30 .. 1e30, and an all-zero row, in
    one product: each row's power of two comes from its own largest |x|, so
    every row keeps the same relative accuracy (the bound of the other
    tensor-core cases, relative to that row's sum |w x|) and the zero row
    gives exact zeros. A scale taken from another row, or one not undone,
    would put rows off by many orders of magnitude or overflow the f16 split."""
    B = binding()
    rows, k, m = 192, 1024, 40
    w = synth.weight_matrix_f32(rows, k, 12, stream=rows + k)
    x = synth.normal_f32((m, k), 12, 1)
    row_scale = np.array([1e-30, 1e-12, 1e-3, 1.0, 1e3, 1e12, 1e30, 0.0], np.float32)
    x = (x * row_scale[np.arange(m) % row_scale.size][:, None]).astype(np.float32)
    wq = gpu_quantize(w)
    packed = _packed(wq, rows, k)
    dy = torch.full((m, rows), float("nan"), dtype=torch.float32, device="cuda")
    B.llama_q8_matmul_ex(packed, rows, k, to_dev(x), m, dy, B.LQ8_MATMUL_TENSOR_CORES)
    torch.cuda.synchronize()
    got = dy.cpu().numpy().astype(np.float64)
    wd = O.dequantize_q8_0(O.quantize_q8_0(w), rows, k).astype(np.float64)
    ref = x.astype(np.float64) @ wd.T
    mag = np.abs(x.astype(np.float64)) @ np.abs(wd).T
    tol = ((k + 16) * U + 2.0 ** -19) * mag
    assert np.all(np.isfinite(got))
    zero_rows = np.arange(m) % row_scale.size == row_scale.size - 1
    assert np.all(got[zero_rows] == 0.0)
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{bad.sum()} elements off"


# ------------------------------------------------------------------ attention

def _attention_case(T, index_pos, nh, nkv, hd, stride, seed, entry="attention"):
    B = binding()
    kv_len = index_pos + T
    q = synth.normal_f32((T, nh, hd), seed, 1)
    kc = synth.normal_f32((nkv, stride, hd), seed, 2)
    vc = synth.normal_f32((nkv, stride, hd), seed, 3)
    kc[:, kv_len:] = np.nan  # positions past kv_len must not be read
    vc[:, kv_len:] = np.nan
    ws_bytes = B.llama_q8_attention_workspace_bytes(nh, nkv, hd, stride)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda")
    out = torch.full((T, nh, hd), float("nan"), dtype=torch.float32, device="cuda")
    dq, dk, dv = to_dev(q), to_dev(kc), to_dev(vc)
    if entry == "attention":
        B.llama_q8_attention(dq, dk, dv, T, index_pos, nh, nkv, hd, stride, out, ws, ws_bytes)
    else:
        B.llama_q8_attention_decode(dq, dk, dv, kv_len, nh, nkv, hd, stride, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    k = np.transpose(kc[:, :kv_len], (1, 0, 2))
    v = np.transpose(vc[:, :kv_len], (1, 0, 2))
    mask = None if T == 1 else O.build_causal_mask(T, index_pos)
    ref = O.attention(q, k, v, mask)
    # Score error <= hd u sum|q k| * scale propagates through exp; the output
    # is a convex combination of v rows: tolerance 2e-4 max|v| covers the
    # worst case for N(0,1) inputs at hd <= 128.
    tol = 2e-4 * float(np.max(np.abs(v)))
    assert np.all(np.isfinite(got))
    err = float(np.max(np.abs(got.astype(np.float64) - ref)))
    assert err <= tol, (err, tol)
    # the workspace counters are left at zero for the next call
    assert int(ws[:4 * nkv].view(torch.int32).abs().sum().item()) == 0


@pytest.mark.parametrize("kv_len", [1, 32, 63, 64, 65, 256, 331, 1024, 4096])
def test_attention_decode_135m(kv_len):
    _attention_case(1, kv_len - 1, 9, 3, 64, 4096, seed=kv_len)


@pytest.mark.parametrize("kv_len", [32, 1024, 4096])
def test_attention_decode_7b(kv_len):
    _attention_case(1, kv_len - 1, 32, 8, 128, 4096, seed=kv_len + 1)


# 16 query rows per CTA for these; (1100, 0) and (1030, 7) give 64 rows per CTA
# prompts whose 16-row tiles leave SMs idle split each tile's keys over a
# cluster: (203, 0) over 2 CTAs, (64, 200) over 4, (64, 512) over 8 at the 135M
# shape; (64, 512) over 2, (16, 100) over 4, (16, 1000) over 8 at the 7B shape
@pytest.mark.parametrize("T,index_pos", [(203, 0), (64, 512), (64, 200), (2, 0), (13, 33), (33, 0), (1100, 0),
                                         (1030, 7)])
def test_attention_prefill_135m(T, index_pos):
    _attention_case(T, index_pos, 9, 3, 64, 4096, seed=T + index_pos)


@pytest.mark.parametrize("T,index_pos", [(512, 0), (64, 512), (5, 8), (300, 100), (16, 100), (16, 1000)])
def test_attention_prefill_7b(T, index_pos):
    _attention_case(T, index_pos, 32, 8, 128, 4096, seed=T * 3 + index_pos)


@pytest.mark.parametrize("kv_len", [1, 5, 8, 9, 63, 64, 65, 331, 513, 1024, 4096])
def test_attention_decode_cluster_135m(kv_len):
    _attention_case(1, kv_len - 1, 9, 3, 64, 4096, seed=kv_len + 7, entry="decode")


@pytest.mark.parametrize("kv_len", [1, 32, 768, 1024, 4096])
def test_attention_decode_cluster_7b(kv_len):
    _attention_case(1, kv_len - 1, 32, 8, 128, 4096, seed=kv_len + 9, entry="decode")


@pytest.mark.parametrize("nh,nkv,hd,kv_len", [(4, 4, 64, 100), (8, 1, 128, 777), (16, 2, 64, 4095),
                                             (6, 3, 128, 17), (8, 8, 128, 2048), (9, 3, 64, 512)])
def test_attention_decode_cluster_group_sizes(nh, nkv, hd, kv_len):
    """Groups of 1, 2 and 8 query heads per KV head, position counts on and off
    the 16-CTA x 32-position grid."""
    _attention_case(1, kv_len - 1, nh, nkv, hd, 4096, seed=nh * 7 + kv_len, entry="decode")


def test_attention_decode_rejects_unaligned_cache():
    B = binding()
    q = torch.zeros(9 * 64, dtype=torch.float32, device="cuda")
    kv = torch.zeros(3 * 64 * 64 + 1, dtype=torch.float32, device="cuda")
    out = torch.zeros(9 * 64, dtype=torch.float32, device="cuda")
    with pytest.raises(B.Q8Error) as e:
        B.llama_q8_attention_decode(q, kv[1:], kv[1:], 10, 9, 3, 64, 64, out)
    assert e.value.status == B.LQ8_ERR_ARG


def test_attention_two_calls_reuse_workspace():
    for kv in (700, 130):
        _attention_case(1, kv - 1, 9, 3, 64, 1024, seed=kv)


# ------------------------------------------------------------------ failure path

def test_bounded_wait_times_out_and_device_stays_usable():
    """A kernel waiting on a barrier that nothing completes gives up after the
    library's ~1 s limit, records its code, and the context keeps working."""
    B = binding()
    import time
    t0 = time.perf_counter()
    code = B.llama_q8_selftest_wait_timeout()
    elapsed = time.perf_counter() - t0
    assert code == 41
    assert 0.5 < elapsed < 30.0
    # the device still computes correctly afterwards
    _matmul_case(64, 64, 1, seed=8)
    torch.cuda.synchronize()
