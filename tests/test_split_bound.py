"""The precision bound the tensor-core tests use for one product, derived on
the host: a token row scaled by the power of two that brings its largest |x|
into [2^14, 2^15) and split as x 2^s = hi + lo (both rounded to f16) keeps
each element to 2^-22 relative, or to 2^-25 absolute (2^-39 of the row's
largest |x| once the scale is undone) where lo falls below the f16 normal
range. The codes are exact in f16, so these are the only input roundings of
the product; the GPU tests allow 2^-21 relative (one more f32 rounding) plus
that absolute term. Computed with numpy's IEEE f16 conversions, independently
of the CUDA code."""
import numpy as np


def _row_shift(mx: np.float32) -> int:
    # exponent e with mx in [2^e, 2^(e+1)); s = 14 - e, clamped as the kernels clamp it
    e = int(np.frexp(np.float64(mx))[1]) - 1 if mx > 0 else -127
    return max(-126, min(126, 14 - e))


def _split(row: np.ndarray):
    s = _row_shift(np.max(np.abs(row)))
    xs = (row.astype(np.float64) * 2.0 ** s).astype(np.float32)  # exact: a power of two
    hi = xs.astype(np.float16)
    lo = (xs - hi.astype(np.float32)).astype(np.float16)
    return s, xs, hi, lo


def test_scaled_row_fits_f16_and_split_is_within_bound():
    rng = np.random.default_rng(7)
    for scale in (1e-30, 1e-6, 1.0, 3.0e4, 1e30):
        for n in (32, 576, 4096):
            row = (rng.standard_normal(n) * scale).astype(np.float32)
            row[rng.integers(0, n, 8)] *= np.float32(1e-7)    # small elements: lo leaves the normal range
            s, xs, hi, lo = _split(row)
            mx = float(np.max(np.abs(xs)))
            assert 2.0 ** 14 <= mx < 2.0 ** 15                  # no f16 overflow, full use of the range
            assert np.all(np.isfinite(hi.astype(np.float32)))
            err = np.abs(xs.astype(np.float64) - hi.astype(np.float64) - lo.astype(np.float64))
            bound = 2.0 ** -22 * np.abs(xs.astype(np.float64)) + 2.0 ** -25
            assert np.all(err <= bound), (scale, n, float(np.max(err / bound)))
            # undone: relative to the original row, 2^-22 relative plus 2^-39 of its largest |x|
            rmax = float(np.max(np.abs(row)))
            err_x = err * 2.0 ** -s
            assert np.all(err_x <= 2.0 ** -22 * np.abs(row.astype(np.float64)) + 2.0 ** -39 * rmax * 2.0)


def test_hi_alone_is_not_enough():
    """Without lo the error is ~2^-12 relative: a kernel that dropped lo would
    fail the 2^-21 bound of the GPU tests by far."""
    rng = np.random.default_rng(8)
    row = rng.standard_normal(4096).astype(np.float32)
    s, xs, hi, lo = _split(row)
    rel = np.abs(xs.astype(np.float64) - hi.astype(np.float64)) / np.abs(xs.astype(np.float64))
    assert np.max(rel) > 2.0 ** -13
    assert np.max(rel) <= 2.0 ** -11


def test_zero_row_and_extreme_rows():
    assert _row_shift(np.float32(0.0)) == 126                    # all-zero row: any scale, x is zero
    s, xs, hi, lo = _split(np.zeros(64, np.float32))
    assert not np.any(hi.astype(np.float32)) and not np.any(lo.astype(np.float32))
    assert _row_shift(np.float32(3.0e38)) == 14 - 127            # 2^-113: the scaled maximum stays below 2^15
    assert _row_shift(np.float32(1e-45)) == 126                  # clamped: 2^126 and 2^-126 stay normal
