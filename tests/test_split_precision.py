"""The prefill's tensor-core operands split every fp32 activation into two fp16 values, hi = fp16(x) and
lo = fp16(x - hi). These host checks pin the precision that split keeps (what lets the tensor-core prefill match
the fp32 oracle within the decode's tolerance): hi + lo recovers x to 2^-21 relative while lo is a normal fp16
(|x| >= 2^-3) and to 2^-25 absolute below (lo then falls into fp16's subnormal range), products of an fp16 weight
with hi or lo are exact in fp32, and a dot product of fp16 weights with the two halves, summed in fp32, stays
within 1e-5 of the sum of |w x| of the fp64 dot product."""
import numpy as np


def split(x):
    hi = x.astype(np.float16)
    lo = (x - hi.astype(np.float32)).astype(np.float16)
    return hi, lo


def test_hi_plus_lo_error_is_2e_21_relative_or_2e_25_absolute():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 8, 200000))).astype(np.float32)
    hi, lo = split(x)
    x64 = x.astype(np.float64)
    err = np.abs(hi.astype(np.float64) + lo.astype(np.float64) - x64)
    big = np.abs(x64) >= 2.0 ** -3
    assert big.sum() > 1000 and (~big).sum() > 1000
    assert np.all(err[big] <= 2.0 ** -21 * np.abs(x64[big]))
    assert np.all(err <= np.maximum(2.0 ** -21 * np.abs(x64), 2.0 ** -25))


def test_fp16_products_with_either_half_are_exact_in_fp32():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal(50000) * 0.02).astype(np.float16)
    hi, lo = split(rng.standard_normal(50000).astype(np.float32))
    for part in (hi, lo):
        p32 = w.astype(np.float32) * part.astype(np.float32)
        p64 = w.astype(np.float64) * part.astype(np.float64)
        np.testing.assert_array_equal(p32.astype(np.float64), p64)


def test_split_dot_product_matches_fp64_to_fp32_rounding():
    rng = np.random.default_rng(2)
    K = 7680
    w = (rng.standard_normal((64, K)) * 0.02).astype(np.float16)
    x = rng.standard_normal(K).astype(np.float32)
    hi, lo = split(x)
    # fp32 accumulation of the two halves, then their sum (the epilogue's hi + lo)
    y = (w.astype(np.float32) @ hi.astype(np.float32)) + (w.astype(np.float32) @ lo.astype(np.float32))
    ref = w.astype(np.float64) @ x.astype(np.float64)
    absdot = np.abs(w.astype(np.float64)) @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(y - ref) <= 1e-5 * absdot)
