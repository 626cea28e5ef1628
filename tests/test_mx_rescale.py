"""The MXFP4 dequantisation the kernel performs, modelled in NumPy: each token
row is taken in units of its largest block scale 2^(max - 127), and every
block's E2M1 values are multiplied in FP16 by 2^(code - max). The product is
exact while it stays within FP16's subnormal range (blocks up to 2^22 below
the row's largest), and below that the row changes by less than 2^-22 of its
largest element, the bounds the kernel relies on."""

import numpy as np

import pa_workloads as pw


def fp16_factor(delta):
    """2^-delta as the kernel builds it in FP16 (0 beyond 2^-24)."""
    return np.where(delta <= 24, np.exp2(-delta.astype(np.float64)), 0.0).astype(np.float16)


def model_row(codes, X):
    """Kernel-order dequantisation of one row: FP16 values times FP16 factors
    (rounded to FP16), then the row factor 2^(max - 127) in float64."""
    mag = pw.E2M1_GRID[codes & 7].astype(np.float16)
    e = np.where(codes & 8, -mag, mag)
    xmax = X.max()
    f = np.repeat(fp16_factor(xmax - X.astype(np.int64)), 32)
    prod = (e.astype(np.float16) * f).astype(np.float16)  # one FP16 multiply, rounded
    return prod.astype(np.float64) * np.exp2(float(xmax) - 127.0)


def exact_row(codes, X):
    mag = pw.E2M1_GRID[codes & 7].astype(np.float64)
    e = np.where(codes & 8, -mag, mag)
    return e * np.repeat(np.exp2(X.astype(np.float64) - 127.0), 32)


def test_exact_within_range():
    rng = np.random.default_rng(0)
    for _ in range(200):
        codes = rng.integers(0, 16, size=128).astype(np.uint8)
        base = int(rng.integers(60, 190))
        X = (base - rng.integers(0, 23, size=4)).astype(np.uint8)  # blocks up to 2^22 below the largest
        assert np.array_equal(model_row(codes, X), exact_row(codes, X))


def test_bounded_beyond_range():
    rng = np.random.default_rng(1)
    for _ in range(200):
        codes = rng.integers(0, 16, size=128).astype(np.uint8)
        codes[:32] = 7  # the largest block holds 6.0
        base = int(rng.integers(100, 200))
        X = np.array([base, base - rng.integers(23, 60), base - rng.integers(0, 60), base - 40], dtype=np.uint8)
        err = np.abs(model_row(codes, X) - exact_row(codes, X)).max()
        row_max = np.abs(exact_row(codes, X)).max()
        assert err <= row_max * 2.0 ** -22
