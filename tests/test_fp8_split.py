"""The two-term e4m3 split used by the tensor-memory consumer's FP8 MMAs
(pa_tc.cuh: e4m3_lead), restated with numpy and checked against torch's
e4m3 (float8_e4m3fn) cast, which rounds to nearest-even with saturation.

A value x is carried as hi + lo with hi = x rounded to 4 significant bits
(0 below 2^-6) and lo = e4m3(x - hi). The claims the kernel relies on:
hi is exactly representable in e4m3 over the range the kernel feeds it
(|x| in [2^-6, 448]); hi + lo reproduces x within 2^-8 relative for
|x| >= 2^-2 (lo is then a normal e4m3 value), and within 2^-10 absolute
below (lo falls to e4m3's subnormal step 2^-9). Q rows are scaled to a
maximum in [128, 256), so the absolute floor is below 2^-17 of a row's
maximum; P lies in (0, 2^8] against row sums of at least 1.
"""

import numpy as np
import torch


def e4m3_lead(x):
    x = np.asarray(x, dtype=np.float32)
    ax = np.abs(x)
    u = ax.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFFF + ((u >> 20) & 1)) & 0xFFF00000
    lead = u.astype(np.uint32).view(np.float32)
    lead = np.where(ax < 0.015625, np.float32(0), lead)
    return np.copysign(lead, x).astype(np.float32)


def e4m3(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.float8_e4m3fn).to(torch.float32).numpy()


def test_lead_is_exact_in_e4m3():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.uniform(2.0 ** -6, 448.0, 200000), -rng.uniform(2.0 ** -6, 448.0, 200000),
                        2.0 ** np.arange(-6, 9, dtype=np.float64)]).astype(np.float32)
    hi = e4m3_lead(x)
    assert np.array_equal(e4m3(hi), hi)


def test_lead_rounds_to_nearest_even_at_four_bits():
    # 1 + 1/16 is halfway between 1 and 1.125: even mantissa (1.0) wins;
    # 1.125 + 1/16 is halfway between 1.125 and 1.25: 1.25 (even) wins
    assert e4m3_lead([1.0625, 1.1875, 1.07])[0] == 1.0
    assert e4m3_lead([1.1875])[0] == 1.25
    assert e4m3_lead([1.07])[0] == 1.125
    assert e4m3_lead([0.01])[0] == 0.0


def test_two_term_sum_precision():
    rng = np.random.default_rng(1)
    x = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(256.0), 400000)).astype(np.float32)
    x = np.concatenate([x, -x])
    hi = e4m3_lead(x)
    lo = e4m3(x - hi)
    err = np.abs((hi.astype(np.float64) + lo) - x)
    big = np.abs(x) >= 2.0 ** -2
    assert np.all(err[big] <= 2.0 ** -8 * np.abs(x[big]))
    assert np.all(err[~big] <= 2.0 ** -10)


def test_bf16_query_rows_scaled_into_range_are_nearly_exact():
    """A BF16 row scaled by a power of two to a maximum in [128, 256) keeps
    every element within 2^-8 relative (2^-10 absolute below 2^-2), and
    most elements exactly."""
    rng = np.random.default_rng(2)
    q = torch.from_numpy(rng.standard_normal((64, 128)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    amax = np.abs(q).max(axis=1, keepdims=True)
    ex = 7 - np.floor(np.log2(amax))
    v = (q * 2.0 ** ex).astype(np.float32)
    hi = e4m3_lead(v)
    lo = e4m3(v - hi)
    big = np.abs(v) >= 2.0 ** -2
    err = np.abs(hi.astype(np.float64) + lo - v)
    assert np.all(err[big] <= 2.0 ** -8 * np.abs(v[big]))
    assert np.all(err[~big] <= 2.0 ** -10)
    assert np.mean(err == 0) > 0.9
