"""The conversion-free rejection test of the draft step's Gumbel-max race is conservative.

The draft step rejects an element without computing its Gumbel key when 1 - u >= t, where u
is the uniform drawn from the word's top 24 bits, u = (2b + 1) 2^-25 with b = bits >> 8.  It
evaluates the test without an integer-to-float conversion: with f = 1 + floor(b / 2) 2^-23
(the word's top 23 bits placed in a binary32 mantissa), it rejects when fl(t + f) <= 2 - 2^-22.
This must never reject an element that the exact test keeps.  Here both are evaluated in
binary64 on sampled words and thresholds (fl(.) emulated by rounding the exact sum once to
binary32), including thresholds within a few units of 1 - u.
"""
import numpy as np


def _f32_from_bits(x):
    return np.asarray(x, dtype=np.uint32).view(np.float32)


def test_conversion_free_rejection_never_rejects_a_kept_element():
    rng = np.random.default_rng(12)
    n = 2_000_000
    bits = rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32)
    b = (bits >> 8).astype(np.int64)
    w_exact = 1.0 - (2 * b + 1) / 2.0 ** 25  # 1 - u, exact in binary64
    f = _f32_from_bits((bits >> 9) | np.uint32(0x3F800000)).astype(np.float64)
    # thresholds: half at random, half within ~1e-6 (relative) of 1 - u; plus the extremes
    t = np.where(rng.random(n) < 0.5, rng.random(n), w_exact * (1 + rng.normal(0, 1e-6, n)))
    t = np.concatenate([t, np.zeros(4), np.full(4, 1.0), np.full(4, 2.0 ** -30)]).astype(np.float32)
    w_exact = np.concatenate([w_exact, w_exact[:12]])
    f = np.concatenate([f, f[:12]])
    s = (t.astype(np.float64) + f).astype(np.float32)  # one rounding, as the FMA
    edge = np.float32(2.0 - 2.0 ** -22)
    rejected = s <= edge
    exact_rejects = w_exact >= t.astype(np.float64)
    assert not np.any(rejected & ~exact_rejects)
    # and it is not vacuous: nearly every exact rejection away from the boundary survives
    far = np.abs(w_exact - t) > 2.0 ** -21
    assert np.array_equal(rejected[far], exact_rejects[far])


def test_mantissa_bound_on_every_24_bit_value():
    # u - (f - 1) is 2^-25 for even b and 3 * 2^-25 for odd b: below 2^-23 for all b
    b = np.arange(2 ** 24, dtype=np.int64)
    bits = (b << 8).astype(np.uint32)
    f = _f32_from_bits((bits >> 9) | np.uint32(0x3F800000)).astype(np.float64)
    gap = (2 * b + 1) / 2.0 ** 25 - (f - 1.0)
    assert gap.min() > 0 and gap.max() < 2.0 ** -23
