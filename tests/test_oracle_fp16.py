"""Pins for the oracle's IEEE binary16 codec.

The codec in oracle.c is written from the format's definition; these tests
compare it with numpy's binary16 conversion (a library routine) over every
bit pattern, on random doubles, and on the tie and overflow boundaries that
round-to-nearest-even fixes.
"""
import numpy as np

import oracle


def test_decode_all_65536_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_encode_roundtrips_every_finite_and_infinite_pattern():
    for b in range(65536):
        x = oracle.half_to_double(b)
        if np.isnan(x):
            assert oracle.double_to_half(x) & 0x7C00 == 0x7C00
            assert oracle.double_to_half(x) & 0x03FF != 0
            continue
        assert oracle.double_to_half(x) == b


def test_encode_matches_numpy_on_random_doubles():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.uniform(-70000, 70000, 200_000),
        rng.standard_normal(200_000),
        rng.standard_normal(200_000) * 1e-5,  # subnormal range
        rng.standard_normal(200_000) * 1e-8,  # underflow to zero
        rng.uniform(-2, 2, 200_000),
    ])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half(v) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_ties_go_to_even_at_every_midpoint():
    # all midpoints between consecutive positive binary16 values, subnormals included
    vals = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (vals[:-1] + vals[1:]) / 2  # exact in fp64
    lo_bits = np.arange(0, 0x7BFF, dtype=np.uint16)
    want = np.where(lo_bits % 2 == 0, lo_bits, lo_bits + 1).astype(np.uint16)
    got = np.array([oracle.double_to_half(m) for m in mids], dtype=np.uint16)
    assert np.array_equal(got, want)
    assert np.array_equal(got, mids.astype(np.float16).view(np.uint16))


def test_overflow_boundary():
    assert oracle.double_to_half(65504.0) == 0x7BFF
    assert oracle.double_to_half(65519.999) == 0x7BFF
    assert oracle.double_to_half(65520.0) == 0x7C00
    assert oracle.double_to_half(-65520.0) == 0xFC00
    assert oracle.double_to_half(float("inf")) == 0x7C00
    assert oracle.double_to_half(-0.0) == 0x8000
    assert oracle.double_to_half(2.0 ** -25) == 0x0000  # tie between 0 and 2^-24 -> even (0)
    assert oracle.double_to_half(3 * 2.0 ** -25) == 0x0002  # tie between 1 and 2 quanta -> 2
