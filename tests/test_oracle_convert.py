"""Pins for the oracle's binary16 / bfloat16 converters.

The oracle writes both conversions from the IEEE 754 definition (round to
nearest, ties to even).  These tests tie them to library casts that implement
the same standard: numpy's float16 cast and torch's CPU bfloat16 cast.
"""

import numpy as np
import pytest


def _all_f16_values():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    return bits, vals


def test_f16_decode_all_patterns(orc):
    bits, vals = _all_f16_values()
    got = orc.f16_bits_to_f64(bits)
    nan = np.isnan(vals)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], vals[~nan])


def test_f32_to_f16_at_values_midpoints_and_neighbours(orc):
    """Every finite fp16 value, every midpoint between neighbours, and the f32
    values one ulp either side of each midpoint (the places where a rounding
    mistake shows)."""
    bits, vals = _all_f16_values()
    finite = np.isfinite(vals) & (vals >= 0)
    v = np.unique(vals[finite])
    mids = (v[:-1] + v[1:]) / 2.0  # exact in f32: 12 significant bits
    cand = np.concatenate([v, mids]).astype(np.float32)
    up = np.nextafter(cand, np.float32(np.inf))
    dn = np.nextafter(cand, np.float32(-np.inf))
    xs = np.concatenate([cand, up, dn, np.float32(65520.0)[None], np.float32(65519.996)[None]])
    xs = np.concatenate([xs, -xs])
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_bits(xs)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, (xs[bad[:5]], got[bad[:5]], want[bad[:5]])


def test_f32_to_f16_random_patterns(orc):
    from block_quantized_decode_rmsnorm_gb300 import synth

    z = synth.raw_u64(1234, 7, 1 << 21)
    pats = (z & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    xs = pats.view(np.float32)
    xs = xs[~np.isnan(xs)]
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16_bits(xs)
    assert np.array_equal(got, want)


def test_f32_to_f16_specials(orc):
    cases = [
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (1.0, 0x3C00),
        (65504.0, 0x7BFF),  # largest finite
        (65520.0, 0x7C00),  # halfway to 2^16: ties to even -> overflow
        (2.0 ** -24, 0x0001),  # smallest subnormal
        (2.0 ** -25, 0x0000),  # halfway to it: ties to even -> 0
        (3 * 2.0 ** -26, 0x0001),
        (2.0 ** -14, 0x0400),  # smallest normal
        (float("inf"), 0x7C00),
    ]
    for x, want in cases:
        assert int(orc.f32_to_f16_bits(np.array([x], np.float32))[0]) == want, x
    assert np.isnan(orc.f16_bits_to_f64(orc.f32_to_f16_bits(np.array([np.nan], np.float32))))[0]


def test_f32_to_bf16_against_torch(orc):
    torch = pytest.importorskip("torch")
    from block_quantized_decode_rmsnorm_gb300 import synth

    z = synth.raw_u64(99, 3, 1 << 21)
    pats = (z & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    # add exact ties (low 16 bits = 0x8000) and neighbours: where ties-to-even decides
    ties = (pats & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    pats = np.concatenate([pats, ties, ties + np.uint32(1), ties - np.uint32(1)])
    xs = pats.view(np.float32)
    xs = xs[~np.isnan(xs)]
    want = torch.from_numpy(xs.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = orc.f32_to_bf16_bits(xs)
    assert np.array_equal(got, want)


def test_bf16_specials(orc):
    cases = [
        (1.0, 0x3F80),
        (-2.0, 0xC000),
        (1.0 + 2.0 ** -8, 0x3F80),  # tie, even stays
        (1.0 + 3 * 2.0 ** -8, 0x3F82),  # tie, odd rounds up
        (float(np.finfo(np.float32).max), 0x7F80),  # rounds past the largest bf16
    ]
    for x, want in cases:
        assert int(orc.f32_to_bf16_bits(np.array([x], np.float32))[0]) == want, x
