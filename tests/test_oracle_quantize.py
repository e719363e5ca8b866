"""Pins for the oracle's Q8_0 activation quantization and weight packing.

Ties the quantizer to hand-derived cases (tests/golden), to the closed-form
bound on its error, and to invariants that a dropped term, a wrong sign or a
wrong rounding mode would break.
"""

import json
import os

import numpy as np

from block_quantized_decode_rmsnorm_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q8_0_quantize_hand_cases.json")


def _pad(vals):
    x = np.zeros(32, np.float32)
    x[: len(vals)] = np.asarray(vals, np.float32)
    return x


def test_hand_cases(orc):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        if c["x"] == "ones":
            x = np.ones(32, np.float32)
            want_q = np.full(32, 127, np.int8)
        else:
            x = _pad(c["x"])
            want_q = np.zeros(32, np.int8)
            want_q[: len(c["q"])] = c["q"]
        q, d = orc.quantize_q8_0(x[None, :])
        assert np.array_equal(q[0], want_q), (c["name"], q[0], want_q)
        assert int(d[0, 0]) == c["d_bits"], (c["name"], int(d[0, 0]))


def test_error_bound_closed_form(orc):
    """|x - d*q| <= d/2 with the f32 scale d = max|x|/127 (plus f32 rounding of
    x/d), and <= d/2 + 127*|d16 - d| with the stored binary16 scale."""
    x = synth.f32_normal(0, 5, (64, 1024))
    q, d16 = orc.quantize_q8_0(x)
    xb = x.reshape(64, 32, 32).astype(np.float64)
    qb = q.reshape(64, 32, 32).astype(np.float64)
    d32 = (np.abs(x.reshape(64, 32, 32)).max(axis=2) / np.float32(127)).astype(np.float64)
    d16v = orc.f16_bits_to_f64(d16.ravel()).reshape(64, 32)
    err32 = np.abs(xb - d32[..., None] * qb)
    # x/d is rounded once in f32: relative 2^-24 of at most 127.5
    assert np.all(err32 <= d32[..., None] * (0.5 + 127.5 * 2.0 ** -24))
    err16 = np.abs(xb - d16v[..., None] * qb)
    assert np.all(err16 <= d32[..., None] * (0.5 + 127.5 * 2.0 ** -24) + 127 * np.abs(d16v - d32)[..., None])
    # the largest magnitude of each block maps to +-127
    idx = np.abs(x.reshape(64, 32, 32)).argmax(axis=2)
    top = np.take_along_axis(qb, idx[..., None], axis=2)[..., 0]
    assert np.all(np.abs(top) == 127)
    assert np.all(np.abs(qb) <= 127)


def test_sign_symmetry_and_power_of_two_scaling(orc):
    x = synth.f32_normal(0, 6, (16, 256))
    q, d = orc.quantize_q8_0(x)
    qn, dn = orc.quantize_q8_0(-x)
    assert np.array_equal(qn, -q)
    assert np.array_equal(dn, d)
    # scaling by 4 scales d by 4 exactly (no binary16 overflow/underflow here)
    q4, d4 = orc.quantize_q8_0(x * np.float32(4.0))
    assert np.array_equal(q4, q)
    assert np.array_equal(orc.f16_bits_to_f64(d4), 4.0 * orc.f16_bits_to_f64(d))


def test_rows_are_independent(orc):
    x = synth.f32_normal(0, 7, (5, 96))
    q, d = orc.quantize_q8_0(x)
    for r in range(5):
        qr, dr = orc.quantize_q8_0(x[r : r + 1])
        assert np.array_equal(qr[0], q[r]) and np.array_equal(dr[0], d[r])


def test_pack_is_byte_permutation(orc):
    blocks, qs, d = synth.q8_0_weight_blocks(0, 40, 37, 96)
    pqs, pd = orc.q8_0_pack(blocks, 37, 96)
    assert np.array_equal(pqs, qs)
    assert np.array_equal(pd, d)
    # first block by hand: bytes 0-1 are the little-endian scale, bytes 2.. the values
    b0 = blocks[0, 0]
    assert int(pd[0, 0]) == int(b0[0]) | (int(b0[1]) << 8)
    assert np.array_equal(pqs[0, :32], b0[2:].view(np.int8))
