"""Pins for the oracle's block rotation (orc_hadamard128).

"Filling in the blanks: Inference using Phobos", PrismML Ternary-Bonsai-2-27B: a
Hadamard matrix transform rotates the activation over the format's block, and the
rotated activation is computed once and shared by the projections that read it.
The transform is pinned to scipy's Hadamard matrix (Sylvester construction, a
library routine), to its algebra (H H^T = 128 I, Parseval) and to closed forms.
"""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth


def test_matches_scipy_hadamard(orc):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(128).astype(np.float64)
    x = synth.f32_normal(0, 91, (4 * 128,))
    z = orc.hadamard128(x)
    ref = (H @ x.astype(np.float64).reshape(4, 128).T).T.ravel()
    # both are f64 sums of the same 128 terms in different orders
    assert np.max(np.abs(z - ref) / np.repeat(np.abs(x).reshape(4, 128).sum(1), 128)) < 1e-14
    # with small integers every sum is exact, so the two agree bit for bit
    xi = synth.uniform_int(0, 92, 3 * 128, -1000, 1000).astype(np.float32)
    zi = orc.hadamard128(xi)
    assert np.array_equal(zi, (H @ xi.astype(np.float64).reshape(3, 128).T).T.ravel())


def test_twice_is_128_times_identity(orc):
    xi = synth.uniform_int(0, 93, 2 * 128, -500, 500).astype(np.float32)
    z = orc.hadamard128(xi)
    assert np.all(np.abs(z) < 2 ** 24)  # exact in f32 below
    zz = orc.hadamard128(z.astype(np.float32))
    assert np.array_equal(zz, 128.0 * xi.astype(np.float64))


def test_parseval_and_closed_forms(orc):
    x = synth.f32_normal(0, 94, (128,))
    z = orc.hadamard128(x)
    assert abs(np.dot(z, z) - 128.0 * np.dot(x.astype(np.float64), x)) < 1e-9 * np.dot(z, z)
    c = np.full(256, 0.75, np.float32)  # a constant block: all of it in entry 0
    zc = orc.hadamard128(c)
    expect = np.zeros(256)
    expect[0] = expect[128] = 96.0
    assert np.array_equal(zc, expect)
    e = np.zeros(128, np.float32)  # one-hot at j: entry i is +1 or -1, +1 at i = 0 and at i = j with even weight
    e[5] = 1.0
    ze = orc.hadamard128(e)
    assert np.all(np.abs(ze) == 1.0) and ze[0] == 1.0 and ze.sum() == 0.0
    assert ze[5] == 1.0 and ze[1] == -1.0 and ze[4] == -1.0  # popcount(5&5)=2, (1&5)=1, (4&5)=1


def test_blocks_are_independent(orc):
    x = synth.f32_normal(0, 95, (3 * 128,))
    z = orc.hadamard128(x)
    for b in range(3):
        assert np.array_equal(z[128 * b:128 * (b + 1)], orc.hadamard128(x[128 * b:128 * (b + 1)]))


def test_rotation_preserves_the_product(orc):
    """y = W x_hat equals (W H^T / 128)(H x_hat): a projection of the rotated
    activation with weights rotated once at load time is the same product."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = scipy_linalg.hadamard(128).astype(np.float64)
    x = synth.f32_normal(0, 96, (256,))
    gamma = synth.f32_normal(0, 97, (256,), 1.0, 0.1)
    z, a, r, xh = orc.rmsnorm_hadamard(x, gamma, 1e-6)
    W = synth.f32_normal(0, 98, (8, 256)).astype(np.float64)
    Hb = np.kron(np.eye(2), H)  # block-diagonal rotation over the two blocks
    y = W @ xh.astype(np.float64)
    yr = (W @ Hb.T / 128.0) @ z
    assert np.max(np.abs(y - yr)) < 1e-12 * np.max(np.abs(W) @ np.abs(xh))
    assert np.all(a >= np.abs(z))


def test_rotation_spreads_an_outlier(orc):
    """The purpose the pages give the rotation: with one large value in a block,
    Q8_0 of the rotated block loses less (relative to the block's norm, which the
    rotation preserves up to the factor sqrt(128)) than Q8_0 of the block itself."""
    x = synth.f32_normal(0, 99, (1024,))
    x[200] = 60.0
    x[777] = -45.0
    gamma = np.ones(1024, np.float32)
    z, _, _, xh = orc.rmsnorm_hadamard(x, gamma, 1e-6)

    def rel_err(v):
        q, d = orc.quantize_q8_0(v.astype(np.float32)[None, :])
        deq = q[0].astype(np.float64) * np.repeat(orc.f16_bits_to_f64(d[0]), 32)
        return np.linalg.norm(deq - v) / np.linalg.norm(v)

    assert rel_err(z) < 0.5 * rel_err(xh.astype(np.float64))
