"""Pins for the oracle's block dots and block-scaled GEMV.

The main pin is a brute-force dequantize-then-matmul in f64 (numpy's float16
decode and f64 matmul, a different algorithm from the oracle's integer block
dot followed by scaling).  When every partial sum is a multiple of one power of
two below 2^53 times that power, both sides are exact and must agree bit for
bit; the test checks that condition before it demands equality.
"""

from fractions import Fraction

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth


def _dequant(qs, d):
    n, k = qs.shape
    scale = d.view(np.float16).astype(np.float64)  # library decode
    return qs.astype(np.float64) * np.repeat(scale, 32, axis=1)


def _exact_sum_guaranteed(wd, xd, a):
    """All terms are integer multiples of 2^emin; if the magnitude sum stays
    below 2^(emin+53), every partial sum in any order is exact in f64."""
    def ulp_exp(d):
        v = d.view(np.float16).astype(np.float64)
        v = v[v != 0]
        _, e = np.frexp(v)
        return int((e - 1 - 10).min())
    emin = ulp_exp(wd) + ulp_exp(xd)
    return float(a.max()) < 2.0 ** (emin + 53)


@pytest.mark.parametrize("n,k,batch", [(7, 32, 1), (13, 64, 3), (40, 96, 2), (256, 1024, 1)])
def test_gemv_equals_bruteforce_dequant_matmul(orc, n, k, batch):
    qs, d = synth.q8_0_weight_planes(n * 7 + k, 10, n, k)
    x = synth.f32_normal(k, 0, (batch, k))
    xq, xd = orc.quantize_q8_0(x)
    y, a = orc.gemv_q8_0(qs, d, xq, xd)
    brute = _dequant(xq, xd) @ _dequant(qs, d).T
    assert _exact_sum_guaranteed(d, xd, a)
    assert np.array_equal(y, brute)
    # a is the sum of the per-block term magnitudes: at least |y|, at most sum |w||x|
    assert np.all(a >= np.abs(y))
    assert np.all(a <= np.abs(_dequant(xq, xd)) @ np.abs(_dequant(qs, d)).T * (1 + 1e-12))


def test_block_dots_against_integer_einsum(orc):
    qs, _ = synth.q8_0_weight_planes(3, 10, 19, 160)
    xq = synth.uniform_int(3, 50, 2 * 160, -127, 127).astype(np.int8).reshape(2, 160)
    s = orc.block_dots(qs, xq)
    want = np.einsum("nbi,xbi->xnb", qs.reshape(19, 5, 32).astype(np.int64), xq.reshape(2, 5, 32).astype(np.int64))
    assert np.array_equal(s, want)
    # extremes: the largest possible block sum fits int32 exactly
    w = np.full((1, 32), -127, np.int8)
    xx = np.full((1, 32), -127, np.int8)
    assert int(orc.block_dots(w, xx)[0, 0, 0]) == 32 * 127 * 127


def test_all_ones_closed_form(orc):
    n, k = 9, 128
    qs, d = synth.q8_0_weight_planes(11, 10, n, k)
    xq, xd = orc.quantize_q8_0(np.ones((1, k), np.float32))
    assert np.all(xq == 127) and np.all(xd == 0x2008)
    y, _ = orc.gemv_q8_0(qs, d, xq, xd)
    dx = Fraction(np.float16(np.uint16(0x2008).view(np.float16)).item())
    for r in range(n):
        exact = Fraction(0)
        for b in range(k // 32):
            dw = Fraction(d[r, b].view(np.float16).item())
            exact += dw * dx * 127 * int(qs[r, 32 * b : 32 * b + 32].astype(np.int64).sum())
        assert y[0, r] == float(exact)


def test_one_hot_closed_form(orc):
    n, k, j, c = 12, 96, 45, 2.75
    qs, d = synth.q8_0_weight_planes(12, 10, n, k)
    x = np.zeros((1, k), np.float32)
    x[0, j] = c
    xq, xd = orc.quantize_q8_0(x)
    assert int(xq[0, j]) == 127 and np.count_nonzero(xq) == 1
    y, _ = orc.gemv_q8_0(qs, d, xq, xd)
    dx = Fraction(np.float16(np.float32(c) / np.float32(127)).item())
    for r in range(n):
        dw = Fraction(d[r, j // 32].view(np.float16).item())
        assert y[0, r] == float(dw * dx * 127 * int(qs[r, j]))


def test_zero_inputs(orc):
    qs, d = synth.q8_0_weight_planes(13, 10, 8, 64)
    xq, xd = orc.quantize_q8_0(np.zeros((1, 64), np.float32))
    y, a = orc.gemv_q8_0(qs, d, xq, xd)
    assert np.all(y == 0) and np.all(a == 0)
    x = synth.f32_normal(13, 0, (1, 64))
    xq, xd = orc.quantize_q8_0(x)
    y, _ = orc.gemv_q8_0(np.zeros_like(qs), d, xq, xd)
    assert np.all(y == 0)


def test_batch_invariance(orc):
    qs, d = synth.q8_0_weight_planes(14, 10, 33, 128)
    x = synth.f32_normal(14, 0, (4, 128))
    xq, xd = orc.quantize_q8_0(x)
    y, _ = orc.gemv_q8_0(qs, d, xq, xd)
    for b in range(4):
        yb, _ = orc.gemv_q8_0(qs, d, xq[b : b + 1], xd[b : b + 1])
        assert np.array_equal(yb[0], y[b])


def test_stacked_gate_up_equals_separate_products(orc):
    """'One level down: #002 the same compiler on a GPU', Emitting for a GPU:
    gate and up are one stacked projection.  The stacked product followed by
    SiLU(g)*u equals the two separate products combined the same way."""
    F, k = 24, 64
    gq, gd = synth.q8_0_weight_planes(15, 10, F, k)
    uq, ud = synth.q8_0_weight_planes(15, 20, F, k)
    x = synth.f32_normal(15, 0, (1, k))
    xq, xd = orc.quantize_q8_0(x)
    st, _ = orc.gemv_q8_0(np.concatenate([gq, uq]), np.concatenate([gd, ud]), xq, xd)
    g, _ = orc.gemv_q8_0(gq, gd, xq, xd)
    u, _ = orc.gemv_q8_0(uq, ud, xq, xd)
    assert np.array_equal(st[0, :F], g[0]) and np.array_equal(st[0, F:], u[0])
    assert np.array_equal(orc.silu_mul(st[0, :F], st[0, F:]), orc.silu_mul(g[0], u[0]))
