"""Pins for the oracle's decode feed-forward composite (orc_decode_ffn) and its
residual add (orc_residual_add).

"Filling in the blanks: Inference using Phobos", Fast Decode: the residual add is
folded into the last matmul; the activation is quantized once and shared by the
stacked projections.  The composite only wires functions that are pinned on their
own (test_oracle_gemv.py, test_oracle_quantize.py, test_oracle_norm_bf16.py);
these tests pin the wiring and the add with cases whose results are known
without the oracle: a down projection of zeros, a one-hot down projection with
unit scales, and hand sums.
"""

import numpy as np

from block_quantized_decode_rmsnorm_gb300 import synth

EPS = 1e-6


def test_residual_add_hand_values(orc):
    res = np.array([1.5, -2.25, 0.0, 3.0e-8], np.float32)
    y = np.array([2.0 ** -30, 3.0, -0.0, -3.0e-8], np.float64)
    out = orc.residual_add(res, y)
    expect = np.array([1.5 + 2.0 ** -30, 0.75, 0.0, float(np.float32(3.0e-8)) - 3.0e-8])
    assert np.array_equal(out, expect)


def _small_case(hidden=256, ffn=512, seed=7):
    return synth.ffn_case(seed, hidden, ffn)


def test_decode_ffn_zero_down_is_identity(orc):
    c = _small_case()
    dn_qs = np.zeros_like(c["dn_qs"])
    r = orc.decode_ffn(c["x"], c["gamma"], EPS, c["gu_qs"], c["gu_d"], dn_qs, c["dn_d"])
    assert np.array_equal(r["out64"], c["x"].astype(np.float64))
    assert np.array_equal(r["out"], c["x"])


def test_decode_ffn_one_hot_down(orc):
    """Down weights: row n0 has code 1 at position j0 (block 0 of h), every other
    code 0, every scale 1.0.  Then out[n0] = x[n0] + d_h[0] * hq[j0] exactly and
    out[n] = x[n] elsewhere (a dropped or negated residual, or a wrong row or
    block index, fails)."""
    c = _small_case()
    k, F = c["dn_qs"].shape
    n0, j0 = 37, 5
    dn_qs = np.zeros((k, F), np.int8)
    dn_qs[n0, j0] = 1
    dn_d = np.full((k, F // 32), 0x3C00, np.uint16)  # binary16 1.0
    r = orc.decode_ffn(c["x"], c["gamma"], EPS, c["gu_qs"], c["gu_d"], dn_qs, dn_d)
    dh = float(np.array([r["hd"].ravel()[0]], np.uint16).view(np.float16)[0])
    expect = c["x"].astype(np.float64)
    expect[n0] += dh * float(r["hq"].ravel()[j0])
    assert r["hq"].ravel()[j0] != 0
    assert np.array_equal(r["out64"], expect)


def test_decode_ffn_wires_pinned_steps(orc):
    """Each intermediate equals the separately pinned step applied to the previous
    one: RMSNorm + Q8_0, the stacked product (gate rows first), SiLU(g) * u
    rounded once to f32, Q8_0 of h, the down product."""
    c = _small_case(seed=11)
    r = orc.decode_ffn(c["x"], c["gamma"], EPS, c["gu_qs"], c["gu_d"], c["dn_qs"], c["dn_d"])
    q, d, rinv, _ = orc.rmsnorm_quantize(c["x"], c["gamma"], EPS)
    assert np.array_equal(r["xq"], q) and np.array_equal(r["xd"], d) and r["r"] == rinv
    gu, a_gu = orc.gemv_q8_0(c["gu_qs"], c["gu_d"], q, d)
    assert np.array_equal(r["gu64"], gu[0]) and np.array_equal(r["a_gu"], a_gu[0])
    F = c["gu_qs"].shape[0] // 2
    h64 = orc.silu_mul(gu[0, :F], gu[0, F:])
    assert np.array_equal(r["h64"], h64)
    assert np.array_equal(r["h"], h64.astype(np.float32))
    hq, hd = orc.quantize_q8_0(r["h"][None, :])
    assert np.array_equal(r["hq"], hq) and np.array_equal(r["hd"], hd)
    y, a_y = orc.gemv_q8_0(c["dn_qs"], c["dn_d"], hq, hd)
    assert np.array_equal(r["y64"], y[0]) and np.array_equal(r["a_y"], a_y[0])
    assert np.array_equal(r["out64"], orc.residual_add(c["x"], y[0]))
