"""Pins for the oracle's RMSNorm statistic, SiLU(g)*u, and the bf16 projection.

RMSNorm's r is compared with a 60-digit evaluation of 1/sqrt(mean(x^2)+eps)
rounded correctly to f32; SiLU with closed forms and a high-precision
evaluation; the bf16 projection with a numpy f64 matmul of the decoded values.
"""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

EPS = 1e-6


def _correct_f32(v_mp, mp):
    """Nearest f32 to the mpmath value v_mp (ties cannot occur here)."""
    c = np.float32(float(v_mp))
    cands = [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))]
    return min(cands, key=lambda f: abs(mp.mpf(float(f)) - v_mp))


def _r_exact(x, eps, mp):
    with mp.workdps(60):
        s = mp.fsum(mp.mpf(float(v)) ** 2 for v in x)
        return _correct_f32(1 / mp.sqrt(s / len(x) + mp.mpf(float(np.float32(eps)))), mp)


def test_rms_inv_is_correctly_rounded(orc):
    mp = pytest.importorskip("mpmath")
    for seed, k in [(0, 1024), (1, 2560), (2, 3584), (3, 32)]:
        x = synth.f32_normal(seed, 0, (k,))
        assert orc.rms_inv(x, EPS) == _r_exact(x, EPS, mp), (seed, k)


@pytest.mark.parametrize("c", [1.0, 0.5, 3.0, 1e-3])
def test_rms_inv_constant_vector_closed_form(orc, c):
    mp = pytest.importorskip("mpmath")
    x = np.full(1024, c, np.float32)
    with mp.workdps(60):
        cc = mp.mpf(float(np.float32(c)))
        want = _correct_f32(1 / mp.sqrt(cc * cc + mp.mpf(float(np.float32(EPS)))), mp)
    assert orc.rms_inv(x, EPS) == want


def test_rmsnorm_quantize_composes_norm_then_quantize(orc):
    x = synth.f32_normal(4, 0, (1024,))
    g = synth.f32_normal(4, 1, (1024,), 1.0, 0.1)
    q, d, r, xh = orc.rmsnorm_quantize(x, g, EPS)
    assert r == orc.rms_inv(x, EPS)
    # x_hat = (x * r) * gamma, two f32 roundings, no fused multiply-add
    assert np.array_equal(xh, (x * np.float32(r)) * g)
    q2, d2 = orc.quantize_q8_0(xh[None, :])
    assert np.array_equal(q, q2[0]) and np.array_equal(d, d2[0])


def test_rmsnorm_scale_invariance_without_eps(orc):
    """With eps = 0, r(4x) = r(x)/4 exactly, so x_hat, q and d are unchanged."""
    x = synth.f32_normal(5, 0, (1024,))
    g = synth.f32_normal(5, 1, (1024,), 1.0, 0.1)
    q, d, r, xh = orc.rmsnorm_quantize(x, g, 0.0)
    q4, d4, r4, xh4 = orc.rmsnorm_quantize(x * np.float32(4), g, 0.0)
    assert r4 == r / 4
    assert np.array_equal(xh4, xh) and np.array_equal(q4, q) and np.array_equal(d4, d)


def test_silu_mul_closed_forms(orc):
    mp = pytest.importorskip("mpmath")
    g = synth.normal(6, 0, 200) * 8.0
    u = synth.normal(6, 1, 200)
    h = orc.silu_mul(g, u)
    one = orc.silu_mul(g, np.ones_like(g))
    neg = orc.silu_mul(-g, np.ones_like(g))
    # silu(g) - silu(-g) = g
    assert np.allclose(one - neg, g, rtol=0, atol=1e-12 * np.abs(g).max())
    assert orc.silu_mul(np.zeros(1), np.ones(1))[0] == 0.0
    # large g: silu(g) -> g; very negative: -> 0
    assert orc.silu_mul(np.array([40.0]), np.ones(1))[0] == 40.0
    assert abs(orc.silu_mul(np.array([-40.0]), np.ones(1))[0]) < 1e-15
    with mp.workdps(40):
        for gi, ui, hi in zip(g[:50], u[:50], h[:50]):
            want = mp.mpf(gi) / (1 + mp.exp(-mp.mpf(gi))) * mp.mpf(ui)
            assert abs(mp.mpf(hi) - want) <= abs(want) * 1e-14 + 1e-300


def test_bf16_gemv_without_norm_matches_f64_matmul(orc):
    case = synth.bf16_case(7, n_rows=64, k=256)
    w = (case["w"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    x = (case["x"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y, a, xh, r = orc.gemv_bf16(case["w"], case["x"], None, EPS)
    assert np.array_equal(xh, case["x"]) and r == 1.0
    assert np.allclose(y, w @ x, rtol=0, atol=1e-13 * a.max())
    assert np.allclose(a, np.abs(w) @ np.abs(x), rtol=1e-13)


def test_bf16_gemv_norm_input(orc):
    torch = pytest.importorskip("torch")
    mp = pytest.importorskip("mpmath")
    case = synth.bf16_case(8, n_rows=16, k=2560)
    y, a, xh, r = orc.gemv_bf16(case["w"], case["x"], case["gamma"], EPS)
    xf = (case["x"].astype(np.uint32) << 16).view(np.float32)
    gf = (case["gamma"].astype(np.uint32) << 16).view(np.float32)
    assert r == _r_exact(xf, EPS, mp)
    t = (xf * np.float32(r)) * gf
    want = torch.from_numpy(t).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(xh, want)
    w = (case["w"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xv = (xh.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.allclose(y, w @ xv, rtol=0, atol=1e-13 * a.max())
