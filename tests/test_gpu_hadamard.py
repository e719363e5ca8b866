"""GPU parity for the rotated activation: RMSNorm, the order-128 Walsh-Hadamard
rotation of each block of 128, Q8_0 (rmsnorm_hadamard_quantize), and the decode
FFN that shares the rotated codes between its stacked gate|up halves.

"Filling in the blanks: Inference using Phobos", PrismML Ternary-Bonsai-2-27B.

Contract: r bit-exact (the oracle's correctly rounded r); the rotated row z
within the normalised tolerance of the oracle's f64 transform (scale: the sum of
the magnitudes of the 128 terms); the codes and scales bit-exact against the
oracle's quantizer applied to the GPU's z (z is a float reduction whose last bit
depends on the summation order, so a code may legitimately differ from one
quantized from the f64 z exactly at a rounding boundary).
"""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

from ._gpu import Guarded, f16_to_np_bits, need_gpu, to_dev, weight
from ._tol import TOL_Q8, assert_close, silu_scale

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.mark.parametrize("rows,k", [(1, 128), (1, 1024), (3, 1024), (17, 256), (2, 4096), (5, 2560), (1, 65536)])
def test_rotated_quantize_parity(torch, orc, rows, k):
    from block_quantized_decode_rmsnorm_gb300 import api

    x = synth.f32_normal(0, 201 + k, (rows, k))
    if rows > 2:
        x[1, 7] *= 100.0  # an outlier row
        x[2] = 0.0        # a zero row: r = 1/sqrt(eps), everything zero after it
    g = synth.f32_normal(0, 202 + k, (k,), 1.0, 0.1)
    q = Guarded(torch, (rows, k), torch.int8)
    d = Guarded(torch, (rows, k // 32), torch.float16)
    z = Guarded(torch, (rows, k), torch.float32)
    r = Guarded(torch, (rows,), torch.float32)
    api.rmsnorm_hadamard_quantize(to_dev(x, torch), to_dev(g, torch), EPS, q=q.view, d=d.view, z=z.view,
                                  inv_rms=r.view)
    torch.cuda.synchronize()
    for b in (q, d, z, r):
        b.check()
    zg, qg, dg, rg = z.view.cpu().numpy(), q.view.cpu().numpy(), f16_to_np_bits(d.view), r.view.cpu().numpy()
    for i in range(rows):
        z64, a, r64, _ = orc.rmsnorm_hadamard(x[i], g, EPS)
        assert rg[i] == r64, (i, rg[i], r64)
        assert_close(zg[i], z64, a, TOL_Q8, f"z row {i}")
        oq, od = orc.quantize_q8_0(zg[i][None, :])
        assert np.array_equal(qg[i], oq[0]), f"codes row {i}"
        assert np.array_equal(dg[i], od[0]), f"scales row {i}"
    if rows > 2:
        assert not qg[2].any() and not dg[2].any()


def test_rotated_matches_plain_quantize_when_rotation_is_skipped(torch, orc):
    """The norm and the quantizer are the library's existing ones: on a row whose
    rotation is known in closed form (a constant block goes to 128 c at index 0),
    the codes are those of rmsnorm_quantize applied to that closed form."""
    from block_quantized_decode_rmsnorm_gb300 import api

    x = np.full((1, 128), 0.5, np.float32)
    g = np.ones(128, np.float32)
    q, d = api.rmsnorm_hadamard_quantize(to_dev(x, torch), to_dev(g, torch), 0.0)
    torch.cuda.synchronize()
    # r = 2 exactly (mean of squares 0.25), x_hat = 1, z = (128, 0, ..., 0)
    qn = q.cpu().numpy()[0]
    assert qn[0] == 127 and not qn[1:].any()
    assert f16_to_np_bits(d)[0, 0] == orc.f32_to_f16_bits(np.float32(128.0 / 127.0))[0]


def test_rotated_ffn_staged_parity(torch, orc):
    """The decode FFN on the 0.8B shape with the rotated activation shared by the
    stacked gate|up (weights standing for the load-time rotated ones), checked
    stage by stage from the GPU's own intermediates."""
    from block_quantized_decode_rmsnorm_gb300 import api

    c = synth.ffn_case(5)
    F = 3584
    layer = api.FFNLayer(to_dev(c["gamma"], torch), weight(c["gu_qs"], c["gu_d"]), weight(c["dn_qs"], c["dn_d"]))
    buf = api.FFNBuffers.allocate(1024, F, "cuda")
    x = to_dev(c["x"], torch)
    api.decode_ffn_q8_0_rotated(x, layer, buf, EPS)
    torch.cuda.synchronize()
    # the rotated codes equal the standalone kernel's
    qs, ds = api.rmsnorm_hadamard_quantize(to_dev(c["x"], torch), layer.gamma, EPS)
    assert np.array_equal(buf.xq.cpu().numpy(), qs.cpu().numpy())
    xq, xd = buf.xq[0].cpu().numpy(), f16_to_np_bits(buf.xd)[0]
    gu, a_gu = orc.gemv_q8_0(c["gu_qs"], c["gu_d"], xq, xd)
    g, u = gu[0, :F], gu[0, F:]
    h = buf.h[0].cpu().numpy()
    assert_close(h, orc.silu_mul(g, u), silu_scale(g, u, a_gu[0, :F], a_gu[0, F:]), TOL_Q8, "h")
    hq, hd = orc.quantize_q8_0(h[None, :])
    assert np.array_equal(buf.hq.cpu().numpy(), hq)
    y, a_y = orc.gemv_q8_0(c["dn_qs"], c["dn_d"], hq, hd)
    exact = c["x"].astype(np.float64) + y[0]
    assert_close(x.cpu().numpy(), exact, a_y[0] + np.abs(c["x"]) + np.abs(exact), TOL_Q8, "out")


@pytest.mark.parametrize("hidden,ffn", [(1024, 3584), (256, 512), (512, 1024)])
def test_fused_rotated_layer(torch, orc, hidden, ffn):
    """qg_decode_ffn_q8_0_rotated (two launches, the rotation inside the fused
    gate|up kernel): its rotated codes equal rmsnorm_hadamard_quantize's, and the
    layer is checked against the oracle stage by stage from its own intermediates."""
    from block_quantized_decode_rmsnorm_gb300 import api

    c = synth.ffn_case(7, hidden, ffn)
    layer = api.FFNLayer(to_dev(c["gamma"], torch), weight(c["gu_qs"], c["gu_d"]), weight(c["dn_qs"], c["dn_d"]))
    buf = api.FFNBuffers.allocate(hidden, ffn, "cuda")
    x = to_dev(c["x"], torch)
    out = Guarded(torch, (hidden,), torch.float32)
    api.qg_decode_ffn_q8_0_rotated(x, out.view, layer, buf, EPS, export_codes=True)
    torch.cuda.synchronize()
    out.check()
    qs, ds = api.rmsnorm_hadamard_quantize(x, layer.gamma, EPS)
    xq, xd = buf.xq[0].cpu().numpy(), f16_to_np_bits(buf.xd)[0]
    assert np.array_equal(xq, qs.cpu().numpy()[0]) and np.array_equal(xd, f16_to_np_bits(ds)[0])
    gu, a_gu = orc.gemv_q8_0(c["gu_qs"], c["gu_d"], xq, xd)
    g, u = gu[0, :ffn], gu[0, ffn:]
    h = buf.h[0].cpu().numpy()
    assert_close(h, orc.silu_mul(g, u), silu_scale(g, u, a_gu[0, :ffn], a_gu[0, ffn:]), TOL_Q8, "h")
    hq, hd = orc.quantize_q8_0(h[None, :])
    assert np.array_equal(buf.hq.cpu().numpy(), hq) and np.array_equal(f16_to_np_bits(buf.hd), hd)
    y, a_y = orc.gemv_q8_0(c["dn_qs"], c["dn_d"], hq, hd)
    exact = c["x"].astype(np.float64) + y[0]
    assert_close(out.view.cpu().numpy(), exact, a_y[0] + np.abs(c["x"]) + np.abs(exact), TOL_Q8, "out")


def test_fused_rotated_layers_chained_in_place(torch, orc):
    """Three rotated layers in place, each compared with the four-launch rotated
    composite run on the fused path's own input to it (same rotated codes, so the
    same h up to the order of the gate|up sums: checked against the oracle)."""
    from block_quantized_decode_rmsnorm_gb300 import api

    cases = [synth.ffn_case(8, 1024, 3584, layer=l) for l in range(3)]
    x = to_dev(cases[0]["x"], torch)
    buf = api.FFNBuffers.allocate(1024, 3584, "cuda")
    for c in cases:
        layer = api.FFNLayer(to_dev(c["gamma"], torch), weight(c["gu_qs"], c["gu_d"]),
                             weight(c["dn_qs"], c["dn_d"]))
        x_in = x.cpu().numpy()
        api.qg_decode_ffn_q8_0_rotated(x, x, layer, buf, EPS, export_codes=True)
        torch.cuda.synchronize()
        z64, a, _, _ = orc.rmsnorm_hadamard(x_in, c["gamma"], EPS)
        xq, xd = buf.xq[0].cpu().numpy(), f16_to_np_bits(buf.xd)[0]
        # the codes dequantize to the exact rotated row within the Q8_0 bound: half a
        # step, plus the binary16 rounding of the scale times |code| <= 127
        dh = np.repeat(orc.f16_bits_to_f64(xd), 32)
        deq = xq.astype(np.float64) * dh
        assert np.max(np.abs(deq - z64) / dh.clip(min=1e-30)) <= 0.5 + 127 * 2.0 ** -11 + 1e-6
        y, a_y = orc.gemv_q8_0(c["dn_qs"], c["dn_d"], buf.hq.cpu().numpy(), f16_to_np_bits(buf.hd))
        exact = x_in.astype(np.float64) + y[0]
        assert_close(x.cpu().numpy(), exact, a_y[0] + np.abs(x_in) + np.abs(exact), TOL_Q8, "out")
