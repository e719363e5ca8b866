"""GPU parity: bf16 projection with fused RMSNorm, and the prompt-sized Q8_0
contraction."""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

from ._gpu import Guarded, need_gpu, to_dev, weight
from ._tol import TOL_BF16, TOL_Q8, assert_close, silu_scale

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _bf16(bits, torch):
    from block_quantized_decode_rmsnorm_gb300.api import bf16_from_bits

    return bf16_from_bits(bits)


@pytest.mark.parametrize("n,k,norm,epi", [
    (18432, 2560, True, "silu_mul"),   # stacked gate|up of the 4B-shaped model
    (7168, 1024, True, "silu_mul"),    # 0.8B-shaped
    (37, 2560, False, "none"),
    (100, 4104, True, "none"),         # k not a multiple of 256 or 16: ragged last group
    (64, 8192, True, "residual"),      # several register super-chunks
    (2, 8, False, "silu_mul"),
])
def test_bf16_gemv(torch, orc, n, k, norm, epi):
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.bf16_case(n + k, n_rows=n, k=k)
    gamma = case["gamma"] if norm else None
    res = synth.f32_normal(1, 30, (n,)) if epi == "residual" else None
    n_out = n // 2 if epi == "silu_mul" else n
    gy = Guarded(torch, (n_out,), torch.float32)
    api.qgemv_bf16(_bf16(case["w"], torch), _bf16(case["x"], torch),
                   None if gamma is None else _bf16(gamma, torch), EPS, epilogue=epi,
                   residual=None if res is None else to_dev(res, torch), y=gy.view)
    torch.cuda.synchronize()
    gy.check()
    y = gy.view.cpu().numpy()
    y64, a64, _, _ = orc.gemv_bf16(case["w"], case["x"], gamma, EPS)
    if epi == "silu_mul":
        F = n // 2
        g, u = y64[:F], y64[F:]
        assert_close(y, orc.silu_mul(g, u), silu_scale(g, u, a64[:F], a64[F:], TOL_BF16), TOL_BF16, "bf16 silu")
    elif epi == "residual":
        exact = res.astype(np.float64) + y64
        assert_close(y, exact, a64 + np.abs(res) + np.abs(exact), TOL_BF16, "bf16 residual")
    else:
        assert_close(y, y64, a64, TOL_BF16, "bf16")


def test_bf16_matches_q8_bound_when_exact(torch, orc):
    """With the norm off the f32 accumulation error is far inside the bf16 bar;
    check the much tighter Q8_0 bar too, so that a lost term cannot hide in 2e-3."""
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.bf16_case(77, n_rows=512, k=2560)
    y = api.qgemv_bf16(_bf16(case["w"], torch), _bf16(case["x"], torch)).cpu().numpy()
    y64, a64, _, _ = orc.gemv_bf16(case["w"], case["x"], None, EPS)
    assert_close(y, y64, a64, TOL_Q8, "bf16 tight")


@pytest.mark.parametrize("m,n,k", [(1, 8, 32), (5, 70, 96), (64, 96, 128), (130, 200, 1024), (128, 64, 3584),
                                   (33, 129, 8192)])
def test_prefill_small(torch, orc, m, n, k):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d = synth.q8_0_weight_planes(m + n, 10, n, k)
    x = synth.f32_normal(m + k, 0, (m, k))
    xq, xd = orc.quantize_q8_0(x)
    gy = Guarded(torch, (m, n), torch.float32)
    api.qgemm_q8_0_prefill(weight(qs, d), to_dev(xq, torch), to_dev(xd, torch, torch.float16), y=gy.view)
    torch.cuda.synchronize()
    gy.check()
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    assert_close(gy.view.cpu().numpy(), y64, a64, TOL_Q8, f"prefill {m}x{n}x{k}")


def test_prefill_full_size_sampled(torch, orc):
    """M=512 prompt rows x W 7168x1024: every output of 24 sampled prompt rows
    (including the first and last) against the oracle."""
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.prefill_case(0)
    xq_t, xd_t = api.quantize_act_q8_0(to_dev(case["x"], torch))
    y = api.qgemm_q8_0_prefill(weight(case["w_qs"], case["w_d"]), xq_t, xd_t).cpu().numpy()
    xq, xd = orc.quantize_q8_0(case["x"])
    assert np.array_equal(xq_t.cpu().numpy(), xq)
    rows = np.array([0, 1, 17, 63, 64, 127, 128, 200, 255, 256, 300, 383, 384, 400, 450, 500, 505, 506, 507, 508,
                     509, 510, 511, 99])
    y64, a64 = orc.gemv_q8_0(case["w_qs"], case["w_d"], xq[rows], xd[rows])
    assert_close(y[rows], y64, a64, TOL_Q8, "prefill full")


def test_prefill_row_equals_gemv(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d = synth.q8_0_weight_planes(4, 10, 256, 1024)
    x = synth.f32_normal(4, 0, (3, 1024))
    xq_t, xd_t = api.quantize_act_q8_0(to_dev(x, torch))
    w = weight(qs, d)
    yp = api.qgemm_q8_0_prefill(w, xq_t, xd_t).cpu().numpy()
    yg = api.qgemv_q8_0(w, xq_t, xd_t).cpu().numpy()
    xq, xd = orc.quantize_q8_0(x)
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    assert_close(yp, yg, a64, 2 * TOL_Q8, "prefill vs gemv")
