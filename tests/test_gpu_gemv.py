"""GPU parity: Q8_0 GEMV (all epilogues, batch 1-8) and the exact block sums."""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

from ._gpu import Guarded, need_gpu, to_dev, weight
from ._tol import TOL_Q8, assert_close, silu_scale

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _case(orc, seed, n, k, batch):
    qs, d = synth.q8_0_weight_planes(seed, 10, n, k)
    x = synth.f32_normal(seed, 0, (batch, k))
    xq, xd = orc.quantize_q8_0(x)
    return qs, d, xq, xd


def _run(torch, api, qs, d, xq, xd, epi, residual=None):
    w = weight(qs, d)
    n, k = qs.shape
    batch = xq.shape[0]
    n_out = n // 2 if epi == "silu_mul" else n
    gy = Guarded(torch, (batch, n_out), torch.float32)
    res = None if residual is None else to_dev(residual, torch)
    api.qgemv_q8_0(w, to_dev(xq, torch), to_dev(xd, torch, torch.float16), epilogue=epi, residual=res, y=gy.view)
    torch.cuda.synchronize()
    gy.check()
    return gy.view.cpu().numpy()


SHAPES = [
    # (n_rows, k, batch): ragged row counts, every register-path width (K up to 4096), the
    # long-K generic path (K > 4096), batch 1-8 including widths that are padded
    (1, 32, 1), (7, 64, 1), (37, 96, 2), (256, 1024, 1), (1000, 1024, 3), (130, 2080, 1), (64, 3584, 1),
    (50, 4096, 2), (33, 8192, 1), (20, 5120, 5), (300, 1024, 8), (129, 512, 4), (17, 2048, 7), (8, 32, 8),
    # tensor-core path with 8 blocks a request group (block count not a multiple of 16)
    (100, 768, 4), (45, 256, 2),
]


@pytest.mark.parametrize("batch", [1, 3])
def test_gemv_longest_guaranteed_k(torch, orc, batch):
    """K = 2^17 (4096 blocks; ragged row count): the longest reduction for which
    the accumulation bound, (ceil(nb / 32) + 6) 2^-24 A, stays inside the
    normalised tolerance."""
    from block_quantized_decode_rmsnorm_gb300 import api

    n, k = 37, 1 << 17
    qs, d, xq, xd = _case(orc, 17 + batch, n, k, batch)
    y = _run(torch, api, qs, d, xq, xd, "none")
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    assert_close(y, y64, a64, TOL_Q8, f"gemv n={n} k={k} b={batch}")


@pytest.mark.parametrize("n,k,batch", SHAPES)
def test_gemv_none(torch, orc, n, k, batch):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d, xq, xd = _case(orc, n + k + batch, n, k, batch)
    y = _run(torch, api, qs, d, xq, xd, "none")
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    assert_close(y, y64, a64, TOL_Q8, f"gemv n={n} k={k} b={batch}")


@pytest.mark.parametrize("n,k,batch", [(2, 32, 1), (14, 64, 2), (7168, 1024, 1), (512, 3584, 1), (66, 96, 8),
                                       (1000, 8192, 1), (6, 1024, 5)])
def test_gemv_silu_mul(torch, orc, n, k, batch):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d, xq, xd = _case(orc, 7 * n + k, n, k, batch)
    h = _run(torch, api, qs, d, xq, xd, "silu_mul")
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    F = n // 2
    for b in range(batch):
        g, u = y64[b, :F], y64[b, F:]
        h64 = orc.silu_mul(g, u)
        assert_close(h[b], h64, silu_scale(g, u, a64[b, :F], a64[b, F:]), TOL_Q8, f"silu b={b}")


@pytest.mark.parametrize("n,k,batch", [(1024, 3584, 1), (37, 96, 3), (256, 1024, 8)])
def test_gemv_residual(torch, orc, n, k, batch):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d, xq, xd = _case(orc, 3 * n + k, n, k, batch)
    res = synth.f32_normal(5, 30, (batch, n))
    out = _run(torch, api, qs, d, xq, xd, "residual", residual=res)
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    exact = res.astype(np.float64) + y64
    assert_close(out, exact, a64 + np.abs(res) + np.abs(exact), TOL_Q8, "residual")


def test_gemv_residual_in_place(torch, orc):
    """residual and y may be the same buffer (the residual stream updated in place)."""
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d, xq, xd = _case(orc, 99, 1024, 3584, 1)
    res = synth.f32_normal(6, 30, (1, 1024))
    buf = to_dev(res, torch)
    api.qgemv_q8_0(weight(qs, d), to_dev(xq, torch), to_dev(xd, torch, torch.float16), epilogue="residual",
                   residual=buf, y=buf)
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    exact = res.astype(np.float64) + y64
    assert_close(buf.cpu().numpy(), exact, a64 + np.abs(res) + np.abs(exact), TOL_Q8, "in place")


@pytest.mark.parametrize("batch", [2, 4])
def test_stacked_equals_separate_and_batch_invariance(torch, orc, batch):
    """Stacked gate|up == the two separate products, bit for bit (same per-row
    arithmetic).  Batch invariance: the tensor-core kernel (batch 2-8) gives each
    row the same bits at any batch it serves (here 2 and 4 against the same rows
    inside a batch of twice the size), and agrees with the batch-1 register-tile
    kernel to the tolerance."""
    from block_quantized_decode_rmsnorm_gb300 import api

    F, k = 3584, 1024
    qs, d, xq, xd = _case(orc, 5, 2 * F, k, batch)
    xq_t, xd_t = to_dev(xq, torch), to_dev(xd, torch, torch.float16)
    st = api.qgemv_q8_0(weight(qs, d), xq_t, xd_t).cpu().numpy()
    g = api.qgemv_q8_0(weight(qs[:F], d[:F]), xq_t, xd_t).cpu().numpy()
    u = api.qgemv_q8_0(weight(qs[F:], d[F:]), xq_t, xd_t).cpu().numpy()
    assert np.array_equal(st[:, :F], g) and np.array_equal(st[:, F:], u)
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    for b in range(batch):
        y1 = api.qgemv_q8_0(weight(qs, d), xq_t[b:b + 1], xd_t[b:b + 1]).cpu().numpy()
        assert_close(y1[0], st[b], a64[b], 2 * TOL_Q8, "batch 1 vs tensor-core batch")
    if batch > 1:
        xq8 = np.concatenate([xq, xq[::-1]])
        xd8 = np.concatenate([xd, xd[::-1]])
        st8 = api.qgemv_q8_0(weight(qs, d), to_dev(xq8, torch), to_dev(xd8, torch, torch.float16)).cpu().numpy()
        assert np.array_equal(st8[:batch], st) and np.array_equal(st8[batch:], st[::-1])


@pytest.mark.parametrize("n,k,batch", [(37, 96, 1), (256, 1024, 2), (5, 3584, 8)])
def test_block_dots_exact(torch, orc, n, k, batch):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d, xq, xd = _case(orc, 11 + n, n, k, batch)
    s = api.qg_debug_block_dots_q8_0(weight(qs, d), to_dev(xq, torch)).cpu().numpy()
    assert np.array_equal(s, orc.block_dots(qs, xq))


def test_extreme_values(torch, orc):
    """All codes at +-127 (largest block sums) and zero scales."""
    from block_quantized_decode_rmsnorm_gb300 import api

    n, k = 64, 1024
    qs = np.full((n, k), -127, np.int8)
    qs[::2] = 127
    d = np.full((n, k // 32), np.float16(0.01).view(np.uint16), np.uint16)
    d[3] = 0
    xq = np.full((1, k), 127, np.int8)
    xd = np.full((1, k // 32), np.float16(0.02).view(np.uint16), np.uint16)
    y = _run(torch, api, qs, d, xq, xd, "none")
    y64, a64 = orc.gemv_q8_0(qs, d, xq, xd)
    assert_close(y, y64, a64, TOL_Q8, "extremes")
    assert y[0, 3] == 0.0
    s = api.qg_debug_block_dots_q8_0(weight(qs, d), to_dev(xq, torch)).cpu().numpy()
    assert np.array_equal(s, orc.block_dots(qs, xq))


@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_output_head_full_size(torch, orc, batch):
    """Output-head-shaped GEMV, W 262144 x 1024 (~285 MB) at batch 1/2/4/8, in the
    bench's launch configuration; checked on every 97th row plus the last rows."""
    from block_quantized_decode_rmsnorm_gb300 import api

    n, k = 262144, 1024
    qs, d = synth.q8_0_weight_planes(0, synth.S_W0, n, k)
    x = synth.f32_normal(0, synth.S_X, (batch, k))
    xq_t, xd_t = api.quantize_act_q8_0(to_dev(x, torch))
    y = api.qgemv_q8_0(weight(qs, d), xq_t, xd_t).cpu().numpy()
    xq, xd = orc.quantize_q8_0(x)
    rows = np.unique(np.concatenate([np.arange(0, n, 97), np.arange(n - 40, n)]))
    y64, a64 = orc.gemv_q8_0(qs[rows], d[rows], xq, xd)
    assert_close(y[:, rows], y64, a64, TOL_Q8, f"head b={batch}")
