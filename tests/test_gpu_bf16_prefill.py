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
    (4865, 1032, False, "none"),       # two rows per task with an odd row count, ragged groups
    (6000, 2816, True, "residual"),
    (5000, 256, True, "silu_mul"),
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


def test_bf16_outputs_independent_of_matrix_size(torch):
    """Output o of the 18432 x 2560 gate|up projection depends on gate row o and
    up row o + 9216 only and is summed in one fixed order, so a 2000-row matrix of
    the first 1000 gate and up rows (another launch shape) gives the same first
    1000 outputs bit for bit."""
    from block_quantized_decode_rmsnorm_gb300 import api

    n, k, F, f = 18432, 2560, 9216, 1000
    case = synth.bf16_case(n + k, n_rows=n, k=k)
    w = _bf16(case["w"], torch)
    x = _bf16(case["x"], torch)
    g = _bf16(case["gamma"], torch)
    big = api.qgemv_bf16(w, x, g, EPS, epilogue="silu_mul")
    small_w = torch.cat([w[:f], w[F:F + f]]).contiguous()
    small = api.qgemv_bf16(small_w, x, g, EPS, epilogue="silu_mul")
    torch.cuda.synchronize()
    assert np.array_equal(big[:f].cpu().numpy().view(np.uint32), small.cpu().numpy().view(np.uint32))


def test_bf16_gemv_weights_16_byte_aligned(torch, orc):
    """Weights starting 16 bytes past a 32-byte boundary (the smallest alignment
    the boundary accepts): same tolerance."""
    from block_quantized_decode_rmsnorm_gb300 import api

    n, k = 96, 1024
    case = synth.bf16_case(5, n_rows=n, k=k)
    big = torch.empty((n * k + 8,), dtype=torch.bfloat16, device="cuda")
    w = big[8:].view(n, k)
    assert w.data_ptr() % 32 == 16
    w.copy_(_bf16(case["w"], torch))
    y = api.qgemv_bf16(w, _bf16(case["x"], torch), _bf16(case["gamma"], torch), EPS, epilogue="silu_mul")
    torch.cuda.synchronize()
    y64, a64, _, _ = orc.gemv_bf16(case["w"], case["x"], case["gamma"], EPS)
    F = n // 2
    g, u = y64[:F], y64[F:]
    assert_close(y.cpu().numpy(), orc.silu_mul(g, u), silu_scale(g, u, a64[:F], a64[F:], TOL_BF16), TOL_BF16,
                 "bf16 silu, 16-byte aligned rows")


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


# ---------------------------------------------------------------------------
# tensor-core path: activation tiles, tcgen05
# ---------------------------------------------------------------------------

def untile(buf: np.ndarray, rows: int, k: int):
    """Activation tiles -> (codes f16 [tiles*128, k], scale bits u16 [tiles*128, k/32])."""
    nb, tiles = k // 32, -(-rows // 128)
    rec = buf.reshape(tiles, nb, 8448)
    codes = np.ascontiguousarray(rec[:, :, :8192]).view(np.float16).reshape(tiles, nb, 4, 128, 8)
    codes = codes.transpose(0, 3, 1, 2, 4).reshape(tiles * 128, k)
    scales = np.ascontiguousarray(rec[:, :, 8192:]).view(np.uint16).reshape(tiles, nb, 128)
    return codes, scales.transpose(0, 2, 1).reshape(tiles * 128, nb)


@pytest.mark.parametrize("rows,k", [(37, 1024), (128, 256), (129, 512), (1, 32)])
def test_quantize_act_tiles_bit_exact(torch, orc, rows, k):
    from block_quantized_decode_rmsnorm_gb300 import api

    x = synth.f32_normal(21 + rows, 0, (rows, k))
    x[min(3, rows - 1), :32] = 0.0
    xt = api.quantize_act_q8_0_tiles(to_dev(x, torch))
    torch.cuda.synchronize()
    codes, scales = untile(xt.buf.cpu().numpy(), rows, k)
    qo, do = orc.quantize_q8_0(x)
    assert np.array_equal(codes[:rows].astype(np.float32), qo.astype(np.float32))
    assert np.array_equal(scales[:rows], do)
    assert not codes[rows:].any() and not scales[rows:].any()  # padding rows are zero


@pytest.mark.parametrize("m,n,k,tile_n", [
    (1, 64, 256, 0), (5, 70, 256, 64), (5, 70, 256, 96), (5, 70, 256, 128),
    (128, 64, 1024, 0), (130, 200, 1024, 96), (256, 128, 3584, 0), (33, 129, 4096, 128),
    (3, 40, 8192, 64),                        # K beyond one scale table
    (300, 1000, 512, 64),                     # more tiles than SMs at BN=64: several tiles per CTA
    (512, 7168, 1024, 0), (512, 7168, 1024, 64), (512, 7168, 1024, 128),
])
def test_prefill_tc(torch, orc, m, n, k, tile_n):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d = synth.q8_0_weight_planes(m + 3 * n, 10, n, k)
    x = synth.f32_normal(m + k + 1, 0, (m, k))
    xt = api.quantize_act_q8_0_tiles(to_dev(x, torch))
    gy = Guarded(torch, (m, n), torch.float32)
    api.qgemm_q8_0_prefill_tc(weight(qs, d), xt, y=gy.view, tile_n=tile_n)
    torch.cuda.synchronize()
    gy.check()
    y = gy.view.cpu().numpy()
    xq, xdo = orc.quantize_q8_0(x)
    rows = np.arange(m) if m <= 300 else np.unique(np.concatenate([np.arange(0, m, 37), [m - 1, 127, 128]]))
    y64, a64 = orc.gemv_q8_0(qs, d, xq[rows], xdo[rows])
    assert_close(y[rows], y64, a64, TOL_Q8, f"prefill tc {m}x{n}x{k} tile {tile_n}")
    assert not np.isnan(y).any()


def test_prefill_tc_matches_mma_sync_path(torch, orc):
    """Both prompt-contraction kernels on the same operands agree within the
    combined tolerance, and the tensor-core one is deterministic across calls."""
    from block_quantized_decode_rmsnorm_gb300 import api

    m, n, k = 200, 300, 2048
    qs, d = synth.q8_0_weight_planes(77, 10, n, k)
    x = synth.f32_normal(78, 0, (m, k))
    xd_ = to_dev(x, torch)
    w = weight(qs, d)
    xt = api.quantize_act_q8_0_tiles(xd_)
    y1 = api.qgemm_q8_0_prefill_tc(w, xt).cpu().numpy()
    y2 = api.qgemm_q8_0_prefill_tc(w, xt).cpu().numpy()
    assert np.array_equal(y1, y2)
    xq_t, xs_t = api.quantize_act_q8_0(xd_)
    ym = api.qgemm_q8_0_prefill(w, xq_t, xs_t).cpu().numpy()
    xq, xdo = orc.quantize_q8_0(x)
    _, a64 = orc.gemv_q8_0(qs, d, xq, xdo)
    assert_close(y1, ym, a64, 2 * TOL_Q8, "tc vs mma.sync")


# ---------------------------------------------------------------------------
# Q8_0 prompt contraction over wide tiles (binary16 codes, block-major scales)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("n,k", [(37, 64), (70, 96), (7168, 1024), (1, 32)])
def test_pack_f16_bit_exact(torch, n, k):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d = synth.q8_0_weight_planes(5 * n + k, 10, n, k)
    p = api.qg_q8_0_pack_f16(weight(qs, d))
    torch.cuda.synchronize()
    codes, sc = p.codes.cpu().numpy(), p.scales_t.cpu().numpy()
    assert sc.shape == (k // 32, (n + 3) // 4 * 4)
    assert np.array_equal(codes.astype(np.float32), qs.astype(np.float32))
    assert np.array_equal(sc[:, :n].T, d.view(np.float16).astype(np.float32))


@pytest.mark.parametrize("rows,k", [(37, 1024), (128, 256), (129, 96), (1, 32), (512, 1024)])
def test_quantize_act_f16_bit_exact(torch, orc, rows, k):
    from block_quantized_decode_rmsnorm_gb300 import api

    x = synth.f32_normal(41 + rows, 0, (rows, k))
    x[min(3, rows - 1), :32] = 0.0
    x[rows // 2, 32 * (k // 64):32 * (k // 64) + 32] *= 1e-30  # subnormal-range block
    xc = api.quantize_act_q8_0_f16(to_dev(x, torch))
    torch.cuda.synchronize()
    qo, do = orc.quantize_q8_0(x)
    assert np.array_equal(xc.codes.cpu().numpy().astype(np.float32), qo.astype(np.float32))
    assert np.array_equal(xc.scales_t.cpu().numpy()[:, :rows].T, do.view(np.float16).astype(np.float32))


@pytest.mark.parametrize("m,n,k,tile_n", [
    (1, 64, 256, 0), (5, 70, 96, 128), (5, 70, 96, 192),   # K = 96: the last step holds one block
    (4, 129, 256, 192), (130, 200, 1024, 192), (37, 129, 4096, 0),
    (3, 40, 8192, 128),                                   # many K steps
    (600, 4000, 256, 128),                                # 160 tiles: more than one per CTA
    (512, 7168, 1024, 0), (512, 7168, 1024, 128), (512, 7168, 1024, 192),
])
def test_prefill_tc2(torch, orc, m, n, k, tile_n):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d = synth.q8_0_weight_planes(m + 3 * n + 1, 10, n, k)
    x = synth.f32_normal(m + k + 2, 0, (m, k))
    w2 = api.qg_q8_0_pack_f16(weight(qs, d))
    x2 = api.quantize_act_q8_0_f16(to_dev(x, torch))
    gy = Guarded(torch, (m, n), torch.float32)
    api.qgemm_q8_0_prefill_tc2(w2, x2, y=gy.view, tile_n=tile_n)
    torch.cuda.synchronize()
    gy.check()
    y = gy.view.cpu().numpy()
    xq, xdo = orc.quantize_q8_0(x)
    rows = np.arange(m) if m <= 300 else np.unique(np.concatenate([np.arange(0, m, 37), [m - 1, 127, 128]]))
    y64, a64 = orc.gemv_q8_0(qs, d, xq[rows], xdo[rows])
    assert_close(y[rows], y64, a64, TOL_Q8, f"prefill tc2 {m}x{n}x{k} tile {tile_n}")
    assert not np.isnan(y).any()


def test_prefill_tc2_matches_tc_and_is_deterministic(torch, orc):
    """The wide-tile kernel and the tile-record kernel agree within the combined
    tolerance on the same operands; both tile widths give identical bits (the
    per-element order of operations does not depend on the tile)."""
    from block_quantized_decode_rmsnorm_gb300 import api

    m, n, k = 200, 384, 2048
    qs, d = synth.q8_0_weight_planes(91, 10, n, k)
    x = synth.f32_normal(92, 0, (m, k))
    xd_ = to_dev(x, torch)
    w = weight(qs, d)
    w2, x2 = api.qg_q8_0_pack_f16(w), api.quantize_act_q8_0_f16(xd_)
    y1 = api.qgemm_q8_0_prefill_tc2(w2, x2, tile_n=128).cpu().numpy()
    y2 = api.qgemm_q8_0_prefill_tc2(w2, x2, tile_n=192).cpu().numpy()
    y3 = api.qgemm_q8_0_prefill_tc2(w2, x2, tile_n=192).cpu().numpy()
    assert np.array_equal(y1, y2) and np.array_equal(y2, y3)
    yt = api.qgemm_q8_0_prefill_tc(w, api.quantize_act_q8_0_tiles(xd_)).cpu().numpy()
    xq, xdo = orc.quantize_q8_0(x)
    _, a64 = orc.gemv_q8_0(qs, d, xq, xdo)
    assert_close(y1, yt, a64, 2 * TOL_Q8, "tc2 vs tc")


def test_prefill_tc2_graph_replay(torch):
    """Quantize + wide-tile contraction captured in a CUDA graph: replays give the
    eager call's bits (the library allocates nothing and takes the stream)."""
    from block_quantized_decode_rmsnorm_gb300 import api

    m, n, k = 130, 400, 512
    qs, d = synth.q8_0_weight_planes(93, 10, n, k)
    w2 = api.qg_q8_0_pack_f16(weight(qs, d))
    x = to_dev(synth.f32_normal(94, 0, (m, k)), torch)
    x2 = api.F16Codes.empty(m, k, "cuda")
    y = torch.empty((m, n), dtype=torch.float32, device="cuda")
    api.quantize_act_q8_0_f16(x, out=x2)
    ref = api.qgemm_q8_0_prefill_tc2(w2, x2).cpu().numpy()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            api.quantize_act_q8_0_f16(x, out=x2, stream=s)
            api.qgemm_q8_0_prefill_tc2(w2, x2, y=y, stream=s)
    for _ in range(2):
        y.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), ref)


# ---------------------------------------------------------------------------
# bf16 projection for a whole prompt on the tensor cores
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("m,n,k,norm,epi", [
    (512, 18432, 2560, True, "silu_mul"),  # 4B-shaped gate|up for a 512-row prompt (rows sampled)
    (3, 256, 64, True, "none"),
    (130, 520, 2560, True, "silu_mul"),    # ragged M tile, ragged last output tile (half = 260)
    (200, 300, 1000, False, "none"),       # k not a multiple of 64: zeros past the row end
    (129, 512, 4104, True, "none"),
    (1, 2, 8, True, "silu_mul"),           # smallest shape
])
def test_bf16_prefill(torch, orc, m, n, k, norm, epi):
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.bf16_case(m + n + k, n_rows=n, k=k)
    xbits = synth.bf16_normal_bits(m + k, 7, (m, k))
    gamma = case["gamma"] if norm else None
    n_out = n // 2 if epi == "silu_mul" else n
    gy = Guarded(torch, (m, n_out), torch.float32)
    xhat = torch.empty((m, k), dtype=torch.bfloat16, device="cuda") if norm else None
    api.qgemm_bf16_prefill(_bf16(case["w"], torch), _bf16(xbits, torch),
                           None if gamma is None else _bf16(gamma, torch), EPS, epilogue=epi, y=gy.view, xhat=xhat)
    torch.cuda.synchronize()
    gy.check()
    y = gy.view.cpu().numpy()
    rows = range(m) if m * n * k <= 200 * 600 * 4104 else [0, 1, m // 2, m - 1]
    for i in rows:
        y64, a64, xh, _ = orc.gemv_bf16(case["w"], xbits[i], gamma, EPS)
        if norm:  # the normalised row, bit for bit
            assert np.array_equal(xhat[i].view(torch.int16).cpu().numpy().view(np.uint16), xh), f"x_hat row {i}"
        if epi == "silu_mul":
            F = n // 2
            g, u = y64[:F], y64[F:]
            assert_close(y[i], orc.silu_mul(g, u), silu_scale(g, u, a64[:F], a64[F:], TOL_BF16), TOL_BF16,
                         f"row {i} silu")
        else:
            assert_close(y[i], y64, a64, TOL_BF16, f"row {i}")


def test_bf16_prefill_rows_match_gemv(torch, orc):
    """Each prompt row equals the decode GEMV of that row (same x_hat bits, the
    same f32 products, only the summation order differs)."""
    from block_quantized_decode_rmsnorm_gb300 import api

    m, n, k = 64, 1024, 1024
    case = synth.bf16_case(91, n_rows=n, k=k)
    xbits = synth.bf16_normal_bits(92, 7, (m, k))
    w, g = _bf16(case["w"], torch), _bf16(case["gamma"], torch)
    x = _bf16(xbits, torch)
    y = api.qgemm_bf16_prefill(w, x, g, EPS, epilogue="silu_mul").cpu().numpy()
    for i in (0, 17, 63):
        yr = api.qgemv_bf16(w, x[i].contiguous(), g, EPS, epilogue="silu_mul").cpu().numpy()
        y64, a64, _, _ = orc.gemv_bf16(case["w"], xbits[i], case["gamma"], EPS)
        F = n // 2
        scale = silu_scale(y64[:F], y64[F:], a64[:F], a64[F:], TOL_BF16)
        assert_close(y[i], yr.astype(np.float64), scale, 2 * TOL_BF16, f"row {i} vs gemv")


def test_bf16_prefill_deterministic_and_graph_replay(torch):
    """The prompt projection sums in a fixed order: repeated calls and graph
    replays give the same bits."""
    from block_quantized_decode_rmsnorm_gb300 import api

    m, n, k = 256, 1024, 2560
    case = synth.bf16_case(93, n_rows=n, k=k)
    w, g = _bf16(case["w"], torch), _bf16(case["gamma"], torch)
    x = _bf16(synth.bf16_normal_bits(94, 7, (m, k)), torch)
    xh = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((m, n // 2), dtype=torch.float32, device="cuda")
    api.qgemm_bf16_prefill(w, x, g, EPS, epilogue="silu_mul", y=y, xhat=xh)
    torch.cuda.synchronize()
    want = y.cpu().numpy().copy()
    api.qgemm_bf16_prefill(w, x, g, EPS, epilogue="silu_mul", y=y, xhat=xh)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), want)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            api.qgemm_bf16_prefill(w, x, g, EPS, epilogue="silu_mul", y=y, xhat=xh, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        y.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), want)
