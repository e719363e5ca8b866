"""The block sums at their extreme: every code +-127, every scale 1.0.

"Filling in the blanks: Inference using Phobos", GPU Performance Heisenbugs: the
prompt runs exact int8 values on the integer tensor cores.  The tcgen05 kernels
here run them as f16 operands with f32 accumulation, exact only while every
partial sum of a 32-value block stays below 2^24; the largest block sum is
32 * 127^2 = 516,128.  With every scale 1.0 every output is an integer of at most
1024 * 127^2 = 16,516,096 < 2^24, so each kernel's f32 result must equal the
oracle's exact value bit for bit, whatever its summation order.
"""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

from ._gpu import Guarded, need_gpu, to_dev, weight

pytestmark = pytest.mark.gpu
ONE = 0x3C00  # binary16 1.0


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _case(m, n, k, pattern):
    if pattern == "all_plus":
        xs = np.ones((m, k), np.float32)
        ws = np.ones((n, k), np.int8)
    elif pattern == "alternating":  # w row signs alternate along k: every block sum is 0
        xs = np.ones((m, k), np.float32)
        ws = np.tile(np.array([1, -1], np.int8), (n, k // 2))
    else:  # random signs on both sides, and row 0 of x all -1 against row 0 of w all +1
        xs = np.where(synth.uniform_int(0, 301, m * k, 0, 1).reshape(m, k) > 0, 1.0, -1.0).astype(np.float32)
        ws = np.where(synth.uniform_int(0, 302, n * k, 0, 1).reshape(n, k) > 0, 1, -1).astype(np.int8)
        xs[0] = -1.0
        ws[0] = 1
    x = (127.0 * xs).astype(np.float32)  # quantizes to codes +-127 with scale 127 / 127 = 1
    qs = (127 * ws.astype(np.int32)).astype(np.int8)
    d = np.full((n, k // 32), ONE, np.uint16)
    return x, qs, d


@pytest.mark.parametrize("pattern", ["all_plus", "alternating", "random"])
def test_prompt_kernels_exact_at_extreme_codes(torch, orc, pattern):
    from block_quantized_decode_rmsnorm_gb300 import api

    m, n, k = 256, 384, 1024
    x, qs, d = _case(m, n, k, pattern)
    xq, xd = orc.quantize_q8_0(x)
    assert np.all(np.abs(xq) == 127) and np.all(xd == ONE)
    y64, _ = orc.gemv_q8_0(qs, d, xq, xd)
    assert np.max(np.abs(y64)) <= 1024 * 127 * 127
    if pattern == "all_plus":
        assert np.all(y64 == 1024 * 127 * 127)
    expect = y64.astype(np.float32)
    assert np.array_equal(expect.astype(np.float64), y64)  # exact in f32

    w = weight(qs, d)
    xdev = to_dev(x, torch)
    outs = {}
    xq_t, xd_t = api.quantize_act_q8_0(xdev)
    outs["mma_sync"] = api.qgemm_q8_0_prefill(w, xq_t, xd_t)
    xt = api.quantize_act_q8_0_tiles(xdev)
    for bn in (64, 128):
        outs[f"tile_records_bn{bn}"] = api.qgemm_q8_0_prefill_tc(w, xt, tile_n=bn)
    w2 = api.qg_q8_0_pack_f16(w)
    x2 = api.quantize_act_q8_0_f16(xdev)
    for bn in (128, 192):
        outs[f"wide_bn{bn}"] = api.qgemm_q8_0_prefill_tc2(w2, x2, tile_n=bn)
    outs["gemv_batch8"] = api.qgemv_q8_0(w, xq_t[:8].contiguous(), xd_t[:8].contiguous())
    torch.cuda.synchronize()
    for name, y in outs.items():
        got = y.cpu().numpy()
        ref = expect[:got.shape[0]]
        bad = int(np.count_nonzero(got != ref))
        assert bad == 0, f"{name}: {bad} outputs differ, e.g. {got[got != ref][:4]} vs {ref[got != ref][:4]}"


def test_block_dots_extreme(torch, orc):
    """The exported exact block sums at +-516,128."""
    from block_quantized_decode_rmsnorm_gb300 import api

    x, qs, d = _case(4, 64, 256, "random")
    xq, _ = orc.quantize_q8_0(x)
    s = api.qg_debug_block_dots_q8_0(weight(qs, d), to_dev(xq, torch)).cpu().numpy()
    ref = orc.block_dots(qs, xq)
    assert np.array_equal(s.reshape(ref.shape), ref)
    assert np.max(np.abs(ref)) == 32 * 127 * 127
