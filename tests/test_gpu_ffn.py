"""GPU parity for the decode FFN step: RMSNorm -> Q8_0 -> stacked gate|up with
SiLU(g)*u -> Q8_0 -> down with the residual folded in (0.8B-shaped: hidden
1024, FFN 3584).

Staged contract: every integer stage must match the oracle bit for bit when fed
the GPU's own input to that stage; every float stage must meet the normalised
tolerance against the oracle's exact value from the same inputs.  The
independent end-to-end comparison is reported with a looser bound, because a
1-ulp difference in h can flip a quantization code of the second projection.
"""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

from ._gpu import f16_to_np_bits, need_gpu, to_dev, weight
from ._tol import TOL_Q8, assert_close, norm_err, silu_scale

pytestmark = pytest.mark.gpu
EPS = 1e-6
HIDDEN, FFN = 1024, 3584


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _layer(torch, case):
    from block_quantized_decode_rmsnorm_gb300 import api

    return api.FFNLayer(to_dev(case["gamma"], torch), weight(case["gu_qs"], case["gu_d"]),
                        weight(case["dn_qs"], case["dn_d"]))


def check_layer_staged(orc, case_np, x_in, buf, x_out, gamma):
    """Check one FFN layer stage by stage from the GPU's own stage inputs."""
    # stage 1: RMSNorm + quantize (bit-exact)
    q, d, r, _ = orc.rmsnorm_quantize(x_in, gamma, EPS)
    assert np.array_equal(buf["xq"], q)
    assert np.array_equal(buf["xd"], d)
    # stage 2: stacked gate|up + SiLU(g)*u from the GPU's xq/xd
    gu, a_gu = orc.gemv_q8_0(case_np["gu_qs"], case_np["gu_d"], buf["xq"], buf["xd"])
    g, u = gu[0, :FFN], gu[0, FFN:]
    assert_close(buf["h"], orc.silu_mul(g, u), silu_scale(g, u, a_gu[0, :FFN], a_gu[0, FFN:]), TOL_Q8, "h")
    # stage 3: quantize the GPU's h (bit-exact)
    hq, hd = orc.quantize_q8_0(buf["h"][None, :])
    assert np.array_equal(buf["hq"], hq[0])
    assert np.array_equal(buf["hd"], hd[0])
    # stage 4: down + residual from the GPU's hq/hd
    y, a_y = orc.gemv_q8_0(case_np["dn_qs"], case_np["dn_d"], buf["hq"], buf["hd"])
    exact = x_in.astype(np.float64) + y[0]
    assert_close(x_out, exact, a_y[0] + np.abs(x_in) + np.abs(exact), TOL_Q8, "out")


def _snapshot(buf):
    return {"xq": buf.xq[0].cpu().numpy(), "xd": f16_to_np_bits(buf.xd)[0], "h": buf.h[0].cpu().numpy(),
            "hq": buf.hq[0].cpu().numpy(), "hd": f16_to_np_bits(buf.hd)[0]}


def test_ffn_staged_parity(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.ffn_case(0)
    layer = _layer(torch, case)
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    x = to_dev(case["x"], torch)
    api.decode_ffn_q8_0(x, layer, buf, EPS)
    torch.cuda.synchronize()
    check_layer_staged(orc, case, case["x"], _snapshot(buf), x.cpu().numpy(), case["gamma"])

    # independent end to end: the oracle from the same x
    ref = orc.decode_ffn(case["x"], case["gamma"], EPS, case["gu_qs"], case["gu_d"], case["dn_qs"], case["dn_d"])
    flips = int(np.count_nonzero(_snapshot(buf)["hq"] != ref["hq"][0]))
    e = norm_err(x.cpu().numpy(), ref["out64"], ref["a_y"] + np.abs(case["x"]) + np.abs(ref["out64"]))
    assert flips <= 8, flips
    assert e.max() <= 1e-4, e.max()


def test_ffn_graph_replay_bit_identical(torch, orc):
    """The four launches recorded once in a CUDA graph and replayed give the
    same bits as eager execution, every time."""
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.ffn_case(1)
    layer = _layer(torch, case)
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    x0 = to_dev(case["x"], torch)
    x = x0.clone()
    api.decode_ffn_q8_0(x, layer, buf, EPS)
    torch.cuda.synchronize()
    eager = x.cpu().numpy()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    xg = x0.clone()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            api.decode_ffn_q8_0(xg, layer, buf, EPS, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(5):
        xg.copy_(x0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(xg.cpu().numpy(), eager)


def test_ffn_layer_chain_parity(torch, orc):
    """Several chained layers with distinct weights (the benchmark's step), each
    layer checked stage by stage from the GPU's own input to it."""
    from block_quantized_decode_rmsnorm_gb300 import api

    n_layers = 3
    cases = [synth.ffn_case(0, layer=l) for l in range(n_layers)]
    layers = [_layer(torch, c) for c in cases]
    bufs = [api.FFNBuffers.allocate(HIDDEN, FFN, "cuda") for _ in range(n_layers)]
    x = to_dev(cases[0]["x"], torch)
    inputs = []
    for l in range(n_layers):
        inputs.append(x.cpu().numpy().copy())
        api.decode_ffn_q8_0(x, layers[l], bufs[l], EPS)
    torch.cuda.synchronize()
    outs = inputs[1:] + [x.cpu().numpy()]
    for l in range(n_layers):
        check_layer_staged(orc, cases[l], inputs[l], _snapshot(bufs[l]), outs[l], cases[l]["gamma"])
