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
    flips = int(np.count_nonzero(_snapshot(buf)["hq"] != ref["hq"].ravel()))
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


# ---------------------------------------------------------------------------
# fused two-launch path: qg_ffn_up_q8_0 + qgemv_q8_0(down, residual)
# ---------------------------------------------------------------------------

def test_fused_up_bit_identical_to_composition_and_oracle(torch, orc):
    """One launch of qg_ffn_up_q8_0 gives the same bits as rmsnorm_quantize ->
    qgemv_q8_0(silu_mul) -> quantize_act_q8_0, and passes the staged oracle checks."""
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.ffn_case(2)
    layer = _layer(torch, case)
    x = to_dev(case["x"], torch)
    xq = torch.empty((HIDDEN,), dtype=torch.int8, device="cuda")
    xd = torch.empty((HIDDEN // 32,), dtype=torch.float16, device="cuda")
    r = torch.empty((1,), dtype=torch.float32, device="cuda")
    h, hq, hd = api.qg_ffn_up_q8_0(x, layer.gamma, layer.gate_up, EPS, xq_out=xq, xd_out=xd, inv_rms_out=r)
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    x2 = x.clone()
    api.decode_ffn_q8_0(x2, layer, buf, EPS)
    torch.cuda.synchronize()
    assert np.array_equal(xq.cpu().numpy(), buf.xq[0].cpu().numpy())
    assert np.array_equal(f16_to_np_bits(xd), f16_to_np_bits(buf.xd)[0])
    assert np.array_equal(h.cpu().numpy(), buf.h[0].cpu().numpy())
    assert np.array_equal(hq.cpu().numpy(), buf.hq[0].cpu().numpy())
    assert np.array_equal(f16_to_np_bits(hd), f16_to_np_bits(buf.hd)[0])
    _, _, r_o, _ = orc.rmsnorm_quantize(case["x"], case["gamma"], EPS)
    assert r.item() == r_o


def test_fused_decode_ffn_matches_unfused_and_oracle(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    n_layers = 3
    cases = [synth.ffn_case(5, layer=l) for l in range(n_layers)]
    layers = [_layer(torch, c) for c in cases]
    buf_f = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    buf_u = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    xf = to_dev(cases[0]["x"], torch)
    xu = xf.clone()
    for l in range(n_layers):
        x_in = xf.cpu().numpy().copy()
        api.qg_decode_ffn_q8_0(xf, layers[l], buf_f, EPS)
        api.decode_ffn_q8_0(xu, layers[l], buf_u, EPS)
        torch.cuda.synchronize()
        assert np.array_equal(xf.cpu().numpy(), xu.cpu().numpy()), f"layer {l}"
        snap = _snapshot(buf_u)
        check_layer_staged(orc, cases[l], x_in, snap, xf.cpu().numpy(), cases[l]["gamma"])


def test_fused_graph_replay(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.ffn_case(6)
    layer = _layer(torch, case)
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    x0 = to_dev(case["x"], torch)
    x = x0.clone()
    api.qg_decode_ffn_q8_0(x, layer, buf, EPS)
    torch.cuda.synchronize()
    eager = x.cpu().numpy()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    xg = x0.clone()
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(4):  # four layers sharing weights: exercises back-to-back PDL edges
                api.qg_decode_ffn_q8_0(xg, layer, buf, EPS, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    ref = x0.clone()
    for _ in range(4):
        api.qg_decode_ffn_q8_0(ref, layer, buf, EPS)
    torch.cuda.synchronize()
    want = ref.cpu().numpy()
    for _ in range(3):
        xg.copy_(x0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(xg.cpu().numpy(), want)
    assert not np.array_equal(want, eager)


def test_no_copy_stalls_in_normal_operation(torch, orc):
    """The stall counter of the decode kernels reads 0 after eager and replayed
    layers (every staged copy lands), and clearing it leaves 0."""
    from block_quantized_decode_rmsnorm_gb300 import api

    api.copy_stalls(clear=True)
    case = synth.ffn_case(7)
    layer = _layer(torch, case)
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    x = to_dev(case["x"], torch)
    for _ in range(8):
        api.qg_decode_ffn_q8_0(x, layer, buf, EPS)
    torch.cuda.synchronize()
    assert np.all(np.isfinite(x.cpu().numpy()))
    assert api.copy_stalls() == 0
    assert api.copy_stalls(clear=True) == 0


def test_decode_ffn_out_of_place_host_buffers(torch, orc):
    """The out-of-place layer with its input read from, and its result written to,
    pinned host memory gives the in-place device result bit for bit, eagerly and
    replayed from a graph (the end-to-end step of the benchmark)."""
    from block_quantized_decode_rmsnorm_gb300 import api

    n_layers = 3
    cases = [synth.ffn_case(7, layer=l) for l in range(n_layers)]
    layers = [_layer(torch, c) for c in cases]
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    x0 = cases[0]["x"]
    ref = to_dev(x0, torch)
    api.qg_decode_ffn_q8_0(ref, layers[0], buf, EPS)
    torch.cuda.synchronize()
    one = ref.cpu().numpy()
    for l in layers[1:]:
        api.qg_decode_ffn_q8_0(ref, l, buf, EPS)
    torch.cuda.synchronize()
    want = ref.cpu().numpy()

    x_host = torch.from_numpy(x0.copy()).pin_memory()
    out_host = torch.zeros_like(x_host).pin_memory()
    api.qg_decode_ffn_q8_0_out(x_host, out_host, layers[0], buf, EPS)  # host to host, one layer
    torch.cuda.synchronize()
    assert np.array_equal(out_host.numpy(), one)
    assert np.array_equal(x_host.numpy(), x0)  # the input is left as it was

    x = torch.empty(x0.shape, dtype=torch.float32, device="cuda")

    def step(stream=None):
        api.qg_decode_ffn_q8_0_out(x_host, x, layers[0], buf, EPS, stream=stream)
        for l in layers[1:-1]:
            api.qg_decode_ffn_q8_0(x, l, buf, EPS, stream=stream)
        api.qg_decode_ffn_q8_0_out(x, out_host, layers[-1], buf, EPS, stream=stream)

    out_host.zero_()
    step()
    torch.cuda.synchronize()
    assert np.array_equal(out_host.numpy(), want)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            step(stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out_host.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out_host.numpy(), want)
    with pytest.raises(ValueError):
        api.qg_decode_ffn_q8_0_out(torch.from_numpy(x0.copy()), x, layers[0], buf, EPS)  # pageable host memory


@pytest.mark.parametrize("hidden,ffn", [(256, 96), (2048, 1024), (768, 64)])
def test_fused_other_shapes(torch, orc, hidden, ffn):
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.ffn_case(7, hidden=hidden, ffn=ffn)
    layer = _layer(torch, case)
    buf = api.FFNBuffers.allocate(hidden, ffn, "cuda")
    x = to_dev(case["x"], torch)
    h, hq, hd = api.qg_ffn_up_q8_0(x, layer.gamma, layer.gate_up, EPS)
    torch.cuda.synchronize()
    q, d, r, _ = orc.rmsnorm_quantize(case["x"], case["gamma"], EPS)
    gu, a_gu = orc.gemv_q8_0(case["gu_qs"], case["gu_d"], q, d)
    g, u = gu[0, :ffn], gu[0, ffn:]
    assert_close(h.cpu().numpy(), orc.silu_mul(g, u), silu_scale(g, u, a_gu[0, :ffn], a_gu[0, ffn:]), TOL_Q8, "h")
    oq, od = orc.quantize_q8_0(h.cpu().numpy()[None, :])
    assert np.array_equal(hq.cpu().numpy(), oq[0]) and np.array_equal(f16_to_np_bits(hd), od[0])
    x_in = case["x"].copy()
    api.qg_decode_ffn_q8_0(x, layer, buf, EPS)
    torch.cuda.synchronize()
    y, a_y = orc.gemv_q8_0(case["dn_qs"], case["dn_d"], buf.hq.cpu().numpy(), f16_to_np_bits(buf.hd))
    exact = x_in.astype(np.float64) + y[0]
    assert_close(x.cpu().numpy(), exact, a_y[0] + np.abs(x_in) + np.abs(exact), TOL_Q8, "out")
