"""GPU parity for the one-launch decode layer (qg_decode_layer_q8_0).

The gate|up half is the same code as qg_ffn_up_q8_0 and must give the same
bits.  The down projection is split along its reduction; the layer leaves its
output unreduced as (r, partials), summed in a fixed order by the next layer or
by qg_decode_layer_finish, so results repeat bit for bit and the next layer's
input must equal the finished output of the previous one exactly.  Outputs are
checked against the oracle from the GPU's own h codes (staged contract)."""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

from ._gpu import f16_to_np_bits, need_gpu, to_dev, weight
from ._tol import TOL_Q8, assert_close

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _layer(torch, case):
    from block_quantized_decode_rmsnorm_gb300 import api

    return api.prepare_one_launch(api.FFNLayer(to_dev(case["gamma"], torch), weight(case["gu_qs"], case["gu_d"]),
                                               weight(case["dn_qs"], case["dn_d"])))


def _check_out(orc, case, x_in, hq, hd, out, what):
    y, a_y = orc.gemv_q8_0(case["dn_qs"], case["dn_d"], hq, hd)
    exact = x_in.astype(np.float64) + y[0]
    assert_close(out, exact, a_y[0] + np.abs(x_in) + np.abs(exact), TOL_Q8, what)


def _bufs(torch, api, hidden, ffn):
    n = api.qg_decode_layer_partials(hidden, ffn)
    z = lambda *s: torch.zeros(s, dtype=torch.float32, device="cuda")
    return z(hidden), z(n, hidden)


def test_column_blocks_bit_exact(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    qs, d = synth.q8_0_weight_planes(3, 10, 70, 256)
    cb = api.qg_q8_0_column_blocks(weight(qs, d))
    torch.cuda.synchronize()
    assert np.array_equal(cb.qs.cpu().numpy(), qs.reshape(70, 8, 32).transpose(1, 0, 2))
    assert np.array_equal(f16_to_np_bits(cb.d), d.T)


# grids of 112, 3, 16, 16 and 6 CTAs: clusters of 8, 1, 8, 8 and 2 (14, 3, 2, 2, 3 partials)
@pytest.mark.parametrize("hidden,ffn", [(1024, 3584), (256, 96), (1792, 512), (2048, 1024), (1280, 512), (768, 192)])
def test_one_launch_layer(torch, orc, hidden, ffn):
    from block_quantized_decode_rmsnorm_gb300 import api

    case = synth.ffn_case(11, hidden=hidden, ffn=ffn)
    layer = _layer(torch, case)
    buf = api.FFNBuffers.allocate(hidden, ffn, "cuda")
    x_in = to_dev(case["x"], torch)
    r_out, p_out = _bufs(torch, api, hidden, ffn)
    api.qg_decode_layer_q8_0(x_in, None, r_out, p_out, layer, buf, EPS)
    out = api.qg_decode_layer_finish(r_out, p_out)
    h_ref, hq_ref, hd_ref = api.qg_ffn_up_q8_0(x_in, layer.gamma, layer.gate_up, EPS)
    torch.cuda.synchronize()
    assert np.array_equal(r_out.cpu().numpy(), case["x"])  # n_in = 0: the input itself
    # the gate|up half: same bits as the standalone kernel
    assert np.array_equal(buf.h[0].cpu().numpy(), h_ref.cpu().numpy())
    assert np.array_equal(buf.hq[0].cpu().numpy(), hq_ref.cpu().numpy())
    assert np.array_equal(f16_to_np_bits(buf.hd)[0], f16_to_np_bits(hd_ref))
    # h codes bit-exact from the GPU's h (staged contract)
    oq, od = orc.quantize_q8_0(buf.h.cpu().numpy())
    assert np.array_equal(buf.hq[0].cpu().numpy(), oq[0]) and np.array_equal(f16_to_np_bits(buf.hd)[0], od[0])
    _check_out(orc, case, case["x"], buf.hq.cpu().numpy(), f16_to_np_bits(buf.hd), out.cpu().numpy(), "out")
    assert np.array_equal(x_in.cpu().numpy(), case["x"])  # input untouched


def test_unreduced_input_is_summed_in_order(torch, orc):
    """x = r + p[0] + p[1] + p[2] in f32, in that order; the layer then runs on x."""
    from block_quantized_decode_rmsnorm_gb300 import api

    hidden, ffn = 1024, 3584
    case = synth.ffn_case(14, hidden=hidden, ffn=ffn)
    layer = _layer(torch, case)
    buf = api.FFNBuffers.allocate(hidden, ffn, "cuda")
    r = synth.f32_normal(15, 0, (hidden,))
    p = synth.f32_normal(15, 1, (3, hidden)) * np.float32(0.25)
    want = r.copy()
    for c in range(3):
        want = (want + p[c]).astype(np.float32)
    r_out, p_out = _bufs(torch, api, hidden, ffn)
    api.qg_decode_layer_q8_0(to_dev(r, torch), to_dev(p, torch), r_out, p_out, layer, buf, EPS)
    out = api.qg_decode_layer_finish(r_out, p_out)
    torch.cuda.synchronize()
    assert np.array_equal(r_out.cpu().numpy(), want)
    _check_out(orc, case, want, buf.hq.cpu().numpy(), f16_to_np_bits(buf.hd), out.cpu().numpy(), "out")


def test_layer_stack_staged_and_consistent(torch, orc):
    """Four layers: each checked from its own GPU input; each layer's input must
    be, bit for bit, the finished output of the layer before."""
    from block_quantized_decode_rmsnorm_gb300 import api

    hidden, ffn, n = 1024, 3584, 4
    cases = [synth.ffn_case(12, hidden=hidden, ffn=ffn, layer=l) for l in range(n)]
    layers = [_layer(torch, c) for c in cases]
    buf = api.FFNBuffers.allocate(hidden, ffn, "cuda")
    st = api.LayerStack(hidden, ffn, "cuda")
    st.load(to_dev(cases[0]["x"], torch))
    prev_out = None
    for l in range(n):
        api.qg_decode_layer_q8_0(st.r[l % 2], st.p[l % 2] if l else None, st.r[(l + 1) % 2], st.p[(l + 1) % 2],
                                 layers[l], buf, EPS)
        out = api.qg_decode_layer_finish(st.r[(l + 1) % 2], st.p[(l + 1) % 2])
        torch.cuda.synchronize()
        x_l = st.r[(l + 1) % 2].cpu().numpy()
        if prev_out is not None:
            assert np.array_equal(x_l, prev_out), f"layer {l} input != finished output of layer {l - 1}"
        _check_out(orc, cases[l], x_l, buf.hq.cpu().numpy(), f16_to_np_bits(buf.hd), out.cpu().numpy(), f"layer {l}")
        prev_out = out.cpu().numpy()
    # run() reproduces the same bits
    st2 = api.LayerStack(hidden, ffn, "cuda")
    st2.load(to_dev(cases[0]["x"], torch))
    got = st2.run(layers, buf, EPS)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), prev_out)


def test_layer_stack_graph_replay_bit_identical(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    hidden, ffn, n = 1024, 3584, 5
    cases = [synth.ffn_case(13, hidden=hidden, ffn=ffn, layer=l % 2) for l in range(n)]
    layers = [_layer(torch, c) for c in cases]
    buf = api.FFNBuffers.allocate(hidden, ffn, "cuda")
    st = api.LayerStack(hidden, ffn, "cuda")
    x0 = to_dev(cases[0]["x"], torch)
    st.load(x0)
    eager = st.run(layers, buf, EPS).cpu().numpy()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            st.run(layers, buf, EPS, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        st.load(x0)
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(st.out.cpu().numpy(), eager)
