"""GPU parity for the persistent decode stack (qg_decode_stack_q8_0): every layer
of a stack of decode FFN blocks in one cooperative launch, the hand-offs between
phases through value+epoch words.

"Filling in the blanks: Inference using Phobos", Q4_K_M (the whole MLP as one
persistent kernel); Fast Decode (quantize once and share, stacked projections,
residual folded into the matmul).

The stack takes every sum in the order of the two-launch layer, so its output
must equal n_layers calls of qg_decode_ffn_q8_0 bit for bit; that path is held
to the oracle stage by stage in test_gpu_ffn.py.  Here the stack is also checked
against the oracle directly, stage by stage from its own exported h.
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


def _layers(torch, hidden, ffn, n, seed=0):
    from block_quantized_decode_rmsnorm_gb300 import api

    cases = [synth.ffn_case(seed, hidden, ffn, layer=l) for l in range(n)]
    layers = [api.FFNLayer(to_dev(c["gamma"], torch), weight(c["gu_qs"], c["gu_d"]), weight(c["dn_qs"], c["dn_d"]))
              for c in cases]
    return cases, layers


def _two_launch(torch, layers, x0):
    """The same layers through qg_decode_ffn_q8_0, one after another."""
    from block_quantized_decode_rmsnorm_gb300 import api

    hidden, ffn = layers[0].gamma.shape[0], layers[0].down.k
    buf = api.FFNBuffers.allocate(hidden, ffn, "cuda")
    x = x0.clone()
    for ly in layers:
        api.qg_decode_ffn_q8_0(x, ly, buf, EPS)
    torch.cuda.synchronize()
    return x.cpu().numpy(), buf.h[0].cpu().numpy(), buf.hq[0].cpu().numpy(), f16_to_np_bits(buf.hd)[0]


def _stack_run(torch, stack, x0, **kw):
    hidden, ffn = stack.hidden, stack.ffn
    out = Guarded(torch, (hidden,), torch.float32)
    h = Guarded(torch, (ffn,), torch.float32)
    hq = Guarded(torch, (ffn,), torch.int8)
    hd = Guarded(torch, (ffn // 32,), torch.float16)
    stack.run(x0, out.view, EPS, h_last=h.view, hq_last=hq.view, hd_last=hd.view, **kw)
    torch.cuda.synchronize()
    for g in (out, h, hq, hd):
        g.check()
    return out.view.cpu().numpy(), h.view.cpu().numpy(), hq.view.cpu().numpy(), f16_to_np_bits(hd.view)


@pytest.mark.parametrize("hidden,ffn,n_layers", [
    (1024, 3584, 1), (1024, 3584, 2), (1024, 3584, 5), (1024, 3584, 24),
    (256, 256, 3), (512, 1024, 4), (768, 2048, 3), (1024, 4096, 2), (1024, 768, 3),
])
def test_stack_equals_two_launch_layers(torch, hidden, ffn, n_layers):
    from block_quantized_decode_rmsnorm_gb300 import api

    cases, layers = _layers(torch, hidden, ffn, n_layers)
    x0 = to_dev(cases[0]["x"], torch)
    ref = _two_launch(torch, layers, x0)
    stack = api.DecodeStack(layers)
    got = _stack_run(torch, stack, x0)
    assert stack.status() == 0
    for name, a, b in zip(("x_out", "h", "hq", "hd"), got, ref):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), name


def test_stack_oracle_staged(torch, orc):
    """One layer of the 0.8B shape against the oracle: h within tolerance from
    the oracle's own RMSNorm + Q8_0 of x (bit-exact codes make it so), the GPU's
    h quantized bit-exactly, the output within tolerance from the GPU's codes."""
    from block_quantized_decode_rmsnorm_gb300 import api

    cases, layers = _layers(torch, 1024, 3584, 1, seed=3)
    c = cases[0]
    stack = api.DecodeStack(layers)
    x_out, h, hq, hd = _stack_run(torch, stack, to_dev(c["x"], torch))
    assert stack.status() == 0
    q, d, _, _ = orc.rmsnorm_quantize(c["x"], c["gamma"], EPS)
    gu, a_gu = orc.gemv_q8_0(c["gu_qs"], c["gu_d"], q, d)
    g, u = gu[0, :3584], gu[0, 3584:]
    assert_close(h, orc.silu_mul(g, u), silu_scale(g, u, a_gu[0, :3584], a_gu[0, 3584:]), TOL_Q8, "h")
    oq, od = orc.quantize_q8_0(h[None, :])
    assert np.array_equal(hq, oq[0])
    assert np.array_equal(hd, od[0])
    y, a_y = orc.gemv_q8_0(c["dn_qs"], c["dn_d"], hq, hd)
    exact = c["x"].astype(np.float64) + y[0]
    assert_close(x_out, exact, a_y[0] + np.abs(c["x"]) + np.abs(exact), TOL_Q8, "out")


def test_stack_relaunch_generation(torch):
    """Launch after launch on one workspace: the same bits every time, the
    status clear, and the generation counter advanced once per launch."""
    from block_quantized_decode_rmsnorm_gb300 import api

    cases, layers = _layers(torch, 1024, 3584, 3, seed=1)
    x0 = to_dev(cases[0]["x"], torch)
    stack = api.DecodeStack(layers)
    first = stack.run(x0).cpu().numpy()
    out = torch.empty_like(x0)
    for _ in range(40):
        stack.run(x0, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), first)
    assert stack.status() == 0
    assert stack.generation() == 41


def test_stack_graph_replay(torch):
    from block_quantized_decode_rmsnorm_gb300 import api

    cases, layers = _layers(torch, 1024, 3584, 4, seed=2)
    x0 = to_dev(cases[0]["x"], torch)
    stack = api.DecodeStack(layers)
    eager = stack.run(x0).cpu().numpy()
    out = torch.zeros_like(x0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            stack.run(x0, out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(5):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), eager)
    assert stack.status() == 0


def test_stack_host_buffers_and_in_place(torch):
    """Input read from, and output written to, pinned host memory by the kernel;
    and the output written over the input."""
    from block_quantized_decode_rmsnorm_gb300 import api

    cases, layers = _layers(torch, 1024, 3584, 2, seed=4)
    x0 = to_dev(cases[0]["x"], torch)
    stack = api.DecodeStack(layers)
    ref = stack.run(x0).cpu().numpy()
    xh = torch.from_numpy(cases[0]["x"].copy()).pin_memory()
    oh = torch.zeros_like(xh).pin_memory()
    stack.run(xh, oh)
    torch.cuda.synchronize()
    assert np.array_equal(oh.numpy(), ref)
    xi = x0.clone()
    stack.run(xi, xi)
    torch.cuda.synchronize()
    assert np.array_equal(xi.cpu().numpy(), ref)
    assert stack.status() == 0


def test_stack_more_layers_than_one_launch(torch):
    """More layers than one launch takes: the stack runs in consecutive
    launches and still equals the two-launch layers."""
    from block_quantized_decode_rmsnorm_gb300 import _lib, api

    cap = _lib.load().qg_decode_stack_max_layers()
    cases, two = _layers(torch, 512, 1024, 2, seed=5)
    layers = [two[i % 2] for i in range(cap + 3)]
    x0 = to_dev(cases[0]["x"], torch)
    ref = _two_launch(torch, layers, x0)
    stack = api.DecodeStack(layers)
    got = _stack_run(torch, stack, x0)
    assert stack.status() == 0
    for name, a, b in zip(("x_out", "h", "hq", "hd"), got, ref):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), name


def test_stack_wait_limit_reports_status(torch):
    """A wait limit far too short for the hand-offs: the launch returns normally,
    the status word says a wait ran out, and after a reset the same workspace
    gives the right result (the context stays usable)."""
    from block_quantized_decode_rmsnorm_gb300 import api

    cases, layers = _layers(torch, 1024, 3584, 4, seed=6)
    x0 = to_dev(cases[0]["x"], torch)
    stack = api.DecodeStack(layers)
    ref = stack.run(x0).cpu().numpy()
    stack.run(x0, torch.empty_like(x0), wait_limit_ns=1)
    torch.cuda.synchronize()
    st = stack.status()
    assert st != 0 and (st & ~3) == 0, st
    stack.reset()
    again = stack.run(x0).cpu().numpy()
    assert stack.status() == 0
    assert np.array_equal(again, ref)
