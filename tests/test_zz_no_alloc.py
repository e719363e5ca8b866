"""The no-allocation layer stack (qg_decode_layers_q8_0_noalloc) against the
same layers run through qg_decode_layer_q8_0 / qg_decode_layer_finish with
caller buffers: two calls in a row give the same bits as the reference run.
(Collected last on purpose: it must pass alone and after every other test.)"""

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

from ._gpu import need_gpu, to_dev, weight

pytestmark = pytest.mark.gpu
EPS = 1e-6
HIDDEN, FFN = 1024, 3584


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.fixture(scope="module")
def layers(torch):
    from block_quantized_decode_rmsnorm_gb300 import api

    cases = [synth.ffn_case(21, hidden=HIDDEN, ffn=FFN, layer=l) for l in range(3)]
    return cases, [api.prepare_one_launch(api.FFNLayer(to_dev(c["gamma"], torch), weight(c["gu_qs"], c["gu_d"]),
                                                       weight(c["dn_qs"], c["dn_d"]))) for c in cases]


def _reference(torch, api, layers, x):
    buf = api.FFNBuffers.allocate(HIDDEN, FFN, "cuda")
    st = api.LayerStack(HIDDEN, FFN, "cuda")
    st.load(x)
    return st.run(layers, buf, EPS).clone()


def test_noalloc_two_calls_match_caller_buffers(torch, layers):
    from block_quantized_decode_rmsnorm_gb300 import api

    cases, lys = layers
    x = to_dev(cases[0]["x"], torch)
    want = _reference(torch, api, lys, x).cpu().numpy()
    a = api.qg_decode_layers_q8_0_noalloc(x, lys, EPS)
    b = api.qg_decode_layers_q8_0_noalloc(x, lys, EPS)
    torch.cuda.synchronize()
    assert np.array_equal(a.cpu().numpy(), want)
    assert np.array_equal(b.cpu().numpy(), want)
    # a different input right after, in place
    x2 = to_dev(synth.f32_normal(22, 0, (HIDDEN,)), torch)
    want2 = _reference(torch, api, lys, x2).cpu().numpy()
    api.qg_decode_layers_q8_0_noalloc(x2, lys, EPS, x_out=x2)
    torch.cuda.synchronize()
    assert np.array_equal(x2.cpu().numpy(), want2)


def test_noalloc_zero_layers_copies(torch, layers):
    from block_quantized_decode_rmsnorm_gb300 import api

    x = to_dev(synth.f32_normal(23, 0, (HIDDEN,)), torch)
    out = api.qg_decode_layers_q8_0_noalloc(x, [], EPS)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), x.cpu().numpy())
