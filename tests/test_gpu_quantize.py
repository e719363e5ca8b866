"""GPU parity: activation quantization and RMSNorm + quantization (bit-exact)."""

import json
import os

import numpy as np
import pytest

from block_quantized_decode_rmsnorm_gb300 import synth

from ._gpu import Guarded, f16_to_np_bits, need_gpu, to_dev

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


@pytest.mark.parametrize("rows,k", [(1, 32), (1, 1024), (3, 3584), (7, 96), (5, 160), (512, 1024), (33, 2560)])
def test_quantize_act_bit_exact(torch, orc, rows, k):
    from block_quantized_decode_rmsnorm_gb300 import api

    x = synth.f32_normal(rows * 31 + k, 0, (rows, k))
    if rows > 2:
        x[1, :32] = 0.0  # an all-zero block
        x[2, 32:64] = np.float32(1.0)  # constant block
    gq = Guarded(torch, (rows, k), torch.int8)
    gd = Guarded(torch, (rows, k // 32), torch.float16)
    api.quantize_act_q8_0(to_dev(x, torch), q=gq.view, d=gd.view)
    torch.cuda.synchronize()
    gq.check()
    gd.check()
    q, d = orc.quantize_q8_0(x)
    assert np.array_equal(gq.view.cpu().numpy(), q)
    assert np.array_equal(f16_to_np_bits(gd.view), d)


def test_quantize_act_hand_cases(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    cases = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "q8_0_quantize_hand_cases.json")))
    rows = []
    for c in cases["cases"]:
        x = np.zeros(32, np.float32)
        if c["x"] == "ones":
            x[:] = 1.0
        else:
            x[: len(c["x"])] = c["x"]
        rows.append(x)
    x = np.stack(rows)
    q, d = api.quantize_act_q8_0(to_dev(x, torch))
    qo, do = orc.quantize_q8_0(x)
    assert np.array_equal(q.cpu().numpy(), qo)
    assert np.array_equal(f16_to_np_bits(d), do)
    for i, c in enumerate(cases["cases"]):
        assert int(f16_to_np_bits(d)[i, 0]) == c["d_bits"], c["name"]


@pytest.mark.parametrize("rows,k", [(1, 32), (1, 1024), (1, 2560), (1, 3584), (3, 1024), (2, 96)])
def test_rmsnorm_quantize_bit_exact(torch, orc, rows, k):
    from block_quantized_decode_rmsnorm_gb300 import api

    x = synth.f32_normal(k + rows, 0, (rows, k))
    g = synth.f32_normal(k + rows, 1, (k,), 1.0, 0.1)
    gq = Guarded(torch, (rows, k), torch.int8)
    q, d, r = api.rmsnorm_quantize(to_dev(x, torch), to_dev(g, torch), EPS, q=gq.view)
    torch.cuda.synchronize()
    gq.check()
    for i in range(rows):
        qo, do, ro, _ = orc.rmsnorm_quantize(x[i], g, EPS)
        assert r[i].item() == ro, (i, r[i].item(), ro)
        assert np.array_equal(q[i].cpu().numpy(), qo)
        assert np.array_equal(f16_to_np_bits(d)[i], do)


def test_rmsnorm_constant_and_tiny(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    k = 1024
    x = np.stack([np.full(k, 0.75, np.float32), np.full(k, 1e-4, np.float32), np.zeros(k, np.float32)])
    g = np.ones(k, np.float32)
    q, d, r = api.rmsnorm_quantize(to_dev(x, torch), to_dev(g, torch), EPS)
    for i in range(3):
        qo, do, ro, _ = orc.rmsnorm_quantize(x[i], g, EPS)
        assert r[i].item() == ro
        assert np.array_equal(q[i].cpu().numpy(), qo)
        assert np.array_equal(f16_to_np_bits(d)[i], do)


def test_pack_matches_oracle(torch, orc):
    from block_quantized_decode_rmsnorm_gb300 import api

    blocks, qs, d = synth.q8_0_weight_blocks(3, 10, 129, 1024)
    w = api.qg_q8_0_pack(to_dev(blocks.reshape(-1), torch), 129, 1024)
    torch.cuda.synchronize()
    oq, od = orc.q8_0_pack(blocks, 129, 1024)
    assert np.array_equal(w.qs.cpu().numpy(), oq)
    assert np.array_equal(f16_to_np_bits(w.d), od)
