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


def _near_midpoint_row(offset_rel):
    """x (f32[1024]) with eps = 0 whose exact r = 1/sqrt(mean(x^2)) is
    r_mid * (1 + offset_rel), r_mid = 1 + 2^-24 the midpoint between f32 1.0 and
    its successor: 1020 ones and four values chosen greedily (each the largest
    f32 whose square fits the remainder) so that the sum of squares S matches
    1024 / r^2 to about 2^-80.  Exact rational arithmetic throughout.
    Returns x, S and the target sum T."""
    from fractions import Fraction as Fr

    r_t = (1 + Fr(1, 2 ** 24)) * (1 + Fr(offset_rel))
    T = Fr(1024) / (r_t * r_t)
    rem = T - 1020

    def f32_below_sqrt(v):
        f = np.float32(float(v) ** 0.5)
        while Fr(float(f)) ** 2 > v:
            f = np.nextafter(f, np.float32(0))
        while Fr(float(np.nextafter(f, np.float32(np.inf)))) ** 2 <= v:
            f = np.nextafter(f, np.float32(np.inf))
        return f

    vals = [np.float32(1.0)] * 1020
    a = f32_below_sqrt(rem - 1)
    vals.append(a)
    rem -= Fr(float(a)) ** 2
    vals.append(np.float32(1.0))
    rem -= 1
    for _ in range(2):
        b = f32_below_sqrt(rem)
        vals.append(b)
        rem -= Fr(float(b)) ** 2
    x = np.array(vals, np.float32)
    S = sum(Fr(float(v)) ** 2 for v in x)
    return x, S, T


def test_rms_inv_near_a_midpoint(torch, orc):
    """r at an f32 rounding midpoint.  r on the GPU (compensated f32, about 2^-46
    relative before its last rounding) and in the oracle (f64) are exact except
    within that distance of a midpoint: there either may take either neighbour,
    so only that is asserted (and which one each took is reported).  2^-40 away
    from the midpoint both must give the correctly rounded value."""
    from fractions import Fraction as Fr

    from block_quantized_decode_rmsnorm_gb300 import api

    lo, hi = np.float32(1.0), np.nextafter(np.float32(1.0), np.float32(2.0))
    mid = 1 + Fr(1, 2 ** 24)
    for offset, must_be_exact in ((0.0, False), (2.0 ** -40, True), (-(2.0 ** -40), True)):
        x, S, T = _near_midpoint_row(offset)
        assert 0 <= T - S < T / 2 ** 70  # the construction hit its target
        # exact r = 1/sqrt(S/1024) lies above the midpoint iff S mid^2 < 1024
        correct = hi if S * mid * mid < 1024 else lo
        g = np.ones(1024, np.float32)
        inv = torch.empty((1,), dtype=torch.float32, device="cuda")
        api.rmsnorm_quantize(to_dev(x, torch), to_dev(g, torch), 0.0, inv_rms=inv)
        torch.cuda.synchronize()
        r_gpu = inv.cpu().numpy()[0]
        _, _, r_orc, _ = orc.rmsnorm_quantize(x, g, 0.0)
        assert r_gpu in (lo, hi) and r_orc in (lo, hi), (r_gpu, r_orc)
        if must_be_exact:
            assert r_gpu == correct and r_orc == correct, (offset, r_gpu, r_orc, correct)
        else:
            print(f"at the midpoint: gpu {r_gpu!r}, oracle {r_orc!r}, correctly rounded {correct!r}")
