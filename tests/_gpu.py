"""Helpers shared by the GPU parity tests (upload, download, guard bands)."""

import numpy as np
import pytest


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_decode_rmsnorm_gb300 import _lib, build

    build()
    _lib.load()
    return torch


def to_dev(a, torch, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def f16_to_np_bits(t):
    return t.detach().cpu().view(__import__("torch").int16).numpy().view(np.uint16)


def weight(qs, d):
    from block_quantized_decode_rmsnorm_gb300.api import q8_weight_from_numpy

    return q8_weight_from_numpy(qs, d)


class Guarded:
    """A device buffer with canary-filled guard bands before and after the
    view that a kernel writes; check() fails if a kernel wrote outside it."""

    PAD = 4096  # bytes each side, keeps 256-byte alignment of the view

    def __init__(self, torch, shape, dtype):
        self.torch = torch
        n = int(np.prod(shape))
        itemsize = torch.empty((), dtype=dtype).element_size()
        pad = self.PAD // itemsize
        self.raw = torch.empty(n + 2 * pad, dtype=dtype, device="cuda")
        self.raw.view(torch.uint8).fill_(0x7F)  # canary
        self.pad = pad
        self.n = n
        self.view = self.raw[pad: pad + n].view(shape)

    def check(self):
        b = self.raw.view(self.torch.uint8)
        p = self.pad * self.raw.element_size()
        head = b[:p]
        tail = b[p + self.n * self.raw.element_size():]
        assert bool((head == 0x7F).all()), "write before the output buffer"
        assert bool((tail == 0x7F).all()), "write past the output buffer"
