"""Seeded synthetic inputs for the Q8_0 / bf16 decode path.

This module is shared by the CUDA path, the CPU oracle and the benchmark, so it
holds no arithmetic of the method itself: it draws raw random numbers and lays
them out in the formats the library reads.  Nothing here quantizes, normalises,
rounds an activation or forms a dot product.

Generator
---------
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) used as a counter-based generator: output i of stream
``(seed, stream)`` is ``mix64(base + (i + 1) * GOLDEN)`` with
``base = seed * GOLDEN + stream * STREAM_MUL`` (all mod 2**64).  Every tensor of
a workload gets its own stream id, so tensors can be drawn independently and in
any order.

* uniform [0, 1):  ``(z >> 11) * 2**-53``
* uniform integer in [lo, hi]:  ``lo + ((z >> 32) * (hi - lo + 1)) >> 32``
  (multiply-shift; the bias is below 2**-24 for the ranges used here)
* standard normal: Box-Muller, ``sqrt(-2 ln(1 - u1)) * cos(2 pi u2)`` from two
  consecutive uniforms (one normal per pair).

Value recipes (the pages' workloads are whole models; these stand in for them)
-----------------------------------------------------------------------------
* Q8_0 weight values: integers uniform in [-127, 127].
* Q8_0 weight scales: uniform [1e-3, 1e-2] in f64, stored as IEEE binary16
  through numpy's float16 cast (a library conversion).
* activations: f32 N(0, 1); RMSNorm gain: f32 N(1, 0.1).
* bf16 tensors: an f32 normal draw whose low 16 bits are dropped (the bf16 bit
  pattern is the top half of the f32 pattern).  This is a sampling choice for
  test data, not the method's rounding.

Weights are produced in the canonical array-of-blocks Q8_0 layout (34 bytes per
32-value block: little-endian fp16 scale, then 32 int8 values) and, for
convenience, directly as the two planes (values ``qs[n][k]``, scales
``d[n][k/32]``) that the packed device layout uses; both carry the same draw.
"""

from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
STREAM_MUL = np.uint64(0xD1B54A32D192ED03)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

QK = 32  # values per Q8_0 block
BLOCK_BYTES = 34  # fp16 scale + 32 int8 values

_CHUNK = 1 << 20
_WORKERS = max(1, min(16, os.cpu_count() or 1))


def _chunked(count: int, fn) -> None:
    """Run fn(lo, hi) over [0, count) in chunks, on host threads when large
    (every output depends only on its own counter, so chunks are independent)."""
    spans = [(lo, min(count, lo + _CHUNK)) for lo in range(0, count, _CHUNK)]
    if len(spans) <= 1 or _WORKERS == 1:
        for lo, hi in spans:
            fn(lo, hi)
        return
    with ThreadPoolExecutor(_WORKERS) as ex:
        list(ex.map(lambda sp: fn(*sp), spans))


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        return np.uint64(seed % (1 << 64)) * GOLDEN + np.uint64(stream % (1 << 64)) * STREAM_MUL


def _raw(base: np.uint64, lo: int, hi: int) -> np.ndarray:
    with np.errstate(over="ignore"):
        ctr = np.arange(lo + 1, hi + 1, dtype=np.uint64)
        return _mix64(base + ctr * GOLDEN)


def raw_u64(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """Outputs ``offset .. offset+count-1`` of SplitMix64 stream (seed, stream)."""
    base = _base(seed, stream)
    out = np.empty(count, dtype=np.uint64)

    def fill(lo, hi):
        out[lo:hi] = _raw(base, offset + lo, offset + hi)

    _chunked(count, fill)
    return out


def uniform01(seed: int, stream: int, count: int) -> np.ndarray:
    """f64 uniforms in [0, 1) with 53 random bits each."""
    base = _base(seed, stream)
    out = np.empty(count, dtype=np.float64)

    def fill(lo, hi):
        out[lo:hi] = (_raw(base, lo, hi) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    _chunked(count, fill)
    return out


def uniform_int(seed: int, stream: int, count: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform in [lo, hi] (inclusive) as int64."""
    base = _base(seed, stream)
    span = np.uint64(hi - lo + 1)
    out = np.empty(count, dtype=np.int64)

    def fill(a, b):
        z = _raw(base, a, b)
        with np.errstate(over="ignore"):
            v = ((z >> np.uint64(32)) * span) >> np.uint64(32)
        out[a:b] = v.astype(np.int64) + lo

    _chunked(count, fill)
    return out


def normal(seed: int, stream: int, count: int, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """f64 normals by Box-Muller over consecutive uniform pairs (outputs 2i, 2i+1)."""
    base = _base(seed, stream)
    out = np.empty(count, dtype=np.float64)

    def fill(a, b):
        z = _raw(base, 2 * a, 2 * b)
        u = ((z >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)).reshape(b - a, 2)
        rad = np.sqrt(-2.0 * np.log1p(-u[:, 0]))
        out[a:b] = mean + std * rad * np.cos(2.0 * np.pi * u[:, 1])

    _chunked(count, fill)
    return out


# --------------------------------------------------------------------------
# Tensors in the library's formats
# --------------------------------------------------------------------------

def f32_normal(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return normal(seed, stream, n, mean, std).astype(np.float32).reshape(shape)


def bf16_normal_bits(seed: int, stream: int, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    """uint16 bf16 bit patterns: the top half of an f32 normal draw."""
    f = f32_normal(seed, stream, shape, mean, std)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def q8_0_weight_planes(seed: int, stream: int, n_rows: int, k: int,
                       d_lo: float = 1e-3, d_hi: float = 1e-2):
    """Random Q8_0 weight as planes: qs int8[n_rows][k], d fp16 bits uint16[n_rows][k/32].

    Values come from stream ``stream``, scales from stream ``stream + 1``.
    """
    if k % QK:
        raise ValueError("k must be a multiple of 32")
    nb = k // QK
    qs = uniform_int(seed, stream, n_rows * k, -127, 127).astype(np.int8).reshape(n_rows, k)
    u = uniform01(seed, stream + 1, n_rows * nb)
    d = (d_lo + (d_hi - d_lo) * u).astype(np.float16).view(np.uint16).reshape(n_rows, nb)
    return qs, d


def q8_0_planes_to_blocks(qs: np.ndarray, d: np.ndarray) -> np.ndarray:
    """Lay planes out as canonical 34-byte blocks: uint8[n_rows][k/32][34].

    A pure byte layout step (little-endian scale, then the 32 values).
    """
    n_rows, k = qs.shape
    nb = k // QK
    out = np.empty((n_rows, nb, BLOCK_BYTES), dtype=np.uint8)
    d_le = d.astype("<u2").view(np.uint8).reshape(n_rows, nb, 2)
    out[:, :, 0:2] = d_le
    out[:, :, 2:] = qs.view(np.uint8).reshape(n_rows, nb, QK)
    return out


def q8_0_weight_blocks(seed: int, stream: int, n_rows: int, k: int):
    """Random Q8_0 weight in the canonical block layout, plus its planes."""
    qs, d = q8_0_weight_planes(seed, stream, n_rows, k)
    return q8_0_planes_to_blocks(qs, d), qs, d


# --------------------------------------------------------------------------
# Workloads (sizes of the pages' 0.8B / 4B shaped models)
# --------------------------------------------------------------------------

# Stream ids, one per tensor of a workload.
S_X, S_GAMMA, S_W0, S_W1, S_RES = 0, 1, 10, 20, 30


def gemv_case(seed: int, n_rows: int, k: int, batch: int = 1):
    """Q8_0 GEMV inputs: weight planes and f32 activations x[batch][k] ~ N(0,1)."""
    qs, d = q8_0_weight_planes(seed, S_W0, n_rows, k)
    x = f32_normal(seed, S_X, (batch, k))
    return {"w_qs": qs, "w_d": d, "x": x}


def ffn_case(seed: int, hidden: int = 1024, ffn: int = 3584, layer: int = 0):
    """Decode FFN inputs: x, gamma, stacked gate|up weight [2*ffn][hidden], down [hidden][ffn]."""
    off = 100 * layer
    x = f32_normal(seed, S_X, (hidden,))
    gamma = f32_normal(seed, S_GAMMA + off, (hidden,), 1.0, 0.1)
    gu_qs, gu_d = q8_0_weight_planes(seed, S_W0 + off, 2 * ffn, hidden)
    dn_qs, dn_d = q8_0_weight_planes(seed, S_W1 + off, hidden, ffn)
    return {"x": x, "gamma": gamma, "gu_qs": gu_qs, "gu_d": gu_d, "dn_qs": dn_qs, "dn_d": dn_d}


def bf16_case(seed: int, n_rows: int = 18432, k: int = 2560):
    """bf16 projection inputs: W ~ N(0, 0.02), x ~ N(0, 1), gamma ~ N(1, 0.1), all bf16 bits."""
    w = bf16_normal_bits(seed, S_W0, (n_rows, k), 0.0, 0.02)
    x = bf16_normal_bits(seed, S_X, (k,))
    gamma = bf16_normal_bits(seed, S_GAMMA, (k,), 1.0, 0.1)
    return {"w": w, "x": x, "gamma": gamma}


def prefill_case(seed: int, m: int = 512, n_rows: int = 7168, k: int = 1024):
    """Prefill inputs: X f32[m][k] ~ N(0,1), Q8_0 weight planes [n_rows][k]."""
    qs, d = q8_0_weight_planes(seed, S_W0, n_rows, k)
    x = f32_normal(seed, S_X, (m, k))
    return {"w_qs": qs, "w_d": d, "x": x}
