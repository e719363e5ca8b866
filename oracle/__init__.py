"""CPU oracle for the Q8_0 / bf16 decode path (TEST INFRASTRUCTURE ONLY).

The arithmetic lives in ``qg_oracle.c`` (plain C, f64 where the definition is
real-valued, built with ``-ffp-contract=off``).  This module compiles it with the
host C compiler and marshals numpy arrays into it; it holds no arithmetic of its
own beyond the f32 rounding of results that the C side returns in f64.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library and its Python binding never do.

Parity pins (tests/test_oracle_*.py) tie every function to something other than
itself: the binary16 / bfloat16 converters to numpy's and torch's casts, the
GEMV to a brute-force dequantize-then-matmul in f64, the quantizer to
hand-derived rounding cases, closed forms and error bounds, RMSNorm to a
high-precision evaluation, and the epilogues to closed forms.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qg_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (host C compiler, no CUDA)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    cc = os.environ.get("CC", "cc")
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run([cc, *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            F = ctypes.c_float
            sig = {
                "orc_f32_to_f16": (ctypes.c_uint16, [F]),
                "orc_f16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
                "orc_f32_to_bf16": (ctypes.c_uint16, [F]),
                "orc_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
                "orc_f32_to_f16_array": (None, [P, I64, P]),
                "orc_f32_to_bf16_array": (None, [P, I64, P]),
                "orc_f16_to_f64_array": (None, [P, I64, P]),
                "orc_q8_0_pack": (None, [P, I64, I64, P, P]),
                "orc_quantize_q8_0": (None, [P, I64, I64, P, P]),
                "orc_rms_inv": (F, [P, I64, F]),
                "orc_rmsnorm_quantize": (None, [P, P, I64, F, P, P, P, P]),
                "orc_block_dots": (None, [P, I64, I64, P, I64, P]),
                "orc_gemv_q8_0": (None, [P, P, I64, I64, P, P, I64, P, P]),
                "orc_silu_mul": (None, [P, P, I64, P]),
                "orc_gemv_bf16": (None, [P, I64, I64, P, P, F, P, P, P, P]),
                "orc_residual_add": (None, [P, P, I64, P]),
                "orc_hadamard128": (None, [P, I64, P]),
                "orc_decode_ffn": (None, [P, P, I64, I64, F, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# scalar / vector conversions
# --------------------------------------------------------------------------

def f32_to_f16_bits(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32).ravel()
    out = np.empty(x.size, np.uint16)
    lib.orc_f32_to_f16_array(_ptr(x), x.size, _ptr(out))
    return out


def f16_bits_to_f64(h) -> np.ndarray:
    lib = _load()
    h = _c(h, np.uint16).ravel()
    out = np.empty(h.size, np.float64)
    lib.orc_f16_to_f64_array(_ptr(h), h.size, _ptr(out))
    return out


def f32_to_bf16_bits(x) -> np.ndarray:
    lib = _load()
    x = _c(x, np.float32).ravel()
    out = np.empty(x.size, np.uint16)
    lib.orc_f32_to_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


def bf16_bits_to_f64(b) -> np.ndarray:
    lib = _load()
    b = np.asarray(b, dtype=np.uint16).ravel()
    return np.fromiter((lib.orc_bf16_to_f64(int(v)) for v in b), dtype=np.float64, count=b.size)


# --------------------------------------------------------------------------
# the path
# --------------------------------------------------------------------------

def q8_0_pack(blocks: np.ndarray, n_rows: int, k: int):
    """Canonical 34-byte blocks -> (qs int8[n][k], d uint16[n][k/32])."""
    lib = _load()
    b = _c(blocks, np.uint8)
    if b.size != n_rows * (k // 32) * 34:
        raise ValueError("block buffer size does not match n_rows, k")
    qs = np.empty((n_rows, k), np.int8)
    d = np.empty((n_rows, k // 32), np.uint16)
    lib.orc_q8_0_pack(_ptr(b), n_rows, k, _ptr(qs), _ptr(d))
    return qs, d


def quantize_q8_0(x: np.ndarray):
    """x f32[rows][k] -> (q int8[rows][k], d uint16 fp16 bits [rows][k/32])."""
    lib = _load()
    x = _c(x, np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    rows, k = x2.shape
    if k % 32:
        raise ValueError("k must be a multiple of 32")
    q = np.empty((rows, k), np.int8)
    d = np.empty((rows, k // 32), np.uint16)
    lib.orc_quantize_q8_0(_ptr(x2), rows, k, _ptr(q), _ptr(d))
    return q.reshape(x.shape), d.reshape(x.shape[:-1] + (k // 32,))


def rms_inv(x: np.ndarray, eps: float) -> np.float32:
    lib = _load()
    x = _c(x, np.float32).ravel()
    return np.float32(lib.orc_rms_inv(_ptr(x), x.size, eps))


def rmsnorm_quantize(x: np.ndarray, gamma: np.ndarray, eps: float):
    """-> (q int8[k], d uint16[k/32], r f32, x_hat f32[k])."""
    lib = _load()
    x = _c(x, np.float32).ravel()
    g = _c(gamma, np.float32).ravel()
    k = x.size
    if k % 32 or g.size != k:
        raise ValueError("bad shapes")
    q = np.empty(k, np.int8)
    d = np.empty(k // 32, np.uint16)
    r = np.zeros(1, np.float32)
    xh = np.empty(k, np.float32)
    lib.orc_rmsnorm_quantize(_ptr(x), _ptr(g), k, eps, _ptr(q), _ptr(d), _ptr(r), _ptr(xh))
    return q, d, r[0], xh


def block_dots(w_qs: np.ndarray, xq: np.ndarray) -> np.ndarray:
    """int32 S[batch][n][k/32]."""
    lib = _load()
    w = _c(w_qs, np.int8)
    n, k = w.shape
    xq2 = _c(xq, np.int8).reshape(-1, k)
    batch = xq2.shape[0]
    s = np.empty((batch, n, k // 32), np.int32)
    lib.orc_block_dots(_ptr(w), n, k, _ptr(xq2), batch, _ptr(s))
    return s


def gemv_q8_0(w_qs, w_d, xq, xd):
    """Block-scaled product; returns (y f64[batch][n], a f64[batch][n])."""
    lib = _load()
    w = _c(w_qs, np.int8)
    wd = _c(w_d, np.uint16)
    n, k = w.shape
    xq2 = _c(xq, np.int8).reshape(-1, k)
    xd2 = _c(xd, np.uint16).reshape(-1, k // 32)
    batch = xq2.shape[0]
    y = np.empty((batch, n), np.float64)
    a = np.empty((batch, n), np.float64)
    lib.orc_gemv_q8_0(_ptr(w), _ptr(wd), n, k, _ptr(xq2), _ptr(xd2), batch, _ptr(y), _ptr(a))
    return y, a


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    lib = _load()
    g = _c(g, np.float64).ravel()
    u = _c(u, np.float64).ravel()
    h = np.empty_like(g)
    lib.orc_silu_mul(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def gemv_bf16(w_bits, x_bits, gamma_bits, eps: float):
    """-> (y f64[n], a f64[n], x_hat bf16 bits [k], r f32)."""
    lib = _load()
    w = _c(w_bits, np.uint16)
    n, k = w.shape
    x = _c(x_bits, np.uint16).ravel()
    xh = np.empty(k, np.uint16)
    r = np.zeros(1, np.float32)
    y = np.empty(n, np.float64)
    a = np.empty(n, np.float64)
    gp = None
    if gamma_bits is not None:
        g = _c(gamma_bits, np.uint16).ravel()
        gp = _ptr(g)
    lib.orc_gemv_bf16(_ptr(w), n, k, _ptr(x), gp, eps, _ptr(xh), _ptr(r), _ptr(y), _ptr(a))
    return y, a, xh, r[0]


# --------------------------------------------------------------------------
# composite steps, in the pages' order
# --------------------------------------------------------------------------

def hadamard128(x) -> np.ndarray:
    """z f64[n]: the order-128 Walsh-Hadamard transform (Sylvester order,
    unnormalised) of each consecutive block of 128 values of x (f32)."""
    lib = _load()
    x = _c(x, np.float32).ravel()
    if x.size % 128:
        raise ValueError("n must be a multiple of 128")
    z = np.empty(x.size, np.float64)
    lib.orc_hadamard128(_ptr(x), x.size, _ptr(z))
    return z


def rmsnorm_hadamard(x, gamma, eps: float):
    """x_hat = (x * r) * gamma (orc_rmsnorm_quantize's), then its rotation z
    (f64) and the magnitude sum a of the 128 terms of each z value."""
    _, _, r, xh = rmsnorm_quantize(x, gamma, eps)
    z = hadamard128(xh)
    a = np.repeat(np.abs(xh.astype(np.float64)).reshape(-1, 128).sum(1), 128)
    return z, a, r, xh


def residual_add(res, y) -> np.ndarray:
    """out f64[n] = res (f32) + y (f64)."""
    lib = _load()
    r = _c(res, np.float32).ravel()
    y = _c(y, np.float64).ravel()
    out = np.empty(r.size, np.float64)
    lib.orc_residual_add(_ptr(r), _ptr(y), r.size, _ptr(out))
    return out


def decode_ffn(x, gamma, eps, gu_qs, gu_d, dn_qs, dn_d):
    """One decode FFN: RMSNorm -> Q8_0 -> stacked gate|up -> SiLU(g)*u -> Q8_0 -> down + x
    (orc_decode_ffn, every step in C).

    Returns a dict with every intermediate: f64 exact values ("*64"), their
    magnitude sums ("a_*"), and the f32 values the step hands on ("h", "out").
    """
    lib = _load()
    x = _c(x, np.float32).ravel()
    g = _c(gamma, np.float32).ravel()
    gq, gd = _c(gu_qs, np.int8), _c(gu_d, np.uint16)
    dq, dd = _c(dn_qs, np.int8), _c(dn_d, np.uint16)
    k = x.size
    F = gq.shape[0] // 2
    if g.size != k or gq.shape != (2 * F, k) or gd.shape != (2 * F, k // 32) or dq.shape != (k, F) \
            or dd.shape != (k, F // 32):
        raise ValueError("bad shapes")
    xq = np.empty(k, np.int8)
    xd = np.empty(k // 32, np.uint16)
    r = np.zeros(1, np.float32)
    gu = np.empty(2 * F, np.float64)
    a_gu = np.empty(2 * F, np.float64)
    h64 = np.empty(F, np.float64)
    h = np.empty(F, np.float32)
    hq = np.empty(F, np.int8)
    hd = np.empty(F // 32, np.uint16)
    y = np.empty(k, np.float64)
    a_y = np.empty(k, np.float64)
    out64 = np.empty(k, np.float64)
    lib.orc_decode_ffn(_ptr(x), _ptr(g), k, F, eps, _ptr(gq), _ptr(gd), _ptr(dq), _ptr(dd), _ptr(xq), _ptr(xd),
                       _ptr(r), _ptr(gu), _ptr(a_gu), _ptr(h64), _ptr(h), _ptr(hq), _ptr(hd), _ptr(y), _ptr(a_y),
                       _ptr(out64))
    return {
        "xq": xq, "xd": xd, "r": r[0],
        "gu64": gu, "a_gu": a_gu, "h64": h64, "h": h,
        "hq": hq[None, :], "hd": hd[None, :], "y64": y, "a_y": a_y,
        "out64": out64, "out": out64.astype(np.float32),
    }
