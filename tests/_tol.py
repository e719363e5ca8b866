"""Tolerance model for comparing f32 GPU results with the f64 oracle.

Element-wise relative error is meaningless where a dot product cancels to
near zero, so each output is compared against the size of what was summed:

    e_n = |y_gpu - y_exact| / A_n,   A_n = sum of |terms| of output n

Any f32 summation order with depth D satisfies e_n <= D * 2^-24 (plus one
rounding of the result), so e_n <= TOL_Q8 = 1e-5 is a sound bar for the Q8_0
path and TOL_BF16 = 2e-3 for the bf16 path.  Through the epilogues the scale is
propagated to first order:

    SiLU(g)*u:  A_h = |silu'(g)| * A_g * |u| + |silu(g)| * A_u + |h|
    residual:   A_o = A_y + |res| + |out|
"""

import numpy as np

TOL_Q8 = 1e-5
TOL_BF16 = 2e-3
# An f32 result below the normal range is rounded to a multiple of 2^-149, so it
# may differ from the exact value by half of that whatever the scale: that much
# absolute slack is granted on top of the normalised bound.
F32_SUBNORMAL_HALF_ULP = 2.0 ** -150


def norm_err(y_gpu, y_exact, a) -> np.ndarray:
    y_gpu = np.asarray(y_gpu, np.float64)
    a = np.maximum(np.asarray(a, np.float64), np.finfo(np.float64).tiny)
    d = np.abs(y_gpu - np.asarray(y_exact, np.float64))
    return np.maximum(d - F32_SUBNORMAL_HALF_ULP, 0.0) / a


def silu_scale(g, u, a_g, a_u, tol=TOL_Q8):
    """Scale for h = silu(g) * u.  The f32 value of silu(g) itself cannot be
    closer than 2^-150 to the exact one when it is subnormal, and that error is
    multiplied by |u|: the term |u| * 2^-150 / tol grants it."""
    g = np.asarray(g, np.float64)
    u = np.asarray(u, np.float64)
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    h = g * sig * u
    return (np.abs(dsilu) * a_g * np.abs(u) + np.abs(g * sig) * a_u + np.abs(h)
            + np.abs(u) * F32_SUBNORMAL_HALF_ULP / tol)


def assert_close(y_gpu, y_exact, a, tol, what=""):
    e = norm_err(y_gpu, y_exact, a)
    worst = int(np.argmax(e)) if e.size else 0
    assert e.size == 0 or e.max() <= tol, (
        f"{what}: max normalised error {e.max():.3e} > {tol:.1e} at {worst}: "
        f"gpu={np.ravel(y_gpu)[worst]!r} exact={np.ravel(y_exact)[worst]!r} scale={np.ravel(a)[worst]!r}")
    return float(e.max()) if e.size else 0.0
