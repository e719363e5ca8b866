"""ctypes view of libqgemv.so (the C ABI declared in include/qgemv.h).

There is no fallback: if the library is missing or a CUDA device is absent, the
calls raise.  Every step of the computation runs in the library's kernels.
"""

from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemv.so")

QG_OK, QG_ERR_NULL, QG_ERR_ALIGN, QG_ERR_SHAPE, QG_ERR_UNSUPPORTED, QG_ERR_CUDA = range(6)
QG_EPI_NONE, QG_EPI_SILU_MUL_HALVES, QG_EPI_RESIDUAL_ADD = 0, 1, 2

P = ctypes.c_void_p
I64 = ctypes.c_int64
F32 = ctypes.c_float
I32 = ctypes.c_int
ST = ctypes.c_int

# name -> (restype, argtypes), in the order of include/qgemv.h
SIGNATURES = {
    "qg_status_str": (ctypes.c_char_p, [ST]),
    "qg_abi_version": (I32, []),
    "qg_q8_0_pack": (ST, [P, I64, I64, P, P, P]),
    "qg_q8_0_column_blocks": (ST, [P, P, I64, I64, P, P, P]),
    "quantize_act_q8_0": (ST, [P, I64, I64, P, P, P]),
    "qg_act_tiles_bytes": (I64, [I64, I64]),
    "quantize_act_q8_0_tiles": (ST, [P, I64, I64, P, P]),
    "rmsnorm_quantize": (ST, [P, P, I64, I64, F32, P, P, P, P]),
    "rmsnorm_hadamard_quantize": (ST, [P, P, I64, I64, F32, P, P, P, P, P]),
    "qgemv_q8_0": (ST, [P, P, I64, I64, P, P, I64, I32, P, P, P]),
    "qgemv_bf16": (ST, [P, I64, I64, P, P, F32, I32, P, P, P]),
    "qgemm_q8_0_prefill": (ST, [P, P, I64, I64, P, P, I64, P, P]),
    "qgemm_q8_0_prefill_tc": (ST, [P, P, I64, I64, P, I64, P, I32, P]),
    "qgemm_bf16_prefill": (ST, [P, I64, I64, P, I64, P, F32, I32, P, P, P]),
    "qg_ffn_up_q8_0": (ST, [P, P, I64, F32, P, P, I64, P, P, P, P, P, P, P]),
    "qg_decode_ffn_q8_0": (ST, [P, P, I64, I64, F32, P, P, P, P, P, P, P, P]),
    "qg_decode_ffn_q8_0_out": (ST, [P, P, P, I64, I64, F32, P, P, P, P, P, P, P, P]),
    "qg_decode_ffn_q8_0_rotated": (ST, [P, P, P, I64, I64, F32, P, P, P, P, P, P, P, P, P, P]),
    "qg_decode_layer_q8_0": (ST, [P, P, I32, P, P, P, I64, I64, F32, P, P, P, P, P, P, P, P]),
    "qg_decode_layer_partials": (I32, [I64, I64]),
    "qg_decode_layer_finish": (ST, [P, P, I32, I64, P, P]),
    "qg_copy_stalls": (ST, [ctypes.POINTER(ctypes.c_uint32), I32]),
    "qg_decode_layers_q8_0_noalloc": (ST, [P, P, I32, P, P, P, P, P, I64, I64, F32, P]),
    "qg_decode_stack_workspace_bytes": (I64, [I64, I64]),
    "qg_decode_stack_max_layers": (I32, []),
    "qg_decode_stack_q8_0": (ST, [P, P, I32, P, P, P, P, P, I64, I64, F32, P, P, P, P, I64, P]),
    "qg_debug_block_dots_q8_0": (ST, [P, I64, I64, P, I64, P, P]),
    "qg_measure_mma_s8": (ST, [I64, P, P, P]),
    "qg_measure_hbm_read_sink_len": (I32, []),
    "qg_measure_hbm_read": (ST, [P, I64, P, I32, P]),
    "qg_measure_launch_chain": (ST, [I32, I32, I32, P]),
    "qg_scales_ld": (I64, [I64]),
    "qg_q8_0_pack_f16": (ST, [P, P, I64, I64, P, P, P]),
    "quantize_act_q8_0_f16": (ST, [P, I64, I64, P, P, P]),
    "qgemm_q8_0_prefill_tc2": (ST, [P, P, I64, I64, P, P, I64, P, I32, P]),
}

_lib = None
_lock = threading.Lock()


class QGError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


def load(path: str | None = None):
    """Load libqgemv.so once; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(
                    f"libqgemv.so not found at {p}: build it first "
                    "(python -m block_quantized_decode_rmsnorm_gb300.builder, or __graft_entry__.build())")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def call(name: str, *args) -> None:
    """Call a qg_status-returning entry point; raise QGError on failure."""
    lib = load()
    st = getattr(lib, name)(*args)
    if st != QG_OK:
        raise QGError(name, st, lib.qg_status_str(st).decode())


def raw(name: str, *args) -> int:
    """Call an entry point and return its status code without raising."""
    return getattr(load(), name)(*args)
