"""CPU checks of the C ABI: the library builds, loads, exports every symbol
include/qgemv.h declares, and rejects bad arguments before touching CUDA.

No call here reaches a kernel: every argument error is detected on the host
before any CUDA runtime call, which is what lets these run without a GPU.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemv.h")


@pytest.fixture(scope="module")
def lib():
    from block_quantized_decode_rmsnorm_gb300 import _lib, build

    build()
    return _lib.load()


def _declared():
    src = open(HEADER).read()
    return re.findall(r"QG_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_header_declares_the_boundary():
    names = set(_declared())
    for need in ["qgemv_q8_0", "qgemv_bf16", "quantize_act_q8_0", "rmsnorm_quantize", "qgemm_q8_0_prefill",
                 "qg_q8_0_pack", "qg_debug_block_dots_q8_0", "qg_status_str", "qg_abi_version"]:
        assert need in names


def test_every_declared_symbol_is_exported(lib):
    from block_quantized_decode_rmsnorm_gb300 import _lib

    for name in _declared():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"
    assert lib.qg_abi_version() == 1


def test_status_strings(lib):
    assert lib.qg_status_str(0) == b"ok"
    assert lib.qg_status_str(3) == b"bad shape"
    assert lib.qg_status_str(99) == b"unknown status"


def test_binding_scale_planes_match_the_library_stride(lib):
    """F16Codes allocates its block-major scale plane with the library's row
    stride (qg_scales_ld), for every residue of the row count."""
    torch = pytest.importorskip("torch")
    from block_quantized_decode_rmsnorm_gb300.api import F16Codes

    for rows in (1, 2, 3, 4, 5, 37, 128, 7169):
        c = F16Codes.empty(rows, 64, "cpu")
        assert c.codes.shape == (rows, 64) and c.codes.dtype == torch.float16
        assert c.scales_t.shape == (2, lib.qg_scales_ld(rows))
        with pytest.raises(ValueError):  # the library's kernels only read device memory here
            c.check("x")


def test_boundary_is_usable_from_c(lib):
    """The header is ISO C11 (warnings as errors, -pedantic), and a C program
    linked against the library gets its status codes back.  Argument errors
    only, so no GPU is needed."""
    import shutil
    import subprocess

    from block_quantized_decode_rmsnorm_gb300 import _lib

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from pathlib import Path

    work = Path(ROOT) / "block_quantized_decode_rmsnorm_gb300" / "_build" / "c_abi_check"  # git-ignored
    work.mkdir(parents=True, exist_ok=True)
    src = work / "use_qgemv.c"
    src.write_text(r"""
#include <stdint.h>
#include <stdio.h>
#include "qgemv.h"
#define FAKE ((void *)(uintptr_t)0x100000) /* well aligned, never dereferenced */
int main(void)
{
    if (qg_abi_version() != 1) return 1;
    /* k not a multiple of 32 */
    if (qgemv_q8_0(FAKE, FAKE, 8, 48, FAKE, FAKE, 1, QG_EPI_NONE, NULL, FAKE, NULL) != QG_ERR_SHAPE) return 2;
    /* a required pointer missing */
    if (quantize_act_q8_0(NULL, 1, 32, FAKE, FAKE, NULL) != QG_ERR_NULL) return 3;
    /* nothing to do */
    if (qgemm_q8_0_prefill_tc2(NULL, NULL, 0, 256, NULL, NULL, 0, NULL, 0, NULL) != QG_OK) return 4;
    printf("%s|%s\n", qg_status_str(QG_ERR_ALIGN), qg_status_str(QG_OK));
    return 0;
}
""")
    exe = work / "use_qgemv"
    libdir = os.path.dirname(_lib.LIB_PATH)
    cudalib = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64")
    subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", f"-I{os.path.join(ROOT, 'include')}",
                    str(src), "-o", str(exe), f"-L{libdir}", "-lqgemv", f"-Wl,-rpath,{libdir}",
                    f"-Wl,-rpath-link,{cudalib}"], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out
    assert out.stdout.strip() == f"{lib.qg_status_str(2).decode()}|{lib.qg_status_str(0).decode()}"


FAKE = 1 << 20  # a well-aligned, never-dereferenced address


def test_gemv_argument_errors(lib):
    q = lib.qgemv_q8_0
    # K not a multiple of 32
    assert q(FAKE, FAKE, 8, 48, FAKE, FAKE, 1, 0, None, FAKE, None) == 3
    # negative rows, zero batch
    assert q(FAKE, FAKE, -1, 64, FAKE, FAKE, 1, 0, None, FAKE, None) == 3
    assert q(FAKE, FAKE, 8, 64, FAKE, FAKE, 0, 0, None, FAKE, None) == 3
    # batch beyond what the kernels serve
    assert q(FAKE, FAKE, 8, 64, FAKE, FAKE, 9, 0, None, FAKE, None) == 4
    # unknown epilogue
    assert q(FAKE, FAKE, 8, 64, FAKE, FAKE, 1, 7, None, FAKE, None) == 4
    # odd rows for the stacked-halves epilogue
    assert q(FAKE, FAKE, 7, 64, FAKE, FAKE, 1, 1, None, FAKE, None) == 3
    # null pointers
    assert q(None, FAKE, 8, 64, FAKE, FAKE, 1, 0, None, FAKE, None) == 1
    assert q(FAKE, FAKE, 8, 64, FAKE, FAKE, 1, 2, None, FAKE, None) == 1  # residual missing
    # weight values must be 32-byte aligned, activations 16
    assert q(FAKE + 16, FAKE, 8, 64, FAKE, FAKE, 1, 0, None, FAKE, None) == 2
    assert q(FAKE, FAKE, 8, 64, FAKE + 8, FAKE, 1, 0, None, FAKE, None) == 2
    # zero rows is a valid no-op (nothing launched)
    assert q(None, None, 0, 64, None, None, 1, 0, None, None, None) == 0


def test_other_argument_errors(lib):
    assert lib.quantize_act_q8_0(FAKE, 1, 33, FAKE, FAKE, None) == 3
    assert lib.quantize_act_q8_0(None, 1, 32, FAKE, FAKE, None) == 1
    assert lib.quantize_act_q8_0(FAKE + 4, 1, 32, FAKE, FAKE, None) == 2
    assert lib.quantize_act_q8_0(None, 0, 32, None, None, None) == 0
    assert lib.rmsnorm_quantize(FAKE, FAKE, 1, 65536 + 32, ctypes.c_float(1e-6), FAKE, FAKE, None, None) == 3
    assert lib.rmsnorm_quantize(FAKE, FAKE, 1, 64, ctypes.c_float(-1.0), FAKE, FAKE, None, None) == 3
    assert lib.rmsnorm_quantize(FAKE, None, 1, 64, ctypes.c_float(1e-6), FAKE, FAKE, None, None) == 1
    assert lib.qgemv_bf16(FAKE, 8, 12, FAKE, None, ctypes.c_float(0.0), 0, None, FAKE, None) == 3
    assert lib.qgemv_bf16(FAKE + 8, 8, 16, FAKE, None, ctypes.c_float(0.0), 0, None, FAKE, None) == 2
    assert lib.qgemm_q8_0_prefill(FAKE, FAKE, 8, 64, FAKE, FAKE, -1, FAKE, None) == 3
    assert lib.qgemm_q8_0_prefill(FAKE, FAKE, 8, 64, FAKE, FAKE, 0, FAKE, None) == 0
    assert lib.qg_q8_0_pack(FAKE, 4, 64, FAKE + 16, FAKE, None) == 2
    assert lib.qg_debug_block_dots_q8_0(FAKE, 4, 64, FAKE, 9, FAKE, None) == 3


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    from block_quantized_decode_rmsnorm_gb300 import api

    with pytest.raises(ValueError, match="CUDA"):
        api.quantize_act_q8_0(torch.zeros(1, 32))


def test_fused_ffn_argument_errors(lib):
    f = lib.qg_ffn_up_q8_0
    eps = ctypes.c_float(1e-6)
    # hidden must be a multiple of 256 and at most 2048 for the one-launch path
    assert f(FAKE, FAKE, 992, eps, FAKE, FAKE, 64, FAKE, FAKE, FAKE, None, None, None, None) == 4
    assert f(FAKE, FAKE, 4096, eps, FAKE, FAKE, 64, FAKE, FAKE, FAKE, None, None, None, None) == 4
    # ffn must be a multiple of 32
    assert f(FAKE, FAKE, 1024, eps, FAKE, FAKE, 48, FAKE, FAKE, FAKE, None, None, None, None) == 3
    # the weight scale plane must be 16-byte aligned (it is staged in 16-byte pieces)
    assert f(FAKE, FAKE, 1024, eps, FAKE, FAKE + 2, 64, FAKE, FAKE, FAKE, None, None, None, None) == 2
    assert f(FAKE, None, 1024, eps, FAKE, FAKE, 64, FAKE, FAKE, FAKE, None, None, None, None) == 1
    d = lib.qg_decode_ffn_q8_0
    assert d(FAKE, FAKE, 1024, 3584, eps, FAKE, FAKE, FAKE, FAKE + 2, FAKE, FAKE, FAKE, None) == 2
    assert d(FAKE, FAKE, 1024, 3584, eps, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 16, FAKE, None) == 2
    assert d(FAKE, FAKE, 1024, 0, eps, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 3


def test_decode_ffn_out_argument_errors(lib):
    f = lib.qg_decode_ffn_q8_0_out
    eps = ctypes.c_float(1e-6)
    g = 1 << 20
    XI, XO = FAKE, FAKE + 8 * g
    args = lambda xi, xo, hidden=1024: (xi, xo, FAKE + 2 * g, hidden, 3584, eps, FAKE + 3 * g, FAKE + 4 * g,
                                        FAKE + 5 * g, FAKE + 6 * g, FAKE + 7 * g, FAKE + 9 * g, FAKE + 10 * g, None)
    # partial overlap of input and output (in place, xi == xo, is allowed)
    assert f(*args(XI, XI + 64)) == 3
    assert f(*args(XI + 4, XO)) == 2
    assert f(*args(XI, XO + 8)) == 2
    assert f(*args(None, XO)) == 1
    assert f(*args(XI, None)) == 1
    assert f(*args(XI, XO, 992)) == 4


def test_prefill_tc_argument_errors(lib):
    tc = lib.qgemm_q8_0_prefill_tc
    # K must be a multiple of 256 for the tensor-core path
    assert tc(FAKE, FAKE, 8, 96, FAKE, 1, FAKE, 0, None) == 4
    # weight scales 16-byte aligned (they are fetched with the tensor-memory accelerator)
    assert tc(FAKE, FAKE + 2, 8, 256, FAKE, 1, FAKE, 0, None) == 2
    # tile widths 0 (library's choice), 64, 96, 128 only
    assert tc(FAKE, FAKE, 8, 256, FAKE, 1, FAKE, 80, None) == 4
    assert tc(FAKE, FAKE, 8, 256, FAKE, 0, FAKE, 0, None) == 0
    assert tc(FAKE, FAKE, 8, 256, FAKE, (1 << 24) + 1, FAKE, 0, None) == 3
    assert tc(None, FAKE, 8, 256, FAKE, 1, FAKE, 0, None) == 1


def test_prefill_tc2_argument_errors(lib):
    assert lib.qg_scales_ld(0) == 0 and lib.qg_scales_ld(1) == 4 and lib.qg_scales_ld(512) == 512
    assert lib.qg_scales_ld(7169) == 7172 and lib.qg_scales_ld(-1) == -1
    g = 1 << 28  # operands placed far apart so that only the checked property fails
    W, WS, X, XS, Y = FAKE, FAKE + g, FAKE + 2 * g, FAKE + 3 * g, FAKE + 4 * g
    tc2 = lib.qgemm_q8_0_prefill_tc2
    assert tc2(W, WS, 64, 48, X, XS, 5, Y, 0, None) == 3           # k a multiple of 32
    assert tc2(W, WS, 64, 256, X, XS, (1 << 24) + 1, Y, 0, None) == 3
    assert tc2(W, WS, 64, 256, X, XS, 5, Y, 64, None) == 4         # tile widths 0, 128, 192
    assert tc2(W, WS, 64, 256, X, XS, 5, Y + 8, 0, None) == 2
    assert tc2(W, WS + 4, 64, 256, X, XS, 5, Y, 0, None) == 2
    assert tc2(W, WS, 64, 256, X, None, 5, Y, 0, None) == 1
    assert tc2(W, WS, 64, 256, X, XS, 5, X + 64, 0, None) == 3     # y over the activation codes
    assert tc2(None, None, 64, 256, None, None, 0, None, 0, None) == 0
    pk = lib.qg_q8_0_pack_f16
    assert pk(W, WS, 8, 40, X, XS, None) == 3
    assert pk(W + 4, WS, 8, 64, X, XS, None) == 2
    assert pk(W, WS, 8, 64, X + 8, XS, None) == 2
    assert pk(W, WS, 8, 64, None, XS, None) == 1
    assert pk(W, WS, 8, 64, W + 64, XS, None) == 3                 # codes over the int8 plane
    qa = lib.quantize_act_q8_0_f16
    assert qa(X, 3, 33, W, WS, None) == 3
    assert qa(X + 4, 3, 64, W, WS, None) == 2
    assert qa(X, 3, 64, W, None, None) == 1
    assert qa(X, 3, 64, X + 128, WS, None) == 3
    assert qa(None, 0, 64, None, None, None) == 0


def test_act_tiles_size_and_errors(lib):
    # one record of 8192 code bytes + 256 scale bytes per (128-row tile, block)
    assert lib.qg_act_tiles_bytes(130, 256) == 2 * 8 * 8448
    assert lib.qg_act_tiles_bytes(128, 32) == 8448
    assert lib.qg_act_tiles_bytes(0, 64) == 0
    assert lib.qg_act_tiles_bytes(1, 33) == -1
    assert lib.qg_act_tiles_bytes((1 << 24) + 1, 32) == -1
    qt = lib.quantize_act_q8_0_tiles
    assert qt(FAKE, 1, 48, FAKE, None) == 3
    assert qt(FAKE, 1, 64, FAKE + 8, None) == 2
    assert qt(None, 1, 64, FAKE, None) == 1
    assert qt(None, 0, 64, None, None) == 0


def test_one_launch_layer_argument_errors(lib):
    f = lib.qg_decode_layer_q8_0
    eps = ctypes.c_float(1e-6)
    xb, pb = 4096, 14 * 4096
    RI, PI, RO, PO = FAKE, FAKE + xb, FAKE + xb + pb, FAKE + 2 * xb + pb
    args = lambda ri, pi, n, ro, po, hidden=1024, ffn=3584: (ri, pi, n, ro, po, FAKE, hidden, ffn, eps, FAKE, FAKE,
                                                             FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert lib.qg_decode_layer_partials(1024, 3584) == 14
    assert lib.qg_decode_layer_partials(256, 96) == 3
    assert lib.qg_decode_layer_partials(2048, 1024) == 4
    assert lib.qg_decode_layer_partials(2304, 1024) == -1
    # hidden beyond 2048, hidden not a multiple of 256, too many partials
    assert f(*args(RI, PI, 14, RO, PO, 2304, 1024)) == 4
    assert f(*args(RI, PI, 14, RO, PO, 992, 3584)) == 4
    assert f(*args(RI, PI, 14, RO, PO, 1024, 32 * 8 * 17)) == 4
    assert f(*args(RI, PI, 17, RO, PO)) == 3
    # outputs overlapping inputs or each other
    assert f(*args(RI, PI, 14, RI, PO)) == 3
    assert f(*args(RI, PI, 14, RO, PI + 4096)) == 3
    assert f(*args(RI, PI, 14, RO, RO)) == 3
    # alignment, null partials with n_in > 0, null output
    assert f(*args(RI + 4, PI, 14, RO, PO)) == 2
    assert f(*args(RI, None, 14, RO, PO)) == 1
    assert f(*args(RI, PI, 14, None, PO)) == 1
    assert lib.qg_copy_stalls(None, 0) == 1
    fin = lib.qg_decode_layer_finish
    assert fin(FAKE, FAKE, 17, 1024, FAKE, None) == 3
    assert fin(FAKE, None, 2, 1024, FAKE, None) == 1
    assert fin(None, None, 0, 0, None, None) == 0


def test_noalloc_stack_argument_errors(lib):
    f = lib.qg_decode_layers_q8_0_noalloc
    eps = ctypes.c_float(1e-6)
    arr = (ctypes.c_void_p * 1)(FAKE)
    # intermediates larger than the fixed scratch array: refused before any launch.
    # The one-launch layer itself serves this shape (16 partials), so the refusal
    # is the scratch array's, not the layer's.
    assert lib.qg_decode_layer_partials(1792, 4096) == 16
    assert f(FAKE, FAKE, 1, arr, arr, arr, arr, arr, 1792, 4096, eps, None) == 4
    # the largest ffn the one-launch layer serves at hidden 1024 fits the array
    assert lib.qg_decode_layer_partials(1024, 4096) == 16
    assert lib.qg_decode_layer_partials(1024, 4096 + 256) == -1
    # unsupported layer shape, negative count
    assert f(FAKE, FAKE, 1, arr, arr, arr, arr, arr, 2304, 1024, eps, None) == 4
    assert f(FAKE, FAKE, -1, arr, arr, arr, arr, arr, 1024, 3584, eps, None) == 3
    # null pointer arrays / entries, misaligned input
    assert f(FAKE, FAKE, 1, None, arr, arr, arr, arr, 1024, 3584, eps, None) == 1
    nul = (ctypes.c_void_p * 1)(None)
    assert f(FAKE, FAKE, 1, arr, nul, arr, arr, arr, 1024, 3584, eps, None) == 1
    assert f(FAKE + 4, FAKE, 1, arr, arr, arr, arr, arr, 1024, 3584, eps, None) == 2
    assert f(None, FAKE, 0, None, None, None, None, None, 1024, 3584, eps, None) == 1


def test_bf16_prefill_argument_errors(lib):
    """qgemm_bf16_prefill refuses bad requests before anything is launched."""
    q = lib.qgemm_bf16_prefill
    e = ctypes.c_float(1e-6)
    # w, n_rows, k, x, m, gamma, eps, epilogue, xhat, y, stream
    assert q(FAKE, 8, 12, FAKE, 4, None, e, 0, None, FAKE, None) == 3      # k not a multiple of 8
    assert q(FAKE, 8, 16, FAKE, -1, None, e, 0, None, FAKE, None) == 3     # negative m
    assert q(FAKE, 7, 16, FAKE, 4, None, e, 1, None, FAKE, None) == 3      # odd rows for SiLU(g)*u
    assert q(FAKE, 8, 16, FAKE, 4, None, e, 2, None, FAKE, None) == 4      # residual epilogue not served
    assert q(FAKE, 8, 16, FAKE, 4, FAKE, e, 0, None, FAKE, None) == 1      # gamma without its work buffer
    assert q(FAKE + 8, 8, 16, FAKE, 4, None, e, 0, None, FAKE, None) == 2  # weights not 16-byte aligned
    assert q(FAKE, 8, 16, FAKE, 4, FAKE, e, 0, FAKE, FAKE, None) == 3      # work buffer overlaps x
    assert q(FAKE, 8, 16, FAKE + 4096, 4, None, e, 0, None, FAKE + 4096, None) == 3  # y overlaps x
    assert q(FAKE, 8, 16, FAKE + 4096, 4, FAKE + 8192, e, 0, FAKE + 16384, FAKE, None) == 3  # y overlaps w
    assert q(None, 0, 16, None, 4, None, e, 0, None, None, None) == 0      # no rows: nothing to do


def test_measure_mma_s8_argument_errors(lib):
    ops = ctypes.c_int64(0)
    assert lib.qg_measure_mma_s8(0, FAKE, ctypes.addressof(ops), None) == 3          # no rounds
    assert lib.qg_measure_mma_s8((1 << 24) + 1, FAKE, ctypes.addressof(ops), None) == 3
    assert lib.qg_measure_mma_s8(10, None, ctypes.addressof(ops), None) == 1          # no sink
    assert lib.qg_measure_mma_s8(10, FAKE, None, None) == 1                           # nowhere to report


def test_decode_stack_argument_errors(lib):
    """qg_decode_stack_q8_0 refuses bad requests before anything is launched."""
    f = lib.qg_decode_stack_q8_0
    eps = ctypes.c_float(1e-6)
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    nul = (ctypes.c_void_p * 2)(FAKE, None)
    mis = (ctypes.c_void_p * 2)(FAKE, FAKE + 16)  # a value plane 16- but not 32-byte aligned
    assert lib.qg_decode_stack_max_layers() == 64
    wsb = lib.qg_decode_stack_workspace_bytes(1024, 3584)
    assert wsb > 256 + 8 * (1024 + 3584 // 4 + 3584 // 32)
    assert lib.qg_decode_stack_workspace_bytes(2048, 3584) == -1  # hidden beyond one K block per lane group
    assert lib.qg_decode_stack_workspace_bytes(1024, 4096 + 256) == -1
    assert lib.qg_decode_stack_workspace_bytes(992, 3584) == -1  # hidden not a multiple of 256
    X, Y, WS = FAKE, FAKE + (1 << 16), FAKE + (1 << 20)

    def call(x=X, y=Y, n=2, g=arr, gq=arr, gd=arr, dq=arr, dd=arr, hidden=1024, ffn=3584, e=eps, ws=WS,
             h=None, hq=None, hd=None, limit=0):
        return f(x, y, n, g, gq, gd, dq, dd, hidden, ffn, e, ws, h, hq, hd, limit, None)

    assert call(n=0) == 3 and call(n=65) == 3          # layer count
    assert call(e=ctypes.c_float(-1.0)) == 3           # negative eps
    assert call(limit=-5) == 3                         # negative wait limit
    assert call(hidden=992) == 4 and call(ffn=3584 + 32) == 4 and call(hidden=2048) == 4
    assert call(ws=None) == 1 and call(x=None) == 1 and call(gq=None) == 1 and call(dd=nul) == 1
    assert call(ws=WS + 128) == 2 and call(x=X + 4) == 2 and call(gq=mis) == 2 and call(h=FAKE + 2) == 2
    assert call(y=X + 64) == 3                         # output overlapping the input in part
    assert call(y=WS + 4096) == 3                      # output inside the workspace
    assert call(h=WS) == 3                             # h_last inside the workspace
