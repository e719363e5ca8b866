"""Torch-tensor front end of libqgemv.so: argument marshalling only.

Each function has the name of the C entry point it calls (include/qgemv.h),
checks dtypes, shapes and devices, allocates outputs that were not given (torch
owns all device memory), and passes raw pointers and the current CUDA stream.
All arithmetic happens in the library's kernels.

Tensor formats
--------------
* Q8_0 values: ``torch.int8 [rows, k]``; Q8_0 scales: ``torch.float16
  [rows, k/32]`` (the library reads the binary16 bit patterns).
* Weights in the packed layout: a ``Q8Weight(qs, d)`` pair as above.
* bf16 tensors: ``torch.bfloat16``.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

from . import _lib
from ._lib import QG_EPI_NONE, QG_EPI_RESIDUAL_ADD, QG_EPI_SILU_MUL_HALVES  # noqa: F401

EPILOGUES = {"none": QG_EPI_NONE, "silu_mul": QG_EPI_SILU_MUL_HALVES, "residual": QG_EPI_RESIDUAL_ADD}


@dataclass
class Q8Weight:
    """Packed Q8_0 weight: values int8 [n_rows, k] and binary16 scales [n_rows, k/32]."""

    qs: torch.Tensor
    d: torch.Tensor

    @property
    def n_rows(self) -> int:
        return self.qs.shape[0]

    @property
    def k(self) -> int:
        return self.qs.shape[1]

    @property
    def nbytes(self) -> int:
        return self.qs.numel() + 2 * self.d.numel()


def _stream_handle(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape=None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _as_2d(x: torch.Tensor) -> torch.Tensor:
    return x.unsqueeze(0) if x.dim() == 1 else x


# --------------------------------------------------------------------------
# entry points
# --------------------------------------------------------------------------

def qg_q8_0_pack(blocks: torch.Tensor, n_rows: int, k: int, out: Q8Weight | None = None, stream=None) -> Q8Weight:
    """Canonical 34-byte Q8_0 blocks (uint8, n_rows*(k/32)*34 bytes) -> packed planes."""
    _need(blocks, "blocks", torch.uint8)
    if blocks.numel() != n_rows * (k // 32) * 34:
        raise ValueError("blocks has the wrong number of bytes for n_rows, k")
    dev = blocks.device
    if out is None:
        out = Q8Weight(torch.empty((n_rows, k), dtype=torch.int8, device=dev),
                       torch.empty((n_rows, k // 32), dtype=torch.float16, device=dev))
    _need(out.qs, "out.qs", torch.int8, (n_rows, k))
    _need(out.d, "out.d", torch.float16, (n_rows, k // 32))
    _lib.call("qg_q8_0_pack", blocks.data_ptr(), n_rows, k, out.qs.data_ptr(), out.d.data_ptr(),
              _stream_handle(stream))
    return out


def quantize_act_q8_0(x: torch.Tensor, q: torch.Tensor | None = None, d: torch.Tensor | None = None, stream=None):
    """f32 [rows, k] (or [k]) -> (q int8 [rows, k], d float16 [rows, k/32])."""
    _need(x, "x", torch.float32)
    x2 = _as_2d(x)
    rows, k = x2.shape
    if q is None:
        q = torch.empty((rows, k), dtype=torch.int8, device=x.device)
    if d is None:
        d = torch.empty((rows, k // 32), dtype=torch.float16, device=x.device)
    _need(q, "q", torch.int8, (rows, k))
    _need(d, "d", torch.float16, (rows, k // 32))
    _lib.call("quantize_act_q8_0", x2.data_ptr(), rows, k, q.data_ptr(), d.data_ptr(), _stream_handle(stream))
    return q, d


class ActTiles:
    """Activation operand of qgemm_q8_0_prefill_tc: `rows` rows of width `k` as
    tensor-core tiles (a uint8 device buffer of qg_act_tiles_bytes(rows, k))."""

    def __init__(self, buf: torch.Tensor, rows: int, k: int):
        self.buf, self.rows, self.k = buf, rows, k

    @staticmethod
    def nbytes(rows: int, k: int) -> int:
        n = _lib.load().qg_act_tiles_bytes(rows, k)
        if n < 0:
            raise ValueError(f"activation tiles: unsupported shape rows={rows} k={k}")
        return n

    @classmethod
    def empty(cls, rows: int, k: int, device) -> "ActTiles":
        return cls(torch.empty((cls.nbytes(rows, k),), dtype=torch.uint8, device=device), rows, k)


def quantize_act_q8_0_tiles(x: torch.Tensor, out: ActTiles | None = None, stream=None) -> ActTiles:
    """f32 [rows, k] -> Q8_0 codes and scales as tensor-core activation tiles."""
    _need(x, "x", torch.float32)
    x2 = _as_2d(x)
    rows, k = x2.shape
    if out is None:
        out = ActTiles.empty(rows, k, x.device)
    if (out.rows, out.k) != (rows, k) or out.buf.numel() != ActTiles.nbytes(rows, k):
        raise ValueError("quantize_act_q8_0_tiles: output tiles of another shape")
    _need(out.buf, "out.buf", torch.uint8)
    _lib.call("quantize_act_q8_0_tiles", x2.data_ptr(), rows, k, out.buf.data_ptr(), _stream_handle(stream))
    return out


def rmsnorm_quantize(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, q=None, d=None, inv_rms=None,
                     stream=None):
    """RMSNorm(x) * gamma quantized to Q8_0; returns (q, d, inv_rms)."""
    _need(x, "x", torch.float32)
    x2 = _as_2d(x)
    rows, k = x2.shape
    _need(gamma, "gamma", torch.float32, (k,))
    if q is None:
        q = torch.empty((rows, k), dtype=torch.int8, device=x.device)
    if d is None:
        d = torch.empty((rows, k // 32), dtype=torch.float16, device=x.device)
    if inv_rms is None:
        inv_rms = torch.empty((rows,), dtype=torch.float32, device=x.device)
    _need(q, "q", torch.int8, (rows, k))
    _need(d, "d", torch.float16, (rows, k // 32))
    _need(inv_rms, "inv_rms", torch.float32, (rows,))
    _lib.call("rmsnorm_quantize", x2.data_ptr(), gamma.data_ptr(), rows, k, float(eps), q.data_ptr(), d.data_ptr(),
              inv_rms.data_ptr(), _stream_handle(stream))
    return q, d, inv_rms


def rmsnorm_hadamard_quantize(x: torch.Tensor, gamma: torch.Tensor, eps: float = 1e-6, q=None, d=None, z=None,
                              inv_rms=None, stream=None):
    """Per row: x_hat = RMSNorm(x) * gamma, rotated by the order-128 Walsh-Hadamard
    transform on each block of 128, then Q8_0 -> (q int8[rows][k], d f16[rows][k/32])."""
    x2 = _as_2d(x)
    rows, k = x2.shape
    _need(x2, "x", torch.float32)
    _need(gamma, "gamma", torch.float32, (k,))
    if q is None:
        q = torch.empty((rows, k), dtype=torch.int8, device=x.device)
    if d is None:
        d = torch.empty((rows, k // 32), dtype=torch.float16, device=x.device)
    _need(q, "q", torch.int8, (rows, k))
    _need(d, "d", torch.float16, (rows, k // 32))
    if z is not None:
        _need(z, "z", torch.float32, (rows, k))
    if inv_rms is not None:
        _need(inv_rms, "inv_rms", torch.float32, (rows,))
    _lib.call("rmsnorm_hadamard_quantize", x2.data_ptr(), gamma.data_ptr(), rows, k, float(eps), q.data_ptr(),
              d.data_ptr(), _ptr(z), _ptr(inv_rms), _stream_handle(stream))
    return q, d


def qgemv_q8_0(w: Q8Weight, xq: torch.Tensor, xd: torch.Tensor, epilogue: str | int = "none",
               residual: torch.Tensor | None = None, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Block-scaled Q8_0 GEMV; y f32 [batch, n_out]."""
    epi = EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)
    _need(w.qs, "w.qs", torch.int8)
    n_rows, k = w.qs.shape
    _need(w.d, "w.d", torch.float16, (n_rows, k // 32))
    xq2, xd2 = _as_2d(xq), _as_2d(xd)
    batch = xq2.shape[0]
    _need(xq2, "xq", torch.int8, (batch, k))
    _need(xd2, "xd", torch.float16, (batch, k // 32))
    n_out = n_rows // 2 if epi == QG_EPI_SILU_MUL_HALVES else n_rows
    if y is None:
        y = torch.empty((batch, n_out), dtype=torch.float32, device=w.qs.device)
    _need(_as_2d(y), "y", torch.float32, (batch, n_out))
    if residual is not None:
        _need(_as_2d(residual), "residual", torch.float32, (batch, n_rows))
    _lib.call("qgemv_q8_0", w.qs.data_ptr(), w.d.data_ptr(), n_rows, k, xq2.data_ptr(), xd2.data_ptr(), batch, epi,
              _ptr(residual), y.data_ptr(), _stream_handle(stream))
    return y


def qgemv_bf16(w: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor | None = None, eps: float = 1e-6,
               epilogue: str | int = "none", residual: torch.Tensor | None = None, y: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """bf16 GEMV with optional fused RMSNorm in front; y f32 [n_out]."""
    epi = EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)
    _need(w, "w", torch.bfloat16)
    n_rows, k = w.shape
    _need(x, "x", torch.bfloat16, (k,))
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (k,))
    n_out = n_rows // 2 if epi == QG_EPI_SILU_MUL_HALVES else n_rows
    if y is None:
        y = torch.empty((n_out,), dtype=torch.float32, device=w.device)
    _need(y, "y", torch.float32, (n_out,))
    if residual is not None:
        _need(residual, "residual", torch.float32, (n_rows,))
    _lib.call("qgemv_bf16", w.data_ptr(), n_rows, k, x.data_ptr(), _ptr(gamma), float(eps), epi, _ptr(residual),
              y.data_ptr(), _stream_handle(stream))
    return y


def qgemm_bf16_prefill(w: torch.Tensor, x: torch.Tensor, gamma: torch.Tensor | None = None, eps: float = 1e-6,
                       epilogue: str | int = "none", y: torch.Tensor | None = None,
                       xhat: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """qgemv_bf16 for m prompt rows at once on the tensor cores: x bf16 [m, k],
    w bf16 [n, k]; y f32 [m, n_out].  xhat (bf16 [m, k]) is the work buffer of
    the normalised rows, allocated here when not given and gamma is."""
    epi = EPILOGUES[epilogue] if isinstance(epilogue, str) else int(epilogue)
    _need(w, "w", torch.bfloat16)
    n_rows, k = w.shape
    if x.dim() != 2 or x.shape[1] != k:
        raise ValueError(f"x: expected [m, {k}], got {tuple(x.shape)}")
    _need(x, "x", torch.bfloat16, tuple(x.shape))
    m = x.shape[0]
    if gamma is not None:
        _need(gamma, "gamma", torch.bfloat16, (k,))
        if xhat is None:
            xhat = torch.empty((m, k), dtype=torch.bfloat16, device=w.device)
        _need(xhat, "xhat", torch.bfloat16, (m, k))
    n_out = n_rows // 2 if epi == QG_EPI_SILU_MUL_HALVES else n_rows
    if y is None:
        y = torch.empty((m, n_out), dtype=torch.float32, device=w.device)
    _need(y, "y", torch.float32, (m, n_out))
    _lib.call("qgemm_bf16_prefill", w.data_ptr(), n_rows, k, x.data_ptr(), m, _ptr(gamma), float(eps), epi,
              _ptr(xhat), y.data_ptr(), _stream_handle(stream))
    return y


def qgemm_q8_0_prefill(w: Q8Weight, xq: torch.Tensor, xd: torch.Tensor, y: torch.Tensor | None = None,
                       stream=None) -> torch.Tensor:
    """Prompt-sized block-scaled contraction; Y f32 [m, n_rows]."""
    _need(w.qs, "w.qs", torch.int8)
    n_rows, k = w.qs.shape
    _need(w.d, "w.d", torch.float16, (n_rows, k // 32))
    m = xq.shape[0]
    _need(xq, "xq", torch.int8, (m, k))
    _need(xd, "xd", torch.float16, (m, k // 32))
    if y is None:
        y = torch.empty((m, n_rows), dtype=torch.float32, device=w.qs.device)
    _need(y, "y", torch.float32, (m, n_rows))
    _lib.call("qgemm_q8_0_prefill", w.qs.data_ptr(), w.d.data_ptr(), n_rows, k, xq.data_ptr(), xd.data_ptr(), m,
              y.data_ptr(), _stream_handle(stream))
    return y


def qgemm_q8_0_prefill_tc(w: Q8Weight, xt: ActTiles, y: torch.Tensor | None = None, tile_n: int = 0,
                          stream=None) -> torch.Tensor:
    """Tensor-core prompt contraction; Y f32 [m, n_rows] from activation tiles of m rows."""
    _need(w.qs, "w.qs", torch.int8)
    n_rows, k = w.qs.shape
    _need(w.d, "w.d", torch.float16, (n_rows, k // 32))
    if xt.k != k:
        raise ValueError(f"qgemm_q8_0_prefill_tc: activation width {xt.k} != weight width {k}")
    _need(xt.buf, "xt.buf", torch.uint8)
    m = xt.rows
    if y is None:
        y = torch.empty((m, n_rows), dtype=torch.float32, device=w.qs.device)
    _need(y, "y", torch.float32, (m, n_rows))
    _lib.call("qgemm_q8_0_prefill_tc", w.qs.data_ptr(), w.d.data_ptr(), n_rows, k, xt.buf.data_ptr(), m,
              y.data_ptr(), tile_n, _stream_handle(stream))
    return y


@dataclass
class F16Codes:
    """Q8_0 operand of qgemm_q8_0_prefill_tc2: codes as binary16 ``torch.float16
    [rows, k]`` (exact integers) and scales as ``torch.float32 [k/32, ld]``, ld =
    rows rounded up to a multiple of four (columns past ``rows`` are padding)."""

    codes: torch.Tensor
    scales_t: torch.Tensor

    @property
    def rows(self) -> int:
        return self.codes.shape[0]

    @property
    def k(self) -> int:
        return self.codes.shape[1]

    @classmethod
    def empty(cls, rows: int, k: int, device) -> "F16Codes":
        return cls(torch.empty((rows, k), dtype=torch.float16, device=device),
                   torch.empty((k // 32, (rows + 3) // 4 * 4), dtype=torch.float32, device=device))

    def check(self, name: str) -> None:
        _need(self.codes, f"{name}.codes", torch.float16)
        _need(self.scales_t, f"{name}.scales_t", torch.float32, (self.k // 32, (self.rows + 3) // 4 * 4))


def qg_q8_0_pack_f16(w: Q8Weight, out: F16Codes | None = None, stream=None) -> F16Codes:
    """Packed Q8_0 weight -> binary16 codes and block-major f32 scales."""
    _need(w.qs, "w.qs", torch.int8)
    n_rows, k = w.qs.shape
    _need(w.d, "w.d", torch.float16, (n_rows, k // 32))
    if out is None:
        out = F16Codes.empty(n_rows, k, w.qs.device)
    out.check("out")
    if (out.rows, out.k) != (n_rows, k):
        raise ValueError("qg_q8_0_pack_f16: output of another shape")
    _lib.call("qg_q8_0_pack_f16", w.qs.data_ptr(), w.d.data_ptr(), n_rows, k, out.codes.data_ptr(),
              out.scales_t.data_ptr(), _stream_handle(stream))
    return out


def quantize_act_q8_0_f16(x: torch.Tensor, out: F16Codes | None = None, stream=None) -> F16Codes:
    """f32 [rows, k] -> Q8_0 codes as binary16 and block-major f32 scales."""
    _need(x, "x", torch.float32)
    x2 = _as_2d(x)
    rows, k = x2.shape
    if out is None:
        out = F16Codes.empty(rows, k, x.device)
    out.check("out")
    if (out.rows, out.k) != (rows, k):
        raise ValueError("quantize_act_q8_0_f16: output of another shape")
    _lib.call("quantize_act_q8_0_f16", x2.data_ptr(), rows, k, out.codes.data_ptr(), out.scales_t.data_ptr(),
              _stream_handle(stream))
    return out


def qgemm_q8_0_prefill_tc2(w: F16Codes, x: F16Codes, y: torch.Tensor | None = None, tile_n: int = 0,
                           stream=None) -> torch.Tensor:
    """Wide-tile tensor-core prompt contraction; Y f32 [m, n_rows]."""
    w.check("w")
    x.check("x")
    if x.k != w.k:
        raise ValueError(f"qgemm_q8_0_prefill_tc2: activation width {x.k} != weight width {w.k}")
    if y is None:
        y = torch.empty((x.rows, w.rows), dtype=torch.float32, device=w.codes.device)
    _need(y, "y", torch.float32, (x.rows, w.rows))
    _lib.call("qgemm_q8_0_prefill_tc2", w.codes.data_ptr(), w.scales_t.data_ptr(), w.rows, w.k,
              x.codes.data_ptr(), x.scales_t.data_ptr(), x.rows, y.data_ptr(), tile_n, _stream_handle(stream))
    return y


def qg_measure_mma_s8(iters: int, stream=None) -> int:
    """Launch the int8 mma.sync rate kernel (time the stream around it); returns
    the int-ops the launch performs."""
    import ctypes

    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    ops = ctypes.c_int64(0)
    _lib.call("qg_measure_mma_s8", int(iters), sink.data_ptr(), ctypes.addressof(ops), _stream_handle(stream))
    return ops.value


def qg_measure_hbm_read(buf: torch.Tensor, sink: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """One streaming read of the whole device buffer `buf` (the pure-read probe);
    returns the per-CTA fold words so that the caller can keep them alive."""
    n = _lib.load().qg_measure_hbm_read_sink_len()
    if sink is None:
        sink = torch.empty((n,), dtype=torch.int32, device=buf.device)
    _lib.call("qg_measure_hbm_read", buf.data_ptr(), buf.numel() * buf.element_size(), sink.data_ptr(), sink.numel(),
              _stream_handle(stream))
    return sink


def qg_measure_launch_chain(n: int, grid: int, block: int, stream=None) -> None:
    """n empty kernels with programmatic dependent launch (the launch floor)."""
    _lib.call("qg_measure_launch_chain", n, grid, block, _stream_handle(stream))


def qg_debug_block_dots_q8_0(w: Q8Weight, xq: torch.Tensor, s: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """Exact int32 block sums s[batch, n_rows, k/32]."""
    n_rows, k = w.qs.shape
    xq2 = _as_2d(xq)
    batch = xq2.shape[0]
    _need(xq2, "xq", torch.int8, (batch, k))
    if s is None:
        s = torch.empty((batch, n_rows, k // 32), dtype=torch.int32, device=w.qs.device)
    _need(s, "s", torch.int32, (batch, n_rows, k // 32))
    _lib.call("qg_debug_block_dots_q8_0", w.qs.data_ptr(), n_rows, k, xq2.data_ptr(), batch, s.data_ptr(),
              _stream_handle(stream))
    return s


# --------------------------------------------------------------------------
# composite: one decode FFN step (four launches, graph-capturable)
# --------------------------------------------------------------------------

@dataclass
class FFNLayer:
    """Weights of one decode feed-forward block: RMSNorm gain, stacked gate|up, down."""

    gamma: torch.Tensor  # f32 [hidden]
    gate_up: Q8Weight    # [2*ffn, hidden]
    down: Q8Weight       # [hidden, ffn]
    down_cb: "Q8Weight | None" = None  # down in the column-block layout (one-launch layer)

    @property
    def nbytes(self) -> int:
        return self.gate_up.nbytes + self.down.nbytes


@dataclass
class FFNBuffers:
    """Stable activation buffers reused by every step (graph replay needs fixed addresses)."""

    xq: torch.Tensor
    xd: torch.Tensor
    h: torch.Tensor
    hq: torch.Tensor
    hd: torch.Tensor

    @staticmethod
    def allocate(hidden: int, ffn: int, device) -> "FFNBuffers":
        return FFNBuffers(
            torch.empty((1, hidden), dtype=torch.int8, device=device),
            torch.empty((1, hidden // 32), dtype=torch.float16, device=device),
            torch.empty((1, ffn), dtype=torch.float32, device=device),
            torch.empty((1, ffn), dtype=torch.int8, device=device),
            torch.empty((1, ffn // 32), dtype=torch.float16, device=device),
        )


def decode_ffn_q8_0(x: torch.Tensor, layer: FFNLayer, buf: FFNBuffers, eps: float = 1e-6, stream=None) -> None:
    """x <- x + down(SiLU(gate(n)) * up(n)), n = Q8_0(RMSNorm(x) * gamma), in place.

    "Filling in the blanks: Inference using Phobos", Fast Decode: the activation
    is quantized once and shared, the projections reading it are stacked, and the
    residual add is folded into the last matmul.
    """
    s = _stream_handle(stream)
    hidden = x.shape[-1]
    ffn = layer.down.k
    _lib.call("rmsnorm_quantize", x.data_ptr(), layer.gamma.data_ptr(), 1, hidden, float(eps), buf.xq.data_ptr(),
              buf.xd.data_ptr(), None, s)
    _lib.call("qgemv_q8_0", layer.gate_up.qs.data_ptr(), layer.gate_up.d.data_ptr(), 2 * ffn, hidden,
              buf.xq.data_ptr(), buf.xd.data_ptr(), 1, QG_EPI_SILU_MUL_HALVES, None, buf.h.data_ptr(), s)
    _lib.call("quantize_act_q8_0", buf.h.data_ptr(), 1, ffn, buf.hq.data_ptr(), buf.hd.data_ptr(), s)
    _lib.call("qgemv_q8_0", layer.down.qs.data_ptr(), layer.down.d.data_ptr(), hidden, ffn, buf.hq.data_ptr(),
              buf.hd.data_ptr(), 1, QG_EPI_RESIDUAL_ADD, x.data_ptr(), x.data_ptr(), s)


def decode_ffn_q8_0_rotated(x: torch.Tensor, layer: FFNLayer, buf: FFNBuffers, eps: float = 1e-6,
                            stream=None) -> None:
    """decode_ffn_q8_0 with the normalised activation rotated once (order-128
    Walsh-Hadamard per block) before it is quantized, in four launches
    (rmsnorm_hadamard_quantize, the stacked gate|up GEMV with SiLU*u, Q8_0 of h,
    down with the residual); the stacked gate|up weights of `layer` are the
    rotated ones (W H^T / 128, quantized at load time), so both halves read the
    one rotated activation.

    "Filling in the blanks: Inference using Phobos", PrismML Ternary-Bonsai-2-27B:
    the rotated activation is computed once and shared by every projection that
    reads the same input.
    """
    s = _stream_handle(stream)
    hidden = x.shape[-1]
    ffn = layer.down.k
    _lib.call("rmsnorm_hadamard_quantize", x.data_ptr(), layer.gamma.data_ptr(), 1, hidden, float(eps),
              buf.xq.data_ptr(), buf.xd.data_ptr(), None, None, s)
    _lib.call("qgemv_q8_0", layer.gate_up.qs.data_ptr(), layer.gate_up.d.data_ptr(), 2 * ffn, hidden,
              buf.xq.data_ptr(), buf.xd.data_ptr(), 1, QG_EPI_SILU_MUL_HALVES, None, buf.h.data_ptr(), s)
    _lib.call("quantize_act_q8_0", buf.h.data_ptr(), 1, ffn, buf.hq.data_ptr(), buf.hd.data_ptr(), s)
    _lib.call("qgemv_q8_0", layer.down.qs.data_ptr(), layer.down.d.data_ptr(), hidden, ffn, buf.hq.data_ptr(),
              buf.hd.data_ptr(), 1, QG_EPI_RESIDUAL_ADD, x.data_ptr(), x.data_ptr(), s)


def qg_decode_ffn_q8_0_rotated(x_in: torch.Tensor, x_out: torch.Tensor, layer: FFNLayer, buf: FFNBuffers,
                               eps: float = 1e-6, export_codes: bool = False, stream=None) -> None:
    """The same layer in two launches: the fused gate|up kernel rotates the
    normalised activation itself (each CTA, one 128-value rotation per warp),
    quantizes it and shares it between the stacked halves; then the down GEMV
    with the residual.  With export_codes, buf.xq / buf.xd receive the rotated
    activation's codes and scales."""
    hidden = layer.gamma.shape[-1]
    ffn = layer.down.k
    _need_reachable(x_in, "x_in", (hidden,))
    _need_reachable(x_out, "x_out", (hidden,))
    _lib.call("qg_decode_ffn_q8_0_rotated", x_in.data_ptr(), x_out.data_ptr(), layer.gamma.data_ptr(), hidden, ffn,
              float(eps), layer.gate_up.qs.data_ptr(), layer.gate_up.d.data_ptr(), layer.down.qs.data_ptr(),
              layer.down.d.data_ptr(), buf.h.data_ptr(), buf.hq.data_ptr(), buf.hd.data_ptr(),
              buf.xq.data_ptr() if export_codes else None, buf.xd.data_ptr() if export_codes else None,
              _stream_handle(stream))


def qg_ffn_up_q8_0(x: torch.Tensor, gamma: torch.Tensor, w: Q8Weight, eps: float = 1e-6, h=None, hq=None, hd=None,
                   xq_out=None, xd_out=None, inv_rms_out=None, stream=None):
    """RMSNorm -> Q8_0 -> stacked gate|up -> SiLU(g)*u -> (h, hq, hd), one launch."""
    hidden = x.shape[-1]
    _need(x, "x", torch.float32, (hidden,))
    _need(gamma, "gamma", torch.float32, (hidden,))
    _need(w.qs, "w.qs", torch.int8)
    n_rows = w.qs.shape[0]
    ffn = n_rows // 2
    _need(w.qs, "w.qs", torch.int8, (2 * ffn, hidden))
    _need(w.d, "w.d", torch.float16, (2 * ffn, hidden // 32))
    dev = x.device
    if h is None:
        h = torch.empty((ffn,), dtype=torch.float32, device=dev)
    if hq is None:
        hq = torch.empty((ffn,), dtype=torch.int8, device=dev)
    if hd is None:
        hd = torch.empty((ffn // 32,), dtype=torch.float16, device=dev)
    _need(h, "h", torch.float32, (ffn,))
    _need(hq, "hq", torch.int8, (ffn,))
    _need(hd, "hd", torch.float16, (ffn // 32,))
    _lib.call("qg_ffn_up_q8_0", x.data_ptr(), gamma.data_ptr(), hidden, float(eps), w.qs.data_ptr(), w.d.data_ptr(),
              ffn, h.data_ptr(), hq.data_ptr(), hd.data_ptr(), _ptr(xq_out), _ptr(xd_out), _ptr(inv_rms_out),
              _stream_handle(stream))
    return h, hq, hd


def qg_decode_ffn_q8_0(x: torch.Tensor, layer: FFNLayer, buf: FFNBuffers, eps: float = 1e-6, stream=None) -> None:
    """x <- x + down(SiLU(g)*u) in two launches (fused gate|up, then down + residual)."""
    hidden = x.shape[-1]
    ffn = layer.down.k
    _lib.call("qg_decode_ffn_q8_0", x.data_ptr(), layer.gamma.data_ptr(), hidden, ffn, float(eps),
              layer.gate_up.qs.data_ptr(), layer.gate_up.d.data_ptr(), layer.down.qs.data_ptr(),
              layer.down.d.data_ptr(), buf.h.data_ptr(), buf.hq.data_ptr(), buf.hd.data_ptr(), _stream_handle(stream))


def _need_reachable(t: torch.Tensor, name: str, shape) -> None:
    """f32 contiguous tensor on a CUDA device or in pinned host memory (which the
    kernels reach directly through unified addressing)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda or (t.device.type == "cpu" and t.is_pinned())):
        raise ValueError(f"{name} must be on a CUDA device or in pinned host memory")
    if t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be contiguous float32 of shape {tuple(shape)}")


def qg_decode_ffn_q8_0_out(x_in: torch.Tensor, x_out: torch.Tensor, layer: FFNLayer, buf: FFNBuffers,
                           eps: float = 1e-6, stream=None) -> None:
    """x_out <- x_in + down(SiLU(g)*u) in two launches; x_in / x_out may be pinned
    host tensors (the first layer of a step reading the host input, the last one
    writing the host result)."""
    hidden = layer.gamma.shape[-1]
    ffn = layer.down.k
    if x_in.numel() != hidden:
        raise ValueError(f"x_in must hold {hidden} values")
    _need_reachable(x_in, "x_in", x_in.shape)
    _need_reachable(x_out, "x_out", x_in.shape)
    _lib.call("qg_decode_ffn_q8_0_out", x_in.data_ptr(), x_out.data_ptr(), layer.gamma.data_ptr(), hidden, ffn,
              float(eps), layer.gate_up.qs.data_ptr(), layer.gate_up.d.data_ptr(), layer.down.qs.data_ptr(),
              layer.down.d.data_ptr(), buf.h.data_ptr(), buf.hq.data_ptr(), buf.hd.data_ptr(), _stream_handle(stream))


def qg_q8_0_column_blocks(w: Q8Weight, stream=None) -> Q8Weight:
    """Row-major planes -> column-block planes: values [k/32, n, 32], scales [k/32, n]
    (returned as a Q8Weight whose tensors have those shapes)."""
    n, k = w.qs.shape
    _need(w.qs, "w.qs", torch.int8, (n, k))
    _need(w.d, "w.d", torch.float16, (n, k // 32))
    out = Q8Weight(torch.empty((k // 32, n, 32), dtype=torch.int8, device=w.qs.device),
                   torch.empty((k // 32, n), dtype=torch.float16, device=w.qs.device))
    _lib.call("qg_q8_0_column_blocks", w.qs.data_ptr(), w.d.data_ptr(), n, k, out.qs.data_ptr(), out.d.data_ptr(),
              _stream_handle(stream))
    return out


def prepare_one_launch(layer: FFNLayer) -> FFNLayer:
    """Give the layer its down weights in the column-block layout (a one-time
    load step; allocates, so do it before capturing a graph)."""
    if layer.down_cb is None:
        layer.down_cb = qg_q8_0_column_blocks(layer.down)
    return layer


def qg_decode_layer_partials(hidden: int, ffn: int) -> int:
    n = _lib.load().qg_decode_layer_partials(hidden, ffn)
    if n < 0:
        raise ValueError(f"one-launch layer: unsupported shape hidden={hidden} ffn={ffn}")
    return n


def qg_decode_layer_q8_0(r_in: torch.Tensor, p_in: torch.Tensor | None, r_out: torch.Tensor, p_out: torch.Tensor,
                         layer: FFNLayer, buf: FFNBuffers, eps: float = 1e-6, stream=None) -> None:
    """One decode FFN layer in one launch on an unreduced input (r_in + rows of
    p_in); writes its input as r_out and its output's partials to p_out."""
    hidden = r_in.shape[-1]
    ffn = layer.down.k
    if layer.down_cb is None:
        raise ValueError("qg_decode_layer_q8_0 needs layer.down_cb (see prepare_one_launch)")
    _need(layer.down_cb.qs, "layer.down_cb.qs", torch.int8, (ffn // 32, hidden, 32))
    _need(layer.down_cb.d, "layer.down_cb.d", torch.float16, (ffn // 32, hidden))
    _need(r_in, "r_in", torch.float32, (hidden,))
    _need(r_out, "r_out", torch.float32, (hidden,))
    n_in = 0
    if p_in is not None:
        _need(p_in, "p_in", torch.float32)
        n_in = p_in.shape[0]
        _need(p_in, "p_in", torch.float32, (n_in, hidden))
    _need(p_out, "p_out", torch.float32, (qg_decode_layer_partials(hidden, ffn), hidden))
    _lib.call("qg_decode_layer_q8_0", r_in.data_ptr(), _ptr(p_in), n_in, r_out.data_ptr(), p_out.data_ptr(),
              layer.gamma.data_ptr(), hidden, ffn, float(eps), layer.gate_up.qs.data_ptr(), layer.gate_up.d.data_ptr(),
              layer.down_cb.qs.data_ptr(), layer.down_cb.d.data_ptr(), buf.h.data_ptr(), buf.hq.data_ptr(),
              buf.hd.data_ptr(), _stream_handle(stream))


def qg_decode_layer_finish(r: torch.Tensor, p: torch.Tensor | None, x: torch.Tensor | None = None,
                           stream=None) -> torch.Tensor:
    """x = r + sum of the rows of p, in row order."""
    hidden = r.shape[-1]
    _need(r, "r", torch.float32, (hidden,))
    n = 0 if p is None else p.shape[0]
    if p is not None:
        _need(p, "p", torch.float32, (n, hidden))
    if x is None:
        x = torch.empty_like(r)
    _need(x, "x", torch.float32, (hidden,))
    _lib.call("qg_decode_layer_finish", r.data_ptr(), _ptr(p), n, hidden, x.data_ptr(), _stream_handle(stream))
    return x


class LayerStack:
    """A stack of one-launch layers: two (r, partials) pairs used in turn, and
    the output as one vector in `out` (r + partials of the last layer)."""

    def __init__(self, hidden: int, ffn: int, device):
        n = qg_decode_layer_partials(hidden, ffn)
        self.r = [torch.zeros((hidden,), dtype=torch.float32, device=device) for _ in range(2)]
        self.p = [torch.zeros((n, hidden), dtype=torch.float32, device=device) for _ in range(2)]
        self.out = torch.zeros((hidden,), dtype=torch.float32, device=device)

    def load(self, x: torch.Tensor) -> None:
        self.r[0].copy_(x)

    def run(self, layers, buf: FFNBuffers, eps: float = 1e-6, stream=None) -> torch.Tensor:
        """Every layer (layer 0 reads r[0] alone), then the finish; returns `out`."""
        for l, layer in enumerate(layers):
            qg_decode_layer_q8_0(self.r[l % 2], self.p[l % 2] if l else None, self.r[(l + 1) % 2],
                                 self.p[(l + 1) % 2], layer, buf, eps, stream=stream)
        last = len(layers) % 2
        return qg_decode_layer_finish(self.r[last], self.p[last] if layers else None, self.out, stream=stream)


def qg_decode_layers_q8_0_noalloc(x_in: torch.Tensor, layers, eps: float = 1e-6, x_out: torch.Tensor | None = None,
                                  stream=None) -> torch.Tensor:
    """A stack of one-launch layers with the library's fixed scratch array instead
    of caller work buffers (layers need down_cb, see prepare_one_launch)."""
    import ctypes

    hidden = x_in.shape[-1]
    _need(x_in, "x_in", torch.float32, (hidden,))
    if x_out is None:
        x_out = torch.empty_like(x_in)
    _need(x_out, "x_out", torch.float32, (hidden,))
    n = len(layers)
    ffn = layers[0].down.k if n else 0
    for ly in layers:
        if ly.down_cb is None:
            raise ValueError("qg_decode_layers_q8_0_noalloc needs down_cb on every layer (see prepare_one_launch)")
    arr = lambda vals: (ctypes.c_void_p * max(n, 1))(*vals) if n else None
    g = arr([ly.gamma.data_ptr() for ly in layers])
    gq = arr([ly.gate_up.qs.data_ptr() for ly in layers])
    gd = arr([ly.gate_up.d.data_ptr() for ly in layers])
    dq = arr([ly.down_cb.qs.data_ptr() for ly in layers])
    dd = arr([ly.down_cb.d.data_ptr() for ly in layers])
    _lib.call("qg_decode_layers_q8_0_noalloc", x_in.data_ptr(), x_out.data_ptr(), n, g, gq, gd, dq, dd, hidden,
              ffn if n else 32, float(eps), _stream_handle(stream))
    return x_out


def copy_stalls(clear: bool = False) -> int:
    """Waits of the decode kernels on their staged weight copies that gave up
    on the current device since the last clear (qg_copy_stalls); 0 normally."""
    import ctypes

    n = ctypes.c_uint32(0)
    _lib.call("qg_copy_stalls", ctypes.byref(n), 1 if clear else 0)
    return int(n.value)


def qg_decode_stack_workspace_bytes(hidden: int, ffn: int) -> int:
    n = _lib.load().qg_decode_stack_workspace_bytes(hidden, ffn)
    if n < 0:
        raise ValueError(f"persistent decode stack: unsupported shape hidden={hidden} ffn={ffn}")
    return n


class DecodeStack:
    """Decode FFN layers run as one persistent launch per up to
    qg_decode_stack_max_layers() layers (qg_decode_stack_q8_0).

    "Filling in the blanks: Inference using Phobos", Q4_K_M: the whole MLP as
    one persistent kernel.  Owns the zero-filled workspace the launches share
    and the host arrays of the layers' device pointers; allocates nothing after
    construction, so run() can be captured into a CUDA graph.
    """

    def __init__(self, layers, device="cuda"):
        import ctypes

        self.layers = list(layers)
        if not self.layers:
            raise ValueError("DecodeStack needs at least one layer")
        self.hidden = self.layers[0].gamma.shape[-1]
        self.ffn = self.layers[0].down.k
        for ly in self.layers:
            _need(ly.gamma, "gamma", torch.float32, (self.hidden,))
            _need(ly.gate_up.qs, "gate_up.qs", torch.int8, (2 * self.ffn, self.hidden))
            _need(ly.gate_up.d, "gate_up.d", torch.float16, (2 * self.ffn, self.hidden // 32))
            _need(ly.down.qs, "down.qs", torch.int8, (self.hidden, self.ffn))
            _need(ly.down.d, "down.d", torch.float16, (self.hidden, self.ffn // 32))
        self.workspace = torch.zeros(qg_decode_stack_workspace_bytes(self.hidden, self.ffn), dtype=torch.uint8,
                                     device=device)
        self.chunk = _lib.load().qg_decode_stack_max_layers()
        self._arrays = []  # per chunk: (n, gamma, wgu_qs, wgu_d, wdn_qs, wdn_d) host pointer arrays
        for c0 in range(0, len(self.layers), self.chunk):
            ch = self.layers[c0:c0 + self.chunk]
            arr = lambda vals: (ctypes.c_void_p * len(vals))(*vals)
            self._arrays.append((len(ch), arr([ly.gamma.data_ptr() for ly in ch]),
                                 arr([ly.gate_up.qs.data_ptr() for ly in ch]),
                                 arr([ly.gate_up.d.data_ptr() for ly in ch]),
                                 arr([ly.down.qs.data_ptr() for ly in ch]),
                                 arr([ly.down.d.data_ptr() for ly in ch])))

    def run(self, x_in: torch.Tensor, x_out: torch.Tensor | None = None, eps: float = 1e-6, h_last=None,
            hq_last=None, hd_last=None, wait_limit_ns: int = 0, stream=None) -> torch.Tensor:
        """x_out <- the stack applied to x_in (either may be pinned host memory;
        x_out may be x_in).  h_last / hq_last / hd_last receive the last layer's
        activation and its Q8_0 codes and scales when given."""
        _need_reachable(x_in, "x_in", (self.hidden,))
        if x_out is None:
            x_out = torch.empty_like(x_in)
        _need_reachable(x_out, "x_out", (self.hidden,))
        if h_last is not None:
            _need(h_last, "h_last", torch.float32, (self.ffn,))
        if hq_last is not None:
            _need(hq_last, "hq_last", torch.int8, (self.ffn,))
        if hd_last is not None:
            _need(hd_last, "hd_last", torch.float16, (self.ffn // 32,))
        s = _stream_handle(stream)
        src = x_in
        for i, (n, g, gq, gd, dq, dd) in enumerate(self._arrays):
            last = i == len(self._arrays) - 1
            _lib.call("qg_decode_stack_q8_0", src.data_ptr(), x_out.data_ptr(), n, g, gq, gd, dq, dd, self.hidden,
                      self.ffn, float(eps), self.workspace.data_ptr(), _ptr(h_last) if last else None,
                      _ptr(hq_last) if last else None, _ptr(hd_last) if last else None, int(wait_limit_ns), s)
            src = x_out
        return x_out

    def status(self) -> int:
        """The workspace status word (0: every launch since the last reset completed
        normally).  Waits for the device."""
        return int(self.workspace[:4].view(torch.int32).item())

    def generation(self) -> int:
        """Launches completed on this workspace since the last reset (mod 2^32)."""
        return int(self.workspace[4:8].view(torch.int32).item()) & 0xFFFFFFFF

    def reset(self) -> None:
        """Zero-fill the workspace again (after a launch that set the status)."""
        self.workspace.zero_()


# --------------------------------------------------------------------------
# host <-> device helpers (plumbing)
# --------------------------------------------------------------------------

def q8_weight_from_numpy(qs, d, device="cuda") -> Q8Weight:
    """Upload numpy planes (int8 values, uint16 binary16 bits) as a packed weight."""
    import numpy as np

    qs_t = torch.from_numpy(np.ascontiguousarray(qs, dtype=np.int8)).to(device)
    d_t = torch.from_numpy(np.ascontiguousarray(d, dtype=np.uint16).view(np.float16)).to(device)
    return Q8Weight(qs_t, d_t)


def bf16_from_bits(bits, device="cuda") -> torch.Tensor:
    import numpy as np

    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).to(device).view(torch.bfloat16)
