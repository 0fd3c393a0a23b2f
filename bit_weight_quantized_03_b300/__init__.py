"""GGUF Q4_0 weight-only-quantized linear layer for NVIDIA B300 (sm_103a).

Python binding of the C ABI in include/q4.h.  Each function below has the
name of the C entry point it calls and does argument marshalling only: torch
tensors supply device pointers, shapes and strides, and the current torch
stream; every step of the computation runs in the library's CUDA kernels.
There is no CPU or PyTorch fallback: the library must be built
(`python -m bit_weight_quantized_03_b300.build`), or the calls raise.

Method: the quantized path of the Rust/Burn port of Voxtral Mini 4B Realtime
(GeekNews, es.news.hada.io/topic?id=26595, "Arquitectura": GGUF Q4_0 weights
through custom GPU shaders; "Soluciones técnicas": Q4 embedding rows looked up
per token).
"""
from __future__ import annotations

from ._lib import (BF16, BLOCK_BYTES, CHAIN_MAX_STAGES, GemvStage, BLOCK_ELEMS, ERR_CUDA, ERR_ID_OUT_OF_RANGE,  # noqa: F401
                   ERR_INVALID_ARG, ERR_MISALIGNED, ERR_NONFINITE, ERR_TIMEOUT,
                   ERR_UNSUPPORTED_SHAPE, ERR_WORKSPACE, F32, FLAG_PDL, FLAG_TEST_STALL,
                   GEMV_MAX_M, GEMV_NOALLOC_SCRATCH_BYTES, OK, Q4Error, check, lib,
                   status_string)

__all__ = [
    "q4_quantize", "q4_dequant_rows", "q4_gemv", "q4_gemv_noalloc", "q4_gemv_chain", "q4_gemm", "q4_embed_gather", "q4_linear",
    "q4_gemv_workspace_bytes", "q4_gemm_workspace_bytes", "q4_linear_workspace_bytes",
    "q4_linear_crossover_m", "Workspace", "Q4Error", "lib", "packed_bytes",
]


def packed_bytes(n: int, k: int) -> int:
    return n * (k // BLOCK_ELEMS) * BLOCK_BYTES


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _row_stride(t, what: str) -> int:
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{what} must be a 2-D tensor with unit column stride")
    return t.stride(0)


class Workspace:
    """A zero-filled device buffer that grows on demand (split-K scratch).

    Sequential calls on one stream may share it: every call that ends without a
    device error leaves it zero-filled again.  Concurrent streams need one each."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        torch = _torch()
        if nbytes <= 0:
            return None
        if self.buf is None or self.buf.numel() < nbytes:
            dev = self.device if self.device is not None else torch.cuda.current_device()
            self.buf = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=dev)
        return self.buf

    def reset(self):
        if self.buf is not None:
            self.buf.zero_()


_default_ws = {}


def _workspace(ws, nbytes: int):
    torch = _torch()
    if nbytes <= 0:
        return None, 0
    if ws is None:
        dev = torch.cuda.current_device()
        ws = _default_ws.setdefault(dev, Workspace(dev))
    if isinstance(ws, Workspace):
        buf = ws.get(nbytes)
    else:
        buf = ws
    return buf, buf.numel() * buf.element_size()


def q4_gemv_workspace_bytes(n: int, k: int, m: int) -> int:
    return int(lib().q4_gemv_workspace_bytes(n, k, m))


def q4_gemm_workspace_bytes(n: int, k: int, m: int) -> int:
    return int(lib().q4_gemm_workspace_bytes(n, k, m))


def q4_linear_workspace_bytes(n: int, k: int, m: int, x_dtype: int = F32) -> int:
    return int(lib().q4_linear_workspace_bytes(n, k, m, x_dtype))


def q4_linear_crossover_m(n: int, k: int) -> int:
    return int(lib().q4_linear_crossover_m(n, k))


def q4_quantize(w, blocks=None, status=None, stream=None):
    """fp32 [n, k] (contiguous) -> Q4_0 blocks, uint8 [n, k/32*18]."""
    torch = _torch()
    n, k = w.shape
    if blocks is None:
        blocks = torch.empty((n, k // BLOCK_ELEMS * BLOCK_BYTES), dtype=torch.uint8,
                             device=w.device)
    check(lib().q4_quantize(_ptr(w), n, k, _ptr(blocks), _ptr(status), _stream(stream)),
          "q4_quantize")
    return blocks


def q4_dequant_rows(blocks, row0: int, n_rows: int, k: int, out=None, out_dtype=None,
                    stream=None):
    torch = _torch()
    out_dtype = torch.float32 if out_dtype is None else out_dtype
    if out is None:
        out = torch.empty((n_rows, k), dtype=out_dtype, device=blocks.device)
    code = BF16 if out.dtype == torch.bfloat16 else F32
    check(lib().q4_dequant_rows(_ptr(blocks), row0, n_rows, k, _ptr(out), code, _stream(stream)),
          "q4_dequant_rows")
    return out


def q4_gemv(W, n: int, k: int, x, y=None, workspace=None, status=None, flags: int = 0,
            stream=None):
    """y[i, r] = sum_j w^[r, j] x[i, j]; x fp32 [m, >=k], y fp32 [m, >=n]."""
    torch = _torch()
    m = x.shape[0]
    ldx = _row_stride(x, "x")
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    ldy = _row_stride(y, "y")
    buf, nbytes = _workspace(workspace, q4_gemv_workspace_bytes(n, k, m))
    check(lib().q4_gemv(_ptr(W), n, k, _ptr(x), m, ldx, _ptr(y), ldy, _ptr(buf), nbytes,
                        _ptr(status), flags, _stream(stream)), "q4_gemv")
    return y


def q4_gemv_noalloc(W, n: int, k: int, x, y=None, status=None, flags: int = 0, stream=None):
    """q4_gemv for callers that cannot allocate device memory: no workspace
    argument; the split-K scratch is a fixed array inside the library (the
    output y is allocated here only when the caller passes none).  Calls that
    may overlap on the GPU share that array and race: keep them on one stream."""
    torch = _torch()
    m = x.shape[0]
    ldx = _row_stride(x, "x")
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    ldy = _row_stride(y, "y")
    check(lib().q4_gemv_noalloc(_ptr(W), n, k, _ptr(x), m, ldx, _ptr(y), ldy, _ptr(status),
                                flags, _stream(stream)), "q4_gemv_noalloc")
    return y


def _chain_array(stages):
    arr = (GemvStage * len(stages))()
    for i, (W, n, k, x, y) in enumerate(stages):
        arr[i].W, arr[i].n, arr[i].k = _ptr(W), n, k
        arr[i].x, arr[i].y = _ptr(x), _ptr(y)
    return arr


def q4_gemv_chain_workspace_bytes(stages) -> int:
    return int(lib().q4_gemv_chain_workspace_bytes(_chain_array(stages), len(stages)))


def q4_gemv_chain(stages, workspace=None, status=None, flags: int = 0, stream=None):
    """Run links (W, n, k, x, y) in order, y = W x each (batch 1, fp32), in one
    launch; x may be a slice of an earlier link's y (torch views)."""
    arr = _chain_array(stages)
    buf, nbytes = _workspace(workspace, int(lib().q4_gemv_chain_workspace_bytes(arr, len(stages))))
    check(lib().q4_gemv_chain(arr, len(stages), _ptr(buf), nbytes, _ptr(status), flags,
                              _stream(stream)), "q4_gemv_chain")


def q4_gemm(W, n: int, k: int, X, Y=None, y_dtype=None, workspace=None, status=None,
            flags: int = 0, stream=None):
    """Y[i, r] = sum_j bf16(w^[r, j]) X[i, j]; X bf16 [m, >=k], Y fp32/bf16 [m, >=n]."""
    torch = _torch()
    m = X.shape[0]
    ldx = _row_stride(X, "X")
    if Y is None:
        Y = torch.empty((m, n), dtype=torch.float32 if y_dtype is None else y_dtype,
                        device=X.device)
    ldy = _row_stride(Y, "Y")
    code = BF16 if Y.dtype == torch.bfloat16 else F32
    buf, nbytes = _workspace(workspace, q4_gemm_workspace_bytes(n, k, m))
    check(lib().q4_gemm(_ptr(W), n, k, _ptr(X), m, ldx, _ptr(Y), code, ldy, _ptr(buf), nbytes,
                        _ptr(status), flags, _stream(stream)), "q4_gemm")
    return Y


def q4_embed_gather(table, vocab: int, k: int, ids, out=None, status=None, stream=None):
    torch = _torch()
    if out is None:
        out = torch.empty((ids.numel(), k), dtype=torch.float32, device=ids.device)
    check(lib().q4_embed_gather(_ptr(table), vocab, k, _ptr(ids), ids.numel(), _ptr(out),
                                _ptr(status), _stream(stream)), "q4_embed_gather")
    return out


def q4_linear(W, n: int, k: int, X, Y=None, workspace=None, status=None, flags: int = 0,
              stream=None):
    torch = _torch()
    m = X.shape[0]
    ldx = _row_stride(X, "X")
    code = BF16 if X.dtype == torch.bfloat16 else F32
    if Y is None:
        Y = torch.empty((m, n), dtype=torch.float32, device=X.device)
    ldy = _row_stride(Y, "Y")
    buf, nbytes = _workspace(workspace, q4_linear_workspace_bytes(n, k, m, code))
    check(lib().q4_linear(_ptr(W), n, k, _ptr(X), code, m, ldx, _ptr(Y), ldy, _ptr(buf), nbytes,
                          _ptr(status), flags, _stream(stream)), "q4_linear")
    return Y
