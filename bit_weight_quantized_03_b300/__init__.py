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

from ._lib import (BF16, BLOCK_BYTES, CHAIN_MAX_LINKS, CHAIN_MAX_STAGES, GemvStage,  # noqa: F401
                   BLOCK_ELEMS, ChainLink, ChainSrc, ERR_CUDA, ERR_ID_OUT_OF_RANGE,
                   ERR_INVALID_ARG, ERR_MISALIGNED, ERR_NONFINITE, ERR_TIMEOUT,
                   ERR_UNSUPPORTED_SHAPE, ERR_WORKSPACE, F32, FLAG_PDL, FLAG_TEST_STALL,
                   GEMV_MAX_M, GEMV_NOALLOC_SCRATCH_BYTES, OK, OP_ARGMAX, OP_RESIDUAL,
                   OP_SWIGLU, Q4Error, REPACK_TILE_BYTES, check, lib, status_string)

__all__ = [
    "q4_quantize", "q4_dequant_rows", "q4_gemv", "q4_gemv_prefetch", "q4_gemv_noalloc", "q4_gemv_chain", "q4_gemm", "q4_embed_gather", "q4_linear",
    "q4_gemv_workspace_bytes", "q4_gemm_workspace_bytes", "q4_linear_workspace_bytes",
    "q4_linear_crossover_m", "Workspace", "Q4Error", "lib", "packed_bytes",
    "q4_repack", "q4_repack_bytes", "q4_chain", "q4_chain_workspace_bytes", "q4_gemv_r",
    "q4_gemv_r_workspace_bytes", "Link", "LinkOut", "interleave_gate_rows", "q4_gemv_q8",
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
# q4_chain / q4_gemv_r carry state in their workspace from call to call (it is
# not left zero-filled), so they never share the default workspace of the
# calls that expect an all-zero one.
_default_chain_ws = {}


def _workspace(ws, nbytes: int, chain: bool = False):
    torch = _torch()
    if nbytes <= 0:
        return None, 0
    if ws is None:
        dev = torch.cuda.current_device()
        pool = _default_chain_ws if chain else _default_ws
        ws = pool.setdefault(dev, Workspace(dev))
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


def q4_gemv_prefetch(W, n: int, k: int, x, prefetch=None, y=None, workspace=None, status=None,
                     flags: int = 0, stream=None):
    """q4_gemv that prefetches the tensor `prefetch` (e.g. the next product's
    weights; contiguous, its byte size a multiple of 16) into L2 while it runs."""
    torch = _torch()
    m = x.shape[0]
    ldx = _row_stride(x, "x")
    if y is None:
        y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    ldy = _row_stride(y, "y")
    pbytes = 0 if prefetch is None else prefetch.numel() * prefetch.element_size()
    buf, nbytes = _workspace(workspace, q4_gemv_workspace_bytes(n, k, m))
    check(lib().q4_gemv_prefetch(_ptr(W), n, k, _ptr(x), m, ldx, _ptr(y), ldy, _ptr(buf), nbytes,
                                 _ptr(status), flags, _ptr(prefetch), pbytes, _stream(stream)),
          "q4_gemv_prefetch")
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


def q4_gemv_q8(W, n: int, k: int, x, y=None, stream=None):
    """y [n] = W x on the integer path: x [k] (or [1, k]) fp32 quantized per 32
    to int8 inside the kernel, exact integer block sums."""
    torch = _torch()
    if x.numel() != k or not x.is_contiguous():
        raise ValueError("x must be a contiguous vector of k elements")
    if y is None:
        y = torch.empty((n,), dtype=torch.float32, device=x.device)
    check(lib().q4_gemv_q8(_ptr(W), n, k, _ptr(x), _ptr(y), _stream(stream)), "q4_gemv_q8")
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


# ------------------------------------------------------------------ repacked layout, chains

def q4_repack_bytes(n: int, k: int) -> int:
    return int(lib().q4_repack_bytes(n, k))


def q4_repack(W, n: int, k: int, R=None, stream=None):
    """GGUF Q4_0 [n, k/32*18] -> the repacked tile layout (uint8, flat)."""
    torch = _torch()
    if R is None:
        R = torch.empty(q4_repack_bytes(n, k), dtype=torch.uint8, device=W.device)
    check(lib().q4_repack(_ptr(W), n, k, _ptr(R), _stream(stream)), "q4_repack")
    return R


class LinkOut:
    """A chain input taken from an earlier link's output, from element `offset`."""

    def __init__(self, link: int, offset: int = 0):
        self.link, self.offset = int(link), int(offset)


class Link:
    """One product of a q4_chain: y = W x (+ residual), W repacked (n x k).

    x, residual: a float32 device tensor (read from memory, `*_offset`
    elements in) or a LinkOut.  ops: OP_SWIGLU | OP_RESIDUAL | OP_ARGMAX
    (OP_SWIGLU: rows are 8 gate rows then 8 up rows per 16-row group, and the
    output is their n/2 gated values)."""

    def __init__(self, R, n, k, x, y=None, residual=None, argmax=None, ops=0, x_offset=0,
                 residual_offset=0):
        self.R, self.n, self.k, self.y, self.argmax, self.ops = R, n, k, y, argmax, ops
        self.x, self.residual = x, residual
        self.offsets = (x_offset, residual_offset)


def _src(v, offset):
    s = ChainSrc()
    if v is None:
        s.ptr, s.link, s.offset = None, -1, 0
    elif isinstance(v, LinkOut):
        s.ptr, s.link, s.offset = None, v.link, v.offset
    else:
        s.ptr, s.link, s.offset = _ptr(v), -1, int(offset)
    return s


def _link_array(links):
    arr = (ChainLink * len(links))()
    for i, l in enumerate(links):
        a = arr[i]
        a.R, a.n, a.k = _ptr(l.R), l.n, l.k
        a.x = _src(l.x, l.offsets[0])
        a.residual = _src(l.residual, l.offsets[1])
        a.y, a.argmax, a.ops = _ptr(l.y), _ptr(l.argmax), l.ops
    return arr


def q4_chain_workspace_bytes(links) -> int:
    return int(lib().q4_chain_workspace_bytes(_link_array(links), len(links)))


def q4_chain(links, workspace=None, status=None, flags: int = 0, stream=None):
    """Run the links in one launch (decode-step chain); see q4.h q4_chain."""
    arr = _link_array(links)
    need = int(lib().q4_chain_workspace_bytes(arr, len(links)))
    buf, nbytes = _workspace(workspace, need, chain=True)
    check(lib().q4_chain(arr, len(links), _ptr(buf), nbytes, _ptr(status), flags,
                         _stream(stream)), "q4_chain")


def q4_gemv_r_workspace_bytes(n: int, k: int) -> int:
    return int(lib().q4_gemv_r_workspace_bytes(n, k))


def q4_gemv_r(R, n: int, k: int, x, y=None, workspace=None, status=None, flags: int = 0,
              stream=None):
    """y = W x (batch 1, fp32) on a repacked matrix; x fp32 [k] (or [1, k])."""
    torch = _torch()
    if y is None:
        y = torch.empty((1, n), dtype=torch.float32, device=x.device)
    buf, nbytes = _workspace(workspace, q4_gemv_r_workspace_bytes(n, k), chain=True)
    check(lib().q4_gemv_r(_ptr(R), n, k, _ptr(x), _ptr(y), _ptr(buf), nbytes, _ptr(status),
                          flags, _stream(stream)), "q4_gemv_r")
    return y


def interleave_gate_rows(W1, W3):
    """Q4_0 rows of the FFN's w1 (gate) and w3 (up), [n, k/32*18] each with
    n % 8 == 0 -> one [2n, k/32*18] matrix of 16-row groups, 8 w1 rows then
    the same 8 rows of w3: the row order q4_chain's OP_SWIGLU takes."""
    torch = _torch()
    n, rb = W1.shape
    if W3.shape != W1.shape or n % 8:
        raise ValueError("w1 and w3 must have the same shape, with rows a multiple of 8")
    return torch.stack([W1.reshape(n // 8, 8, rb), W3.reshape(n // 8, 8, rb)], dim=1).reshape(2 * n, rb)
