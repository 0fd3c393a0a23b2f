"""CPU oracle for the GGUF Q4_0 linear layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and
shares no code with it.  The arithmetic lives in ``q4_oracle.c`` (plain C99,
fp64 sums, no fast-math); this module builds it with gcc and marshals numpy
arrays through ctypes.

Method source: GeekNews on the Rust/Burn port of Voxtral Mini 4B Realtime
(es.news.hada.io/topic?id=26595), section "Arquitectura" (the quantized path
uses GGUF Q4_0 weights through custom GPU shaders) and section "Soluciones
técnicas" (the embedding table is held as Q4 rows and looked up per token).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q4_oracle.c")
_HDR = os.path.join(_HERE, "q4_oracle.h")
_LIB = os.path.join(_HERE, "libq4oracle.so")

BLOCK_ELEMS = 32
BLOCK_BYTES = 18
OK = 0
ERR_INVALID_ARG = 1
ERR_NONFINITE = 4
ERR_ID_OUT_OF_RANGE = 5

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle to ``oracle/libq4oracle.so`` (gcc, -O2, no FMA contraction)."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall", "-Wextra", "-pthread",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int32)
            i64 = ctypes.c_int64
            L.q4o_half_to_float.argtypes = [ctypes.c_uint16]
            L.q4o_half_to_float.restype = ctypes.c_float
            L.q4o_float_to_half_rne.argtypes = [ctypes.c_float]
            L.q4o_float_to_half_rne.restype = ctypes.c_uint16
            L.q4o_decode_block.argtypes = [u8p, f32p]
            L.q4o_decode_block.restype = None
            L.q4o_quantize_block.argtypes = [f32p, u8p]
            L.q4o_quantize_block.restype = ctypes.c_int
            L.q4o_quantize.argtypes = [f32p, i64, i64, u8p, ctypes.POINTER(i64)]
            L.q4o_quantize.restype = ctypes.c_int
            L.q4o_dequant_rows.argtypes = [u8p, i64, i64, f32p]
            L.q4o_dequant_rows.restype = ctypes.c_int
            L.q4o_matmul.argtypes = [u8p, i64, i64, f32p, i64, i64, f64p, f64p, i64, ctypes.c_int]
            L.q4o_matmul.restype = ctypes.c_int
            L.q4o_embed_gather.argtypes = [u8p, i64, i64, i32p, i64, f32p]
            L.q4o_embed_gather.restype = ctypes.c_int
            L.q4o_matmul_f64.argtypes = [u8p, i64, i64, f64p, i64, i64, f64p, f64p, i64,
                                         ctypes.c_int]
            L.q4o_matmul_f64.restype = ctypes.c_int
            L.q4o_swiglu.argtypes = [f64p, f64p, i64, f64p]
            L.q4o_swiglu.restype = None
            L.q4o_argmax.argtypes = [f64p, i64]
            L.q4o_argmax.restype = i64
            L.q4o_quantize_q8.argtypes = [f32p, i64, ctypes.POINTER(ctypes.c_int8), f32p]
            L.q4o_quantize_q8.restype = ctypes.c_int
            L.q4o_matmul_q8.argtypes = [u8p, i64, i64, f32p, i64, i64, f64p, f64p, i64]
            L.q4o_matmul_q8.restype = ctypes.c_int
            L.q4o_repack_bytes.argtypes = [i64, i64]
            L.q4o_repack_bytes.restype = i64
            L.q4o_repack.argtypes = [u8p, i64, i64, u8p]
            L.q4o_repack.restype = ctypes.c_int
            L.q4o_unrepack.argtypes = [u8p, i64, i64, u8p]
            L.q4o_unrepack.restype = ctypes.c_int
            _lib = L
    return _lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _blocks(W: np.ndarray, rows: int, k: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8)
    if W.size != rows * (k // BLOCK_ELEMS) * BLOCK_BYTES:
        raise ValueError(f"packed size {W.size} does not match {rows}x{k}")
    return W


def half_to_float(bits: int) -> float:
    return float(lib().q4o_half_to_float(int(bits) & 0xFFFF))


def float_to_half(x: float) -> int:
    return int(lib().q4o_float_to_half_rne(float(np.float32(x))))


def decode_block(blk) -> np.ndarray:
    b = np.ascontiguousarray(np.frombuffer(bytes(blk), dtype=np.uint8))
    assert b.size == BLOCK_BYTES
    out = np.empty(32, np.float32)
    lib().q4o_decode_block(_ptr(b, ctypes.c_uint8), _ptr(out, ctypes.c_float))
    return out


def quantize_block(x32) -> tuple[bytes, int]:
    x = np.ascontiguousarray(x32, dtype=np.float32)
    assert x.size == 32
    blk = np.empty(BLOCK_BYTES, np.uint8)
    rc = lib().q4o_quantize_block(_ptr(x, ctypes.c_float), _ptr(blk, ctypes.c_uint8))
    return blk.tobytes(), int(rc)


def quantize(w: np.ndarray) -> tuple[np.ndarray, int, int]:
    """fp32 [n, k] -> packed uint8 [n, k/32*18]; returns (blocks, status, n_bad)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    out = np.empty((n, k // BLOCK_ELEMS * BLOCK_BYTES), np.uint8)
    bad = ctypes.c_int64(0)
    rc = lib().q4o_quantize(_ptr(w, ctypes.c_float), n, k, _ptr(out, ctypes.c_uint8),
                            ctypes.byref(bad))
    if rc == ERR_INVALID_ARG:
        raise ValueError("q4o_quantize: invalid arguments")
    return out, int(rc), int(bad.value)


def dequant_rows(W: np.ndarray, rows: int, k: int) -> np.ndarray:
    W = _blocks(W, rows, k)
    out = np.empty((rows, k), np.float32)
    rc = lib().q4o_dequant_rows(_ptr(W, ctypes.c_uint8), rows, k, _ptr(out, ctypes.c_float))
    if rc != OK:
        raise ValueError("q4o_dequant_rows: invalid arguments")
    return out


def matmul(W: np.ndarray, n: int, k: int, X: np.ndarray, nthreads: int = 1):
    """fp64 Y[m, n] = X[m, :] . W^[n, :] and S[m, n] = sum |W^ X| (exact inputs)."""
    W = _blocks(W, n, k)
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float32)
    m = X.shape[0]
    if X.shape[1] != k:
        raise ValueError("X has the wrong width")
    Y = np.empty((m, n), np.float64)
    S = np.empty((m, n), np.float64)
    rc = lib().q4o_matmul(_ptr(W, ctypes.c_uint8), n, k, _ptr(X, ctypes.c_float), m, k,
                          _ptr(Y, ctypes.c_double), _ptr(S, ctypes.c_double), n, int(nthreads))
    if rc != OK:
        raise ValueError("q4o_matmul: invalid arguments")
    return Y, S


def quantize_q8(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """fp32 x [k] -> (int8 codes [k], fp32 block scales [k/32]) (Q4 x Q8 reading)."""
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    q = np.empty(x.size, np.int8)
    d = np.empty(x.size // BLOCK_ELEMS, np.float32)
    rc = lib().q4o_quantize_q8(_ptr(x, ctypes.c_float), x.size, _ptr(q, ctypes.c_int8),
                               _ptr(d, ctypes.c_float))
    if rc != OK:
        raise ValueError("q4o_quantize_q8: invalid arguments")
    return q, d


def matmul_q8(W: np.ndarray, n: int, k: int, X: np.ndarray):
    """Q4 x Q8 product: fp64 Y[m, n] and S[m, n] (each row of X quantized per 32)."""
    W = _blocks(W, n, k)
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float32)
    m = X.shape[0]
    if X.shape[1] != k:
        raise ValueError("X has the wrong width")
    Y = np.empty((m, n), np.float64)
    S = np.empty((m, n), np.float64)
    rc = lib().q4o_matmul_q8(_ptr(W, ctypes.c_uint8), n, k, _ptr(X, ctypes.c_float), m, k,
                             _ptr(Y, ctypes.c_double), _ptr(S, ctypes.c_double), n)
    if rc != OK:
        raise ValueError("q4o_matmul_q8: invalid arguments")
    return Y, S


def matmul_f64(W: np.ndarray, n: int, k: int, X: np.ndarray):
    """As matmul, with X taken in fp64 exactly as given."""
    W = _blocks(W, n, k)
    X = np.ascontiguousarray(np.atleast_2d(X), dtype=np.float64)
    m = X.shape[0]
    if X.shape[1] != k:
        raise ValueError("X has the wrong width")
    Y = np.empty((m, n), np.float64)
    S = np.empty((m, n), np.float64)
    rc = lib().q4o_matmul_f64(_ptr(W, ctypes.c_uint8), n, k, _ptr(X, ctypes.c_double), m, k,
                              _ptr(Y, ctypes.c_double), _ptr(S, ctypes.c_double), n, 1)
    if rc != OK:
        raise ValueError("q4o_matmul_f64: invalid arguments")
    return Y, S


def swiglu(a, b) -> np.ndarray:
    """fp64 SiLU-gated unit a * sigmoid(a) * b (the gated FFN activation reading)."""
    a = np.ascontiguousarray(a, dtype=np.float64).ravel()
    b = np.ascontiguousarray(b, dtype=np.float64).ravel()
    if a.size != b.size:
        raise ValueError("a and b differ in size")
    out = np.empty(a.size, np.float64)
    lib().q4o_swiglu(_ptr(a, ctypes.c_double), _ptr(b, ctypes.c_double), a.size,
                     _ptr(out, ctypes.c_double))
    return out


def argmax(y) -> int:
    y = np.ascontiguousarray(y, dtype=np.float64).ravel()
    return int(lib().q4o_argmax(_ptr(y, ctypes.c_double), y.size))


def repack_bytes(n: int, k: int) -> int:
    return int(lib().q4o_repack_bytes(n, k))


def repack(W: np.ndarray, n: int, k: int) -> np.ndarray:
    """GGUF Q4_0 rows -> the repacked 16 x 256 tile layout (uint8, flat)."""
    W = _blocks(W, n, k)
    R = np.empty(repack_bytes(n, k), np.uint8)
    if R.size == 0 or lib().q4o_repack(_ptr(W, ctypes.c_uint8), n, k,
                                       _ptr(R, ctypes.c_uint8)) != OK:
        raise ValueError("q4o_repack: invalid arguments")
    return R


def unrepack(R: np.ndarray, n: int, k: int) -> np.ndarray:
    R = np.ascontiguousarray(R, dtype=np.uint8).ravel()
    if R.size != repack_bytes(n, k):
        raise ValueError("repacked size does not match")
    W = np.empty((n, k // BLOCK_ELEMS * BLOCK_BYTES), np.uint8)
    if lib().q4o_unrepack(_ptr(R, ctypes.c_uint8), n, k, _ptr(W, ctypes.c_uint8)) != OK:
        raise ValueError("q4o_unrepack: invalid arguments")
    return W


def embed_gather(table: np.ndarray, vocab: int, k: int, ids) -> tuple[np.ndarray, int]:
    table = _blocks(table, vocab, k)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.empty((ids.size, k), np.float32)
    rc = lib().q4o_embed_gather(_ptr(table, ctypes.c_uint8), vocab, k,
                                _ptr(ids, ctypes.c_int32), ids.size, _ptr(out, ctypes.c_float))
    if rc == ERR_INVALID_ARG:
        raise ValueError("q4o_embed_gather: invalid arguments")
    return out, int(rc)


def cpu_count() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1
