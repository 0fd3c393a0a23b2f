"""ctypes loader for libq4.so (the C ABI declared in include/q4.h).

Fails loudly: there is no fallback of any kind when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libq4.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_MISALIGNED = 2
ERR_UNSUPPORTED_SHAPE = 3
ERR_NONFINITE = 4
ERR_ID_OUT_OF_RANGE = 5
ERR_TIMEOUT = 6
ERR_CUDA = 7
ERR_WORKSPACE = 8
F32 = 0
BF16 = 1
FLAG_PDL = 1
FLAG_TEST_STALL = 1 << 30
GEMV_MAX_M = 16
GEMV_NOALLOC_SCRATCH_BYTES = 4 << 20
BLOCK_ELEMS = 32
BLOCK_BYTES = 18

class GemvStage(ctypes.Structure):
    """struct q4_gemv_stage of include/q4.h."""
    _fields_ = [("W", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


CHAIN_MAX_STAGES = 128
CHAIN_MAX_LINKS = 128
OP_SWIGLU = 1
OP_RESIDUAL = 2
OP_ARGMAX = 4
REPACK_TILE_BYTES = 2304


class ChainSrc(ctypes.Structure):
    """struct q4_chain_src of include/q4.h."""
    _fields_ = [("ptr", ctypes.c_void_p), ("link", ctypes.c_int32), ("offset", ctypes.c_int32)]


class ChainLink(ctypes.Structure):
    """struct q4_chain_link of include/q4.h."""
    _fields_ = [("R", ctypes.c_void_p), ("n", ctypes.c_int64), ("k", ctypes.c_int64),
                ("x", ChainSrc), ("residual", ChainSrc),
                ("y", ctypes.c_void_p), ("argmax", ctypes.c_void_p), ("ops", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32)]


# Every symbol include/q4.h declares, with its ctypes signature.
_vp, _i64, _sz, _u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint32
_st = ctypes.c_int
SIGNATURES = {
    "q4_quantize": (_st, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "q4_dequant_rows": (_st, [_vp, _i64, _i64, _i64, _vp, ctypes.c_int, _vp]),
    "q4_gemv": (_st, [_vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _sz, _vp, _u32, _vp]),
    "q4_gemv_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "q4_gemv_prefetch": (_st, [_vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _sz, _vp, _u32,
                               _vp, _sz, _vp]),
    "q4_gemv_noalloc": (_st, [_vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _u32, _vp]),
    "q4_gemv_q8": (_st, [_vp, _i64, _i64, _vp, _vp, _vp]),
    "q4_gemv_chain": (_st, [ctypes.POINTER(GemvStage), ctypes.c_int32, _vp, _sz, _vp, _u32, _vp]),
    "q4_gemv_chain_workspace_bytes": (_sz, [ctypes.POINTER(GemvStage), ctypes.c_int32]),
    "q4_gemm": (_st, [_vp, _i64, _i64, _vp, _i64, _i64, _vp, ctypes.c_int, _i64, _vp, _sz, _vp,
                      _u32, _vp]),
    "q4_gemm_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "q4_embed_gather": (_st, [_vp, _i64, _i64, _vp, _i64, _vp, _vp, _vp]),
    "q4_linear": (_st, [_vp, _i64, _i64, _vp, ctypes.c_int, _i64, _i64, _vp, _i64, _vp, _sz, _vp,
                        _u32, _vp]),
    "q4_linear_workspace_bytes": (_sz, [_i64, _i64, _i64, ctypes.c_int]),
    "q4_linear_crossover_m": (_i64, [_i64, _i64]),
    "q4_repack_bytes": (_sz, [_i64, _i64]),
    "q4_repack": (_st, [_vp, _i64, _i64, _vp, _vp]),
    "q4_chain_workspace_bytes": (_sz, [ctypes.POINTER(ChainLink), ctypes.c_int32]),
    "q4_chain": (_st, [ctypes.POINTER(ChainLink), ctypes.c_int32, _vp, _sz, _vp, _u32, _vp]),
    "q4_gemv_r_workspace_bytes": (_sz, [_i64, _i64]),
    "q4_gemv_r": (_st, [_vp, _i64, _i64, _vp, _vp, _vp, _sz, _vp, _u32, _vp]),
    "q4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "q4_version": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


class Q4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(self.status)} (status {self.status})")


def lib() -> ctypes.CDLL:
    """The loaded libq4.so.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m bit_weight_quantized_03_b300.build` (needs nvcc)")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(st: int) -> str:
    try:
        return lib().q4_status_string(int(st)).decode()
    except ImportError:
        return "unknown"


def check(st: int, where: str) -> None:
    if st != OK:
        raise Q4Error(st, where)
