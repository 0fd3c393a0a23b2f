"""Shared helpers for the GPU parity tests (compare the CUDA path, called
through the C ABI, with the CPU oracle on the same seeded inputs)."""
import numpy as np


def same_float(a, b) -> bool:
    """Bit-for-bit equality of fp32 arrays, any NaN matching any NaN."""
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    if a.shape != b.shape:
        return False
    nan = np.isnan(a) & np.isnan(b)
    return bool(np.all(nan | (a.view(np.uint32) == b.view(np.uint32))))


def within_tol(y, Y, S, rel):
    """|y - Y| <= rel * S elementwise (Y, S from the fp64 oracle)."""
    y = np.asarray(y, np.float64)
    err = np.abs(y - Y)
    bound = rel * S
    ok = err <= bound
    if not np.all(ok):
        idx = np.argwhere(~ok)[:5]
        detail = [(tuple(i), float(y[tuple(i)]), float(Y[tuple(i)]), float(S[tuple(i)]))
                  for i in idx]
        return False, detail
    worst = float(np.max(err / np.where(S > 0, S, 1))) if err.size else 0.0
    return True, worst


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and widen back, via torch on the host."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()
