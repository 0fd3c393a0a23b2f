"""CPU-only checks of the C ABI: libq4.so loads, exports every entry point that
include/q4.h declares, and rejects bad arguments on the host (nothing here
launches a kernel or needs a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q4.h")


@pytest.fixture(scope="module")
def q4():
    from bit_weight_quantized_03_b300 import build
    build.build()
    import bit_weight_quantized_03_b300 as q4mod
    return q4mod


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q4_[a-z0-9_]+)\s*\(", text)))


def header_constants():
    text = open(HEADER).read()
    consts = {m.group(1): int(m.group(2), 0) for m in
              re.finditer(r"#define\s+(Q4_\w+)\s+\(?([0-9xu]+?)u?\b", text)}
    enums = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(Q4_\w+)\s*=\s*(\d+)", text)}
    return consts, enums


def test_every_declared_symbol_is_exported(q4):
    names = declared_functions()
    assert len(names) >= 12, names
    L = q4.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    from bit_weight_quantized_03_b300._lib import SIGNATURES
    assert sorted(SIGNATURES) == names


def test_constants_match_header(q4):
    consts, enums = header_constants()
    assert enums["Q4_OK"] == q4.OK == 0
    assert enums["Q4_ERR_INVALID_ARG"] == q4.ERR_INVALID_ARG
    assert enums["Q4_ERR_MISALIGNED"] == q4.ERR_MISALIGNED
    assert enums["Q4_ERR_UNSUPPORTED_SHAPE"] == q4.ERR_UNSUPPORTED_SHAPE
    assert enums["Q4_ERR_NONFINITE"] == q4.ERR_NONFINITE
    assert enums["Q4_ERR_ID_OUT_OF_RANGE"] == q4.ERR_ID_OUT_OF_RANGE
    assert enums["Q4_ERR_TIMEOUT"] == q4.ERR_TIMEOUT
    assert enums["Q4_ERR_CUDA"] == q4.ERR_CUDA
    assert enums["Q4_ERR_WORKSPACE"] == q4.ERR_WORKSPACE
    assert enums["Q4_F32"] == q4.F32 and enums["Q4_BF16"] == q4.BF16
    assert consts["Q4_BLOCK_ELEMS"] == 32 and consts["Q4_BLOCK_BYTES"] == 18
    assert consts["Q4_GEMV_MAX_M"] == q4.GEMV_MAX_M
    assert consts["Q4_FLAG_PDL"] == q4.FLAG_PDL
    assert consts["Q4_OP_SWIGLU"] == q4.OP_SWIGLU and consts["Q4_OP_RESIDUAL"] == q4.OP_RESIDUAL
    assert consts["Q4_OP_ARGMAX"] == q4.OP_ARGMAX
    assert consts["Q4_CHAIN_MAX_LINKS"] == q4.CHAIN_MAX_LINKS


def test_status_strings(q4):
    L = q4.lib()
    for code in range(9):
        s = L.q4_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.q4_status_string(99).decode() == "unknown status"
    assert b"sm_103a" in L.q4_version()


# Fake, never-dereferenced device addresses: validation must reject the call
# before anything touches them.
A16 = 0x7F0000000000
A2 = A16 + 2


def test_host_validation_rejects_bad_arguments(q4):
    L = q4.lib()
    # null pointers / sizes
    assert L.q4_gemv(None, 8, 64, A16, 1, 64, A16, 8, None, 0, None, 0, None) == q4.ERR_INVALID_ARG
    assert L.q4_gemv(A16, 0, 64, A16, 1, 64, A16, 8, None, 0, None, 0, None) == q4.ERR_INVALID_ARG
    assert L.q4_gemv(A16, 8, 64, A16, 0, 64, A16, 8, None, 0, None, 0, None) == q4.ERR_INVALID_ARG
    # k not a multiple of 32
    assert L.q4_gemv(A16, 8, 48, A16, 1, 48, A16, 8, None, 0, None, 0, None) == q4.ERR_UNSUPPORTED_SHAPE
    # batch above the GEMV limit
    assert L.q4_gemv(A16, 8, 64, A16, 17, 64, A16, 8, None, 0, None, 0, None) == q4.ERR_UNSUPPORTED_SHAPE
    # leading dimensions
    assert L.q4_gemv(A16, 8, 64, A16, 1, 32, A16, 8, None, 0, None, 0, None) == q4.ERR_INVALID_ARG
    assert L.q4_gemv(A16, 8, 64, A16, 1, 64, A16, 7, None, 0, None, 0, None) == q4.ERR_INVALID_ARG
    # misalignment
    assert L.q4_gemv(A2, 8, 64, A16, 1, 64, A16, 8, None, 0, None, 0, None) == q4.ERR_MISALIGNED
    assert L.q4_gemv(A16, 8, 64, A2, 1, 64, A16, 8, None, 0, None, 0, None) == q4.ERR_MISALIGNED
    assert L.q4_gemv(A16, 8, 64, A16, 2, 66, A16, 8, None, 0, None, 0, None) == q4.ERR_MISALIGNED
    # quantize
    assert L.q4_quantize(None, 2, 64, A16, None, None) == q4.ERR_INVALID_ARG
    assert L.q4_quantize(A16, 2, 40, A16, None, None) == q4.ERR_UNSUPPORTED_SHAPE
    assert L.q4_quantize(A2, 2, 64, A16, None, None) == q4.ERR_MISALIGNED
    # dequant
    assert L.q4_dequant_rows(A16, 0, 4, 64, None, 0, None) == q4.ERR_INVALID_ARG
    assert L.q4_dequant_rows(A16, 0, 4, 64, A16, 7, None) == q4.ERR_INVALID_ARG
    assert L.q4_dequant_rows(A16, -1, 4, 64, A16, 0, None) == q4.ERR_INVALID_ARG
    assert L.q4_dequant_rows(A16, 0, 4, 64, A2, 0, None) == q4.ERR_MISALIGNED
    # gather
    assert L.q4_embed_gather(A16, 10, 64, None, 3, A16, None, None) == q4.ERR_INVALID_ARG
    assert L.q4_embed_gather(A16, 10, 64, A16, 0, A16, None, None) == q4.ERR_INVALID_ARG
    assert L.q4_embed_gather(A16, 10, 64, A16 + 1, 3, A16, None, None) == q4.ERR_MISALIGNED
    # gemm: k must be a multiple of 256, X rows 16-byte aligned
    assert L.q4_gemm(A16, 8, 288, A16, 4, 288, A16, 0, 8, None, 0, None, 0, None) == q4.ERR_UNSUPPORTED_SHAPE
    assert L.q4_gemm(A16, 8, 256, A16, 4, 260, A16, 0, 8, None, 0, None, 0, None) == q4.ERR_MISALIGNED
    assert L.q4_gemm(A16, 8, 256, A16, 4, 256, A16, 5, 8, None, 0, None, 0, None) == q4.ERR_INVALID_ARG
    # linear: bad dtype
    assert L.q4_linear(A16, 8, 256, A16, 3, 4, 256, A16, 8, None, 0, None, 0, None) == q4.ERR_INVALID_ARG
    # linear, fp32 X beyond the GEMV batch with k % 256 != 0: the tensor-core
    # path cannot take k, and the call is refused before the bf16 conversion
    # (the fake addresses are never dereferenced; no CUDA call is made)
    assert L.q4_linear(A16, 8, 3104, A16, 0, 17, 3104, A16, 8, A16, 1 << 30, None, 0,
                       None) == q4.ERR_UNSUPPORTED_SHAPE
    # noalloc: every q4_gemv rule is applied before anything touches the device
    assert L.q4_gemv_noalloc(A16, 8, 64, A16, 1, 32, A16, 8, None, 0, None) == q4.ERR_INVALID_ARG
    assert L.q4_gemv_noalloc(A16, 8, 64, A2, 1, 64, A16, 8, None, 0, None) == q4.ERR_MISALIGNED
    assert L.q4_gemv_noalloc(A16, 8, 64, A16, 2, 66, A16, 8, None, 0, None) == q4.ERR_MISALIGNED


def _bad_link(q4, **kw):
    from bit_weight_quantized_03_b300._lib import ChainLink
    arr = (ChainLink * 2)()
    for a in arr:
        a.R, a.n, a.k = A16, 64, 256
        a.x.ptr, a.x.link, a.x.offset = A16, -1, 0
        a.residual.link = -1
        a.y, a.ops = A16, 0
    for key, v in kw.items():
        obj, field = (arr[1], key) if "." not in key else (getattr(arr[1], key.split(".")[0]),
                                                           key.split(".")[1])
        setattr(obj, field, v)
    return arr


def test_gemv_prefetch_host_validation(q4):
    """The prefetch region of q4_gemv_prefetch is checked before anything is
    launched: NULL with a size, a pointer off 16 bytes or a size off a multiple
    of 16 is refused; the other arguments are q4_gemv's."""
    L = q4.lib()
    W, X, Y, P = (i << 20 for i in (1, 2, 3, 4))  # 16-byte aligned fake device addresses
    args = (W, 8, 256, X, 1, 256, Y, 8, None, 0, None, 0)
    assert L.q4_gemv_prefetch(*args, None, 16, None) == q4.ERR_INVALID_ARG
    assert L.q4_gemv_prefetch(*args, P + 8, 16, None) == q4.ERR_MISALIGNED
    assert L.q4_gemv_prefetch(*args, P, 24, None) == q4.ERR_MISALIGNED
    # a good region gets as far as q4_gemv's own checks (no workspace here)
    assert L.q4_gemv_prefetch(*args, P, 32, None) == q4.ERR_WORKSPACE
    assert L.q4_gemv_prefetch(W, 8, 48, X, 1, 48, Y, 8, None, 0, None, 0, P, 16,
                              None) == q4.ERR_UNSUPPORTED_SHAPE


def test_gemv_q8_host_validation(q4):
    L = q4.lib()
    A16 = 1 << 20  # a 16-byte-aligned fake address: nothing is launched on these paths
    assert L.q4_gemv_q8(None, 4, 64, A16, A16, None) == q4.ERR_INVALID_ARG
    assert L.q4_gemv_q8(A16, 0, 64, A16, A16, None) == q4.ERR_INVALID_ARG
    assert L.q4_gemv_q8(A16, 4, 48, A16, A16, None) == q4.ERR_UNSUPPORTED_SHAPE
    assert L.q4_gemv_q8(A16, 4, 12288 + 32, A16, A16, None) == q4.ERR_UNSUPPORTED_SHAPE
    assert L.q4_gemv_q8(A16 + 2, 4, 64, A16, A16, None) == q4.ERR_MISALIGNED
    assert L.q4_gemv_q8(A16, 4, 64, A16 + 2, A16, None) == q4.ERR_MISALIGNED


def test_repacked_and_chain_host_validation(q4):
    L = q4.lib()
    assert L.q4_repack_bytes(4, 288) == 0
    assert L.q4_repack_bytes(17, 256) == 2 * 2304
    assert L.q4_repack_bytes(16, 512) == 2 * 2304
    assert L.q4_repack(None, 4, 256, A16, None) == q4.ERR_INVALID_ARG
    assert L.q4_repack(A16, 4, 288, A16, None) == q4.ERR_UNSUPPORTED_SHAPE
    assert L.q4_repack(A2, 4, 256, A16, None) == q4.ERR_MISALIGNED
    assert L.q4_gemv_r_workspace_bytes(4096, 3072) > 0
    assert L.q4_gemv_r_workspace_bytes(4096, 3000) == 0
    good = _bad_link(q4)
    assert L.q4_chain_workspace_bytes(good, 2) > 0
    cases = [
        (dict(k=288), q4.ERR_UNSUPPORTED_SHAPE),            # k % 256
        (dict(k=12544), q4.ERR_UNSUPPORTED_SHAPE),          # k above the kernel's limit
        (dict(R=A2), q4.ERR_MISALIGNED),
        (dict(R=None), q4.ERR_INVALID_ARG),
        (dict(n=0), q4.ERR_INVALID_ARG),
        (dict(ops=8), q4.ERR_INVALID_ARG),                   # unknown op
        (dict(ops=q4.OP_ARGMAX), q4.ERR_INVALID_ARG),        # argmax without an output
        (dict(**{"x.link": 1}), q4.ERR_INVALID_ARG),         # not an earlier link
        (dict(**{"x.link": 0, "x.offset": 2}), q4.ERR_MISALIGNED),   # offset % 4
        (dict(**{"x.link": 0, "x.offset": 16}), q4.ERR_INVALID_ARG),  # past the source's n
        (dict(**{"x.ptr": A16 + 4}), q4.ERR_MISALIGNED),
        (dict(**{"x.offset": 2}), q4.ERR_MISALIGNED),
        (dict(ops=q4.OP_SWIGLU, n=72), q4.ERR_INVALID_ARG),  # gate rows: n % 16
        (dict(ops=q4.OP_SWIGLU | q4.OP_RESIDUAL, **{"residual.ptr": A16}),
         q4.ERR_INVALID_ARG),                                # the gate stands alone
        (dict(ops=q4.OP_RESIDUAL, n=62, **{"residual.ptr": A16}), q4.ERR_UNSUPPORTED_SHAPE),
    ]
    for kw, want in cases:
        arr = _bad_link(q4, **kw)
        assert L.q4_chain(arr, 2, A16, 1 << 30, None, 0, None) == want, kw
        assert L.q4_chain_workspace_bytes(arr, 2) == 0, kw
    assert L.q4_chain(good, 0, A16, 1 << 30, None, 0, None) == q4.ERR_INVALID_ARG
    assert L.q4_chain(good, 129, A16, 1 << 30, None, 0, None) == q4.ERR_INVALID_ARG
    assert L.q4_chain(good, 2, None, 0, None, 0, None) == q4.ERR_WORKSPACE
    assert L.q4_chain(good, 2, A16, 16, None, 0, None) == q4.ERR_WORKSPACE
    assert L.q4_chain(good, 2, A16 + 16, 1 << 30, None, 0, None) == q4.ERR_MISALIGNED


def test_workspace_sizes_are_consistent(q4):
    L = q4.lib()
    assert L.q4_gemv_workspace_bytes(8, 48, 1) == 0          # invalid k
    assert L.q4_gemv_workspace_bytes(8, 64, 17) == 0         # m above the limit
    assert L.q4_gemv_workspace_bytes(4096, 288, 1) == 0      # generic kernel: no split-K
    w1 = L.q4_gemv_workspace_bytes(4096, 3072, 1)
    w8 = L.q4_gemv_workspace_bytes(4096, 3072, 8)
    assert 0 < w1 < w8
    assert L.q4_linear_crossover_m(4096, 3072) >= 1
    assert L.q4_linear_crossover_m(4096, 288) == q4.GEMV_MAX_M


def _gemm_split_ws(n, m, splits, bn_tiles):
    """Workspace of a q4_gemm that splits K: the per-tile arrival counters
    (rounded up to 256 bytes), then splits x m x n fp32 partials."""
    return (bn_tiles * 4 + 255) // 256 * 256 + splits * m * n * 4


@pytest.mark.parametrize("n,k,m,expect", [
    # K = 1280 at M = 375 (64-token tiles): a 2-way split would remove only 10
    # k-steps per CTA, less than its fixed cost -> whole tiles, no workspace
    (1280, 1280, 375, 0),
    (3840, 1280, 375, 0),
    # K = 5120 at M = 375: the 2-way split removes 40 k-steps -> split
    (1280, 5120, 375, _gemm_split_ws(1280, 375, 2, 10 * 6)),
    # small M (32-token tiles): the splits that pay stay
    (4096, 3072, 8, _gemm_split_ws(4096, 8, 4, 32)),
    (1280, 1280, 8, _gemm_split_ws(1280, 8, 5, 10)),
    (9216, 3072, 8, _gemm_split_ws(9216, 8, 2, 72)),
    # large M: one wave or more of whole tiles
    (3840, 1280, 3000, 0),
    (1280, 5120, 3000, 0),
])
def test_gemm_split_k_plan(q4, n, k, m, expect):
    """The GEMM planner splits K only when that removes more than 24 * BN / 64
    of a CTA's 64-wide k-steps (148 SMs assumed without a GPU); the workspace
    query shows the decision."""
    assert q4.lib().q4_gemm_workspace_bytes(n, k, m) == expect


# q4_linear's measured table: the largest M sent to the fp32 GEMV per shape
CROSSOVER_TABLE = {(4096, 3072): 4, (1024, 3072): 6, (3072, 4096): 4, (9216, 3072): 4,
                   (3072, 9216): 4, (3840, 1280): 8, (1280, 1280): 6, (5120, 1280): 8,
                   (1280, 5120): 6}


def test_linear_crossover_table_and_nearest_shape(q4):
    """Each measured shape returns its entry; another shape takes the entry
    whose weight count is nearest on a log scale; k % 256 != 0 has no
    tensor-core path and returns the GEMV's limit."""
    L = q4.lib()
    for (n, k), m in CROSSOVER_TABLE.items():
        assert L.q4_linear_crossover_m(n, k) == m, (n, k)
    import math

    def nearest(n, k):
        return min(CROSSOVER_TABLE.items(),
                   key=lambda e: abs(math.log(n * k / (e[0][0] * e[0][1]))))[1]
    for n, k in [(4096, 2048), (2048, 1280), (100, 256), (131072, 3072), (7000, 5120)]:
        assert L.q4_linear_crossover_m(n, k) == nearest(n, k), (n, k)
    assert L.q4_linear_crossover_m(4096, 3104) == q4.GEMV_MAX_M
    assert L.q4_linear_crossover_m(0, 3072) == q4.GEMV_MAX_M


def test_gemv_workspace_covers_every_launch_of_a_batched_call(q4):
    """A q4_gemv call with m >= 2 rows (k % 256 == 0) runs launches of up to 4
    rows of the batched tile kernel (8 warps per SM) and, for a single leftover
    row, the batch-1 kernel (up to 16 warps per SM).  Each warp of a launch may
    publish one 64-bit word per row of x and output row of its 32-row group, so
    the workspace must hold the per-group counters (rounded to 256 B) plus
    warps x rows x 32 x 8 bytes for the largest launch.  Without a GPU the
    library assumes 148 SMs."""
    L = q4.lib()
    sms = 148
    for n, k in [(4096, 3072), (3072, 9216), (1000, 256), (131072, 3072), (33, 512)]:
        groups = (n + 31) // 32
        units = groups * (k // 256)
        cnt = (groups * 4 + 255) // 256 * 256
        for m in range(2, 17):
            need = cnt + max(min(units, sms * 8) * min(m, 4) * 32 * 8,
                             min(units, sms * 16) * 32 * 8 if m % 4 == 1 else 0)
            got = L.q4_gemv_workspace_bytes(n, k, m)
            assert got >= need, (n, k, m, got, need)


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import bit_weight_quantized_03_b300._lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        L.lib()
