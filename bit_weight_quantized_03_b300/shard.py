"""Row-sharded form of the Q4_0 products over the ranks of a process group.

The products of the quantized path (GeekNews, es.news.hada.io/topic?id=26595,
"Arquitectura": the decoder linears and the output head; "Soluciones
técnicas": the Q4 embedding rows) are independent per output row, so they
split over G ranks by rows with no reduction inside a product:

  * a linear y = W x: rank r holds rows [r0, r1) of W (whole 16-row groups,
    so that a repacked shard is whole tiles), computes its slice of y with
    the library's kernel on its own GPU, and one all-gather puts y together
    on every rank;
  * the embedding gather: rank r holds the table rows [v0, v1), fills the
    output rows whose id it holds and -0.0 elsewhere, and one sum all-reduce
    combines them; -0.0 is the additive identity of IEEE arithmetic
    (v + -0.0 == v for every v, +0 and -0 included), so the sum is the
    owner's value bit for bit.

Every rank computes with its own device's kernels; peers' memory is only
touched by the collective (NCCL across GPUs, gloo in the CPU tests).  The
local product is a parameter so that the partition and the collectives can be
tested on CPU ranks; its default is the library's CUDA entry point.
"""
from __future__ import annotations

from typing import Callable, Optional, Tuple


def row_range(n: int, rank: int, world: int) -> Tuple[int, int]:
    """Rows [r0, r1) of an n-row matrix held by `rank` of `world`: the 16-row
    groups split as evenly as whole groups allow (r1 == r0 when a rank gets
    none)."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("bad rank / world / n")
    groups = (n + 15) // 16
    g0, g1 = groups * rank // world, groups * (rank + 1) // world
    return min(n, 16 * g0), min(n, 16 * g1)


def vocab_range(vocab: int, rank: int, world: int) -> Tuple[int, int]:
    """Table rows [v0, v1) held by `rank` (contiguous, sizes differ by <= 1)."""
    if world < 1 or not 0 <= rank < world or vocab < 0:
        raise ValueError("bad rank / world / vocab")
    return vocab * rank // world, vocab * (rank + 1) // world


def _default_gemv(W, n, k, x):
    from . import q4_gemv
    return q4_gemv(W, n, k, x)


def _default_gather(table, vocab, k, ids):
    from . import q4_embed_gather
    return q4_embed_gather(table, vocab, k, ids)


def sharded_gemv(W_local, n: int, k: int, x, rank: int, world: int, group=None,
                 local: Optional[Callable] = None):
    """y = W x for a row-sharded W: W_local holds rows row_range(n, rank, world)
    as Q4_0 blocks; x [m, k] fp32 is replicated.  Returns y [m, n] on every
    rank (one all-gather of equal-sized padded slices)."""
    import torch
    import torch.distributed as dist
    local = local or _default_gemv
    r0, r1 = row_range(n, rank, world)
    m = x.shape[0]
    width = max(b - a for a, b in (row_range(n, r, world) for r in range(world)))
    part = torch.zeros((m, width), dtype=torch.float32, device=x.device)
    if r1 > r0:
        part[:, :r1 - r0] = local(W_local, r1 - r0, k, x)
    parts = [torch.empty_like(part) for _ in range(world)]
    dist.all_gather(parts, part, group=group)
    y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    for r in range(world):
        a, b = row_range(n, r, world)
        y[:, a:b] = parts[r][:, :b - a]
    return y


def sharded_embed_gather(table_local, vocab: int, k: int, ids, rank: int, world: int, group=None,
                         local: Optional[Callable] = None):
    """out[b] = dequant(row ids[b]) for a table sharded by rows: table_local
    holds rows vocab_range(vocab, rank, world).  Returns (out [B, k] fp32,
    out_of_range) on every rank; ids outside [0, vocab) give rows of +0.0."""
    import torch
    import torch.distributed as dist
    local = local or _default_gather
    v0, v1 = vocab_range(vocab, rank, world)
    ids = ids.to(torch.int64)
    mine = (ids >= v0) & (ids < v1)
    out = torch.full((ids.numel(), k), -0.0, dtype=torch.float32, device=ids.device)
    if bool(mine.any()) and v1 > v0:
        sel = torch.nonzero(mine).flatten()
        rows = local(table_local, v1 - v0, k, (ids[sel] - v0).to(torch.int32))
        out[sel] = rows
    dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    bad = (ids < 0) | (ids >= vocab)
    out[bad] = 0.0
    return out, bool(bad.any())
