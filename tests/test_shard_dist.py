"""The row-sharded form of the products (bit_weight_quantized_03_b300.shard)
on two gloo ranks on CPU: the partition, the all-gather of a linear's output
and the sum all-reduce of a sharded embedding gather, each rank's local
product done by the oracle.  Splitting by rows leaves every output's
arithmetic unchanged, so the result must equal the single-rank oracle result
bit for bit (the gather's -0.0 rows included)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

import synth
from bit_weight_quantized_03_b300.shard import row_range, vocab_range


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("n", [1, 15, 16, 17, 100, 4096, 6144])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_row_range_partition(n, world):
    got = [row_range(n, r, world) for r in range(world)]
    assert got[0][0] == 0 and got[-1][1] == n
    for (a, b), (c, d) in zip(got, got[1:]):
        assert b == c and a <= b
    for a, b in got:
        assert a % 16 == 0 and (b % 16 == 0 or b == n)
    sizes = [(b - a + 15) // 16 for a, b in got]
    assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("vocab,world", [(1, 2), (37, 2), (37, 3), (131072, 8)])
def test_vocab_range_partition(vocab, world):
    got = [vocab_range(vocab, r, world) for r in range(world)]
    assert got[0][0] == 0 and got[-1][1] == vocab
    assert all(b == c for (_, b), (c, _) in zip(got, got[1:]))
    assert max(b - a for a, b in got) - min(b - a for a, b in got) <= 1


N, K, M, VOCAB, KE = 100, 256, 3, 37, 64


def _worker(rank, world, port, out):
    import torch
    import torch.distributed as dist
    import oracle
    from bit_weight_quantized_03_b300.shard import sharded_embed_gather, sharded_gemv
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # linear: every rank quantizes the same seeded matrix and keeps its rows
    W, rc, _ = oracle.quantize(synth.np_weights(N, K, seed=41))
    assert rc == 0
    x = torch.from_numpy(synth.np_activations(M, K, seed=42))
    r0, r1 = row_range(N, rank, world)

    def local_gemv(Wl, n, k, xx):
        Y, _ = oracle.matmul(Wl, n, k, xx.numpy())
        return torch.from_numpy(Y.astype(np.float32))

    y = sharded_gemv(W[r0:r1], N, K, x, rank, world, local=local_gemv)
    # gather: the table split by rows; ids inside, at both ends and outside
    T, rc, _ = oracle.quantize(synth.np_weights(VOCAB, KE, seed=43))
    assert rc == 0
    v0, v1 = vocab_range(VOCAB, rank, world)
    ids = torch.tensor([0, 36, 5, 18, 19, -1, 37, 5, 20, 1000], dtype=torch.int32)

    def local_gather(Tl, vocab, k, lid):
        o, _ = oracle.embed_gather(Tl, vocab, k, lid.numpy())
        return torch.from_numpy(o)

    g, bad = sharded_embed_gather(T[v0:v1], VOCAB, KE, ids, rank, world, local=local_gather)
    out[rank] = (y.numpy().tobytes(), g.numpy().tobytes(), bad)
    dist.destroy_process_group()


def test_sharded_gemv_and_gather_on_two_gloo_ranks():
    import oracle
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    W, _, _ = oracle.quantize(synth.np_weights(N, K, seed=41))
    Y, _ = oracle.matmul(W, N, K, synth.np_activations(M, K, seed=42))
    y_ref = Y.astype(np.float32)
    T, _, _ = oracle.quantize(synth.np_weights(VOCAB, KE, seed=43))
    g_ref, rc = oracle.embed_gather(T, VOCAB, KE, [0, 36, 5, 18, 19, -1, 37, 5, 20, 1000])
    assert rc == oracle.ERR_ID_OUT_OF_RANGE
    assert np.any(np.signbit(g_ref) & (g_ref == 0))  # the table has -0.0 entries
    for r in range(2):
        yb, gb, bad = out[r]
        assert yb == y_ref.tobytes()
        assert gb == g_ref.tobytes()
        assert bad
