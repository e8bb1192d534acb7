"""Host logic of the N > 1 path on the CPU: two gloo ranks.

The layer partitions by tokens (replicated weights, no exchange): each rank
runs its own slice of tokens and the slices together are bitwise the one-rank
result.  The timing helpers bench.py uses under torchrun (process-group set-up,
barrier, max over ranks) are exercised with the same two ranks."""
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(rng, T=12, d=64, E=16, F=32):
    from oracle import Expert, Matrix
    bf = lambda a: torch.as_tensor(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    x = bf(rng.standard_normal((T, d)))
    wr = bf(rng.standard_normal((E, d)) / np.sqrt(d))
    ex = [Expert(Matrix(bf(rng.standard_normal((F, d)) * 0.1)), Matrix(bf(rng.standard_normal((F, d)) * 0.1)),
                 Matrix(bf(rng.standard_normal((d, F)) * 0.1))) for _ in range(E)]
    return x, wr, ex


def _rank_main(rank, world, port, result_q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    import oracle

    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    assert bench.max_over_ranks(w, float(rank + 1)) == float(world)

    x, wr, ex = _layer(np.random.default_rng(0))
    T = x.shape[0]
    mine = np.arange(rank, T, world)           # this rank's tokens
    res = oracle.layer_forward(x[mine], wr, None, lambda e: ex[e], [], 8)
    parts = [None] * world
    dist.all_gather_object(parts, (mine, res.out, res.ids))
    if rank == 0:
        full = oracle.layer_forward(x, wr, None, lambda e: ex[e], [], 8)
        out = np.empty_like(full.out)
        ids = np.empty_like(full.ids)
        for idx, o, i in parts:
            out[idx] = o
            ids[idx] = i
        result_q.put(bool(np.array_equal(out, full.out) and np.array_equal(ids, full.ids)))
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_tokens_bitwise():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    assert q.get(timeout=5) is True
