"""The multi-GPU path is independent replicas (one batch per rank, no collective on
the data path).  Its host logic runs here as two gloo ranks on the CPU: each rank
draws a different batch, and the bench reduces the per-rank timings by max and the
per-rank bytes by sum."""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from mla_absorbed_decode_absorb_gb300 import workloads as W
        inp = W.generate(W.custom("replica", [100, 70], n_q=1), seed=rank)
        times, total = bench.reduce_over_ranks([1.0 + rank, 5.0 - rank], 1000 * (rank + 1))
        out[rank] = (times, total, float(inp.c_kv.float().sum()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_and_draw_distinct_batches():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        times, total, _ = res[r]
        assert times == [2.0, 5.0]      # max over ranks, element-wise
        assert total == 3000.0          # sum of bytes
    assert res[0][2] != res[1][2]       # seed = rank: different batches


def test_single_process_reduction_is_identity():
    import bench
    assert bench.reduce_over_ranks([1.5, 2.5], 7) == ([1.5, 2.5], 7.0)
