"""The benchmark's multi-process path on CPU (gloo, world size 2): every rank runs
its own full problem (weak scaling, no data-path collective), ranks draw
distinct input streams, and the reported time is the maximum over ranks."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from mqa_attention_gb300.workloads import by_index

    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    t = bench.max_over_ranks(10.0 + rank, w)
    wl = by_index(1)
    mine = bench.host_inputs(wl, r)["q"]
    results[rank] = (t, int(mine[0, 0, 0, 0]), int(mine.sum()))
    import torch.distributed as dist

    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_gloo_replicas():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    assert res[0][0] == res[1][0] == 11.0          # max over ranks
    assert res[0][1:] != res[1][1:]                # each rank draws its own inputs


def test_single_process_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    import bench

    assert bench.dist_setup() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
