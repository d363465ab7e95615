"""The bench's N > 1 path on the CPU: two replica processes over a gloo
process group (127.0.0.1).  The layer shards by tokens with no exchange, so
the only cross-process steps are the timing barrier and the max-over-ranks
reduction of the step time; each rank draws its own tokens with the shared
weights."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    import workloads as W
    import torch.distributed as dist
    w, r, local = bench.setup_dist()
    try:
        assert (w, r) == (world, rank) and dist.get_backend() == "gloo"
        bench.barrier(w)
        # the slowest rank's time is the job's
        ms = bench.max_over_ranks(1.0 + rank, w, torch.device("cpu"))
        # own tokens per rank, the same weights everywhere
        x = W.rms_rows(16, 64, bench.rank_seed(rank))
        Wg = W.randn((64, 8), 64 ** -0.5, W._seed(W.BASE_SEED, "Wg"))
        xs = [torch.empty_like(x) for _ in range(w)]
        dist.all_gather(xs, x)
        wgs = [torch.empty_like(Wg) for _ in range(w)]
        dist.all_gather(wgs, Wg)
        out[rank] = (ms, bool(torch.equal(xs[0], xs[1])), bool(torch.equal(wgs[0], wgs[1])))
    finally:
        dist.destroy_process_group()


def test_two_replicas_over_gloo():
    if torch.cuda.is_available():
        pytest.skip("the gloo replica test runs on hosts without CUDA")
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in range(world):
        ms, same_x, same_w = res[rank]
        assert ms == 2.0          # max over ranks
        assert not same_x         # each replica routes its own tokens
        assert same_w             # through the same model
