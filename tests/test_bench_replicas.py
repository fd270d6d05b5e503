"""bench.py's whole-job figure for N replicas (one process per GPU, launched by torchrun): every
rank's bytes over the slowest rank's time. Checked here with two gloo ranks on CPU, each
reporting a different time, which is the same collective path without a GPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, port: int, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import bench
    # rank 0 took 100 ms, rank 1 took 125 ms for the same 5e9 bytes and 4000 tokens each
    ms, gbs, toks = bench.aggregate_over_ranks([100.0, 125.0][rank], 5e9, 4000, 2, torch.device("cpu"))
    results[rank] = (ms, gbs, toks)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_replica_throughput_uses_slowest_rank_and_all_bytes():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(90)
        assert all(p.exitcode == 0 for p in procs)
        for r in range(2):
            ms, gbs, toks = results[r]
            assert ms == 125.0                       # max over ranks, on every rank
            assert gbs == pytest.approx(2 * 5e9 / 0.125 / 1e9)
            assert toks == pytest.approx(2 * 4000 / 0.125)


def test_single_rank_needs_no_collective():
    import bench
    ms, gbs, toks = bench.aggregate_over_ranks(50.0, 1e9, 100, 1, torch.device("cpu"))
    assert (ms, gbs, toks) == (50.0, pytest.approx(20.0), pytest.approx(2000.0))
