"""The benchmark's multi-process path on CPU: two gloo ranks (one process per GPU on a multi-GPU machine)
run the same barrier / max-over-ranks / weak-scaling aggregation the benchmark uses."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench.dist_setup("gloo")
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    ms_local = 10.0 + 5.0 * rank            # rank 1 is the slow one
    ms = bench.max_over_ranks(ms_local, w, device="cpu")
    out[rank] = (ms, bench.job_throughput(100.0, w, ms))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 ranks x 100 units in the slowest rank's 15 ms
    assert res[0][1] == pytest.approx(2 * 100.0 / 0.015)


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_setup("gloo") == (1, 0, 0)
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_throughput(50.0, 1, 10.0) == pytest.approx(5000.0)
