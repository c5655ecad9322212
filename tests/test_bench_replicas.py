"""The multi-GPU path of bench.py is replicas only (batch-1 decode does not shard):
the timing aggregation over ranks is checked here with two gloo ranks on CPU."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [120.0, 150.0][rank]                 # rank 1 is the slower replica
    ms_max, tokens = bench.aggregate(ms, 1280, world, device="cpu")
    q.put((rank, ms_max, tokens))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replica_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out == [(0, 150.0, 2560), (1, 150.0, 2560)]


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(12.5, 128, 1) == (12.5, 128)
