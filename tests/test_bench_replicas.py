"""The multi-GPU bench path on CPU: replicas on 2 gloo ranks.

The decode does not shard across GPUs here (replicas only); what the N > 1 path
adds is the slowest-rank timing and the whole-job throughput.  Two gloo ranks
with different local times must agree on the maximum and report
world_size x steps x pixels / max time.
"""
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=2)
    local_seconds = 2.0 if rank == 0 else 3.0
    slowest = bench.max_over_ranks(local_seconds)
    value = bench.replica_throughput(dist.get_world_size(), 5, 1048576, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, value))


def test_two_gloo_replicas_agree_on_slowest_rank():
    pytest.importorskip("torch")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, slowest, value in res:
        assert slowest == 3.0
        assert value == pytest.approx(2 * 5 * 1048576 / 3.0 / 1e6)


def test_single_process_is_its_own_maximum():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.replica_throughput(1, 10, 1000, 2.0) == pytest.approx(10 * 1000 / 2.0 / 1e6)
