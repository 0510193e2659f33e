"""The multi-GPU form of the benchmark is N independent replicas: the job time
is the slowest rank's, the value sums the replicas' payload.  Exercised with
two gloo ranks on the CPU (no GPU, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    mine = 10.0 + 5.0 * rank  # rank 1 is the slower replica
    t = bench.max_over_ranks(mine, ws, "cpu")
    ms_step, value = bench.replica_throughput(t, steps=5, T=1 << 30, ws=ws)
    q.put((rank, t, ms_step, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_time():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, ms_step, value in got:
        assert t == 15.0
        assert ms_step == pytest.approx(3.0)
        assert value == pytest.approx(2 * 2 * (1 << 30) / 3.0e-3 / 1e9)


def test_single_replica_is_identity():
    import bench
    assert bench.max_over_ranks(7.5, 1, "cpu") == 7.5
    ms, v = bench.replica_throughput(20.0, 10, 1 << 30, 1)
    assert ms == 2.0 and v == pytest.approx(2 * (1 << 30) / 2e-3 / 1e9)
