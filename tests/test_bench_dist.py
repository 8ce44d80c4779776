"""The multi-process (torchrun) path of bench.py on CPU: two gloo ranks.

Replicas do the same work each; the job's time is the slowest rank's, so the
whole-job value is world x work / max(time).  The reference arm runs on rank
0 only: any other rank returns without work or output."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    import bench
    dist, r, local, ws = bench._dist("gloo")
    # rank r took (10 + r) ms for the device-timed step and (20 + 2 r) ms end to end
    out = bench.replica_throughput(dist, ws, 1e12, 10.0 + r, 20.0 + 2 * r, torch.device("cpu"))
    if r == 1:
        class A:
            workload = "gqa16x2_L131072_d128_fwdbwd"
            steps = 1
            warmup = 0
            cpu_rows = 8
        ran = bench.run_reference(A())
        out = out + (ran,)
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, out))


def test_two_gloo_ranks_replica_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(world):
        value, e2e, ms, e2e_ms = res[r][:4]
        assert ms == 11.0 and e2e_ms == 22.0                 # max over ranks
        assert abs(value - 2 * 1e12 / 11e-3 / 1e12) < 1e-9   # world x work / slowest time
        assert abs(e2e - 2 * 1e12 / 22e-3 / 1e12) < 1e-9
    assert res[1][4] is None                                 # reference arm: rank 1 does nothing
