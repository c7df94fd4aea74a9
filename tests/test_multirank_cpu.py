"""The multi-GPU host logic of bench.py, as two gloo ranks on the CPU.

Frame pairs are independent, so an N-GPU run is N replicas (weak scaling):
no frame data crosses ranks, the step time is the maximum over ranks and
the job's throughput counts every rank's frames.  Only rank 0 prints."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 100.0 + 25.0 * rank       # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, world)
        value = bench.job_throughput(240, 10, world, ms / 1e3)
        assert bench.dist_env() == (rank, rank, world)
        buf = io.StringIO()

        class A:
            workload, steps, warmup = "c5_4k_10b", 1, 0
        os.environ["RANK"] = str(rank)
        if rank != 0:
            with redirect_stdout(buf):
                bench.run_reference(A)   # ranks other than 0 do nothing
        q.put((rank, ms, value, buf.getvalue()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    mp = pytest.importorskip("torch.multiprocessing")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, value, out in res:
        assert ms == 125.0                      # max over ranks
        assert value == pytest.approx(240 * 10 * 2 / 0.125)
        assert out == ""                        # only rank 0 prints


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(16, 4, 1, 2.0) == 32.0
