"""The multi-GPU form of the bench is independent replicas (the mixer has no exchange
step): each rank times its own copy of the workload, the job takes the slowest rank's time,
and the value counts every rank's tokens.  Checked here with two gloo ranks on the CPU."""
import io
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import bench
    ms = (3.0, 5.0)[rank]
    slow = bench.slowest_rank(ms)
    q.put((rank, slow, bench.replica_throughput(128 * 10, 2, slow)))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_time_the_slowest_rank_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    assert all(abs(r[2] - 1280 * 2 / 5e-3) < 1e-6 for r in res)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank(4.0) == 4.0
    assert bench.replica_throughput(128, 1, 2.0) == 64000.0


def test_reference_arm_prints_only_on_rank_zero(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), dict(steps=1, warmup=3, gpus=2))()
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args)
    assert buf.getvalue() == ""
