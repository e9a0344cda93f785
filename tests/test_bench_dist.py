"""The N>1 path of bench.py on CPU: two gloo ranks, weak scaling.

Every rank runs its own replica (the work shards by sequence and kv head with
no exchange), so the job rate is all ranks' work over the slowest rank's time.
"""
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist(enable=True, backend="gloo")
    d.barrier()
    rate, ms = bench.whole_job_rate(10.0, 100.0 * (rank + 1), d)
    q.put((rank, rate, ms, d.world))
    d.close()


def test_two_rank_weak_scaling_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, rate, ms, world in got:
        assert world == 2
        assert ms == 200.0  # the slowest rank's time
        assert abs(rate - 10.0 * 2 / 0.2) < 1e-9  # both ranks' work over it


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist(enable=True)
    assert d.world == int(os.environ.get("WORLD_SIZE", "1")) and d.pg is None
    rate, ms = bench.whole_job_rate(5.0, 50.0, d)
    assert ms == 50.0 and abs(rate - 100.0) < 1e-9
