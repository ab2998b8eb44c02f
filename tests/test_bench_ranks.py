"""The replica path of bench.py on two gloo ranks (CPU): every rank runs the
same workload on its own GPU with no data exchange, the slowest rank sets
the time, and the reported value is the whole job's throughput."""
import os
import socket
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    e = bench.max_over_ranks(times[rank], dist, "cpu")
    out[rank] = (e, bench.aggregate_tflops(world, 2.0e12, 3, e))
    dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_whole_job():
    times = [0.5, 0.8]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, _free_port(), times, out), nprocs=2, join=True)
        res = dict(out)
    for r in range(2):
        e, v = res[r]
        assert e == 0.8
        assert abs(v - 2 * 2.0e12 * 3 / 0.8 / 1e12) < 1e-9


def test_single_process_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25) == 0.25
    assert bench.aggregate_tflops(1, 1e12, 4, 0.5) == 8.0
    # replicas draw different inputs (seed = rank)
    w = bench.WORKLOADS["h16-s8192"]
    small = dict(w, H=1, S=64)
    a, b = bench.make_inputs(small, 0), bench.make_inputs(small, 1)
    assert not (a[0] == b[0]).all()
