"""The replica path of bench.py on CPU: two gloo ranks (no GPU)."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(ws),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    class Args:
        impl = "reference"      # the CPU arm: gloo, no device selection
    got_ws, got_rank, _ = bench.dist_setup(Args)
    ms = bench.max_over_ranks([1.0 + rank, 10.0 - rank], device="cpu")
    rate = bench.whole_job_rate(47, got_ws, ms[0])
    dist.barrier()
    dist.destroy_process_group()
    q.put((got_rank, got_ws, ms, rate))


def test_two_ranks_take_the_slowest_time_and_sum_the_work():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, ms, rate) in enumerate(out):
        assert (r, w) == (rank, 2)
        assert ms == [2.0, 10.0]                      # element-wise max over ranks
        assert rate == pytest.approx(2 * 47 / 2e-3)   # both ranks' units over the slowest time


def test_single_process_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5], device="cpu") == [3.0, 4.5]
    assert bench.whole_job_rate(8192, 1, 1.0) == pytest.approx(8192e3)
