"""The benchmark's multi-rank host logic on CPU (gloo, world size 2): one
replica of the workload per rank, no collective on the data path, the job's
time is the slowest rank's, and only rank 0 reports."""
import io
import os
import sys
import contextlib

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _rank_main(rank, world, port, values, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        out[rank] = bench.max_over_ranks(values[rank], dist, "cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_max_over_ranks_gloo_world2():
    import torch.multiprocessing as mp
    world = 2
    values = [3.25, 7.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), values, out), nprocs=world, join=True)
        got = dict(out)
    assert got == {0: 7.5, 1: 7.5}


def test_whole_job_value_counts_every_replica():
    import bench
    nbytes = bench.bytes_fp8_to_mx(bench.ROWS, bench.COLS) + bench.bytes_mx_to_fp8(bench.ROWS, bench.COLS)
    assert nbytes == 2 * 91750400                       # 1.5625 B per element, both kernels
    one = bench.whole_job_gbs(nbytes, 0.0305, 1)
    assert bench.whole_job_gbs(nbytes, 0.0305, 8) == pytest.approx(8 * one)
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5


def test_reference_arm_other_ranks_do_no_work():
    import bench

    class Args:
        steps, warmup, gpus = 3, 3, 2
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.run_reference(Args(), rank=1, world=2)
    assert buf.getvalue() == ""
