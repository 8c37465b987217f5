"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks (no GPU).

bench.py runs one independent replica per rank (heads are independent; no
collective on the data path).  The only cross-rank steps are the barrier
around the timed region and the max over ranks of the step time; the whole
job's value is all ranks' FLOPs over that max.  These tests run those steps
in two spawned gloo processes.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        w, r, local = bench._dist()
        assert (w, r, local) == (ws, rank, rank)
        bench._barrier(w)
        ms_local = 1.0 + rank          # rank 1 is the slow one
        ms_max = bench._max_over_ranks(ms_local, w, torch.device("cpu"))
        value = bench.replica_value(w, 1e9, ms_max)
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            f.write("%r %r\n" % (ms_max, value))
        bench._barrier(w)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn", join=True)
    vals = [open(tmp_path / ("rank%d.txt" % r)).read().split() for r in range(2)]
    for ms_max, value in vals:
        assert float(ms_max) == 2.0                       # max over ranks, seen by both
        assert abs(float(value) - 2 * 1e9 / 2e-3 / 1e12) < 1e-12   # both ranks' FLOPs over the max time


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    bench._barrier(1)
    assert bench.replica_value(1, 2e12, 1000.0) == pytest.approx(2.0)
