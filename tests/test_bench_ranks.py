"""The benchmark's multi-process logic on CPU: one process per rank over
gloo (world size 2), as torchrun would launch it.  Each rank integrates its
own replica, so the only cross-rank steps are the barriers and the
maximum / sum of the timings and unit counts."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    r, local, w = bench.dist_setup()
    bench.barrier(w)
    mx = bench.max_over_ranks(10.0 + r, w)
    sm = bench.sum_over_ranks(100.0 * (r + 1), w)
    bench.barrier(w)
    out[rank] = (r, w, mx, sm)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_rank_timing_reduction():
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, start_method="spawn")
    assert out[0] == (0, 2, 11.0, 300.0)
    assert out[1] == (1, 2, 11.0, 300.0)


def _reference_rank(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import contextlib
    import io
    import sys
    import bench
    buf = io.StringIO()
    sys.argv = ["bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                "--warmup", "0"]
    with contextlib.redirect_stdout(buf):
        bench.main()
    out[rank] = buf.getvalue()


def test_reference_arm_prints_on_rank_zero_only(oracle_mod):
    import json
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_reference_rank, args=(2, _free_port(), out), nprocs=2,
                       start_method="spawn")
    assert out[1] == ""
    line = json.loads(out[0].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"
