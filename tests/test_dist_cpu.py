"""Multi-process host logic of the benchmark on CPU (gloo, world size 2).

The attention problems are independent per (b, h), so several GPUs run replicas with no
collective on the data path: each rank times its own replica, the job's time per step is the
slowest rank's, the whole-job rate counts the units of every rank, and the reference arm
(the oracle on the host cores) runs on rank 0 alone.  These are the pieces bench.py uses under
torchrun; here two gloo ranks exercise them without a GPU.
"""
import argparse
import contextlib
import io
import json
import os
import socket

import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_setup()
        ms = 10.0 + 5.0 * r                      # this rank's time per step
        slowest = bench.max_over_ranks(ms, w, "cpu")
        rate = bench.job_rate(w, 2.0e12, slowest)  # 2 TFLOP per rank per step
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            rc = bench.run_reference(argparse.Namespace(steps=1, warmup=0, ref_seconds=0.0))
        queue.put((r, w, slowest, rate, rc, out.getvalue()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_slowest_time_whole_job_rate_reference_on_rank0():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, queue)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        results = sorted(queue.get(timeout=600) for _ in range(world))
    finally:
        for p in procs:
            p.join(120)
    assert [p.exitcode for p in procs] == [0, 0]
    for r, w, slowest, rate, rc, _ in results:
        assert w == world and rc == 0
        assert slowest == 15.0                   # the slower rank's 15 ms, seen by both ranks
        assert abs(rate - 2 * 2.0 / 15e-3) < 1e-9  # both ranks' 4 TFLOP over 15 ms, in TFLOP/s
    line = json.loads(results[0][5].strip())
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 1
    assert results[1][5] == ""                   # rank 1 exits without work or output


def test_single_process_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert abs(bench.job_rate(1, 1e9, 1.0, 1e9) - 1000.0) < 1e-9
