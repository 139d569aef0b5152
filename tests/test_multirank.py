"""Multi-rank host logic of bench.py on CPU: two ranks over gloo.

With N GPUs each rank runs an independent request (weak scaling, no
data-path collective); the ranks meet only to take the maximum of each
timing, and rank 0 alone prints the JSON line.  The same holds for the
reference arm, which rank 0 alone runs.
"""
import contextlib
import io
import json
import os
import socket
from types import SimpleNamespace

import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist

    import bench
    from sparse_chunked_kv_gb300 import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        timings = [1.0 + rank, 10.0 - rank, 5.0 * (rank + 1)]   # dec, pre, step ms
        got = bench.max_over_ranks(timings, torch.device("cpu"))
        buf = io.StringIO()
        args = SimpleNamespace(steps=1, warmup=0, gpus=WORLD)
        with contextlib.redirect_stdout(buf):
            bench.run_reference(args, wl.TINY, rank)
        out.put((rank, got, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_max_and_rank0_alone_reports():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, out)) for r in range(WORLD)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(WORLD):
        rank, got, printed = out.get(timeout=240)
        results[rank] = (got, printed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(WORLD):
        assert results[rank][0] == [2.0, 10.0, 10.0]
    assert results[1][1] == ""
    lines = results[0][1].strip().splitlines()
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == WORLD


def test_job_throughput_counts_every_rank():
    import bench
    one = bench.job_tflops(1, 6.0e9, 64, 2.0)
    assert abs(one - 6.0e9 * 64 / 2.0e-3 / 1e12) < 1e-9
    assert abs(bench.job_tflops(2, 6.0e9, 64, 2.0) - 2 * one) < 1e-9

