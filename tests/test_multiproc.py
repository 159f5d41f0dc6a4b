"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks check the
max-over-ranks job time and the whole-job throughput aggregation (replicas
of the step, no data-path collective)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    got_ws, got_rank, _ = bench._dist()
    my_ms = 2.0 + rank  # rank 1 is the slow replica
    mx = bench._sync_max(my_ms, got_ws)
    bench._barrier(got_ws)
    val = bench.job_tflops(1e12, mx, got_ws)
    out.put((got_rank, got_ws, mx, val))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ws, mx, val in res:
        assert ws == 2
        assert mx == 3.0  # max over ranks
        assert val == pytest.approx(2 * 1e12 / 3e-3 / 1e12)
