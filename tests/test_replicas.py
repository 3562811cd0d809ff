"""The multi-GPU path is independent replicas: each rank times its own copy of the layer and the
job's throughput is all ranks' tokens over the slowest rank's time.  Checked on the CPU with two
gloo ranks (no GPU, no data-path collective)."""
import os
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.0, 3.5][rank]  # rank 1 is the slow replica
    got = bench.max_over_ranks(ms, dist)
    q.put((rank, got, bench.job_tokens_per_s(32, world, got)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_report_max_time_and_summed_tokens():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, tps in res:
        assert got == 3.5
        assert abs(tps - 64 / 3.5e-3) < 1e-6


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.25, None) == 1.25
    assert bench.job_tokens_per_s(4096, 1, 2.0) == 4096 / 2e-3
    assert torch.tensor(0).numel() == 1
