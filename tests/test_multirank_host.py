"""Host logic of the multi-GPU benchmark, on two gloo ranks on the CPU: each rank
draws its own batch (rows shard by rank, no collective on the data path), and
the job's time is the slowest rank's, combined with a MAX all-reduce."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [10.0, 25.0][rank]
        total = bench.max_over_ranks(local_ms, dist, "cpu")
        c = dict(synth.WORKLOADS[synth.TINY])
        c["seed"] = bench.rank_seed(c["seed"], rank)
        p = synth.make_problem(**c)
        digest = torch.tensor([int(p.X[:4, :4].astype("int64").sum())], dtype=torch.int64)
        gathered = [torch.zeros_like(digest) for _ in range(world)]
        dist.all_gather(gathered, digest)
        out[rank] = (total, [int(g.item()) for g in gathered],
                     bench.job_tflops(world, bench.credited_flops(p.n, p.h, p.v), 5, total))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_batches():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    t0, digests0, v0 = out[0]
    t1, digests1, v1 = out[1]
    assert t0 == t1 == 25.0                      # the slowest rank decides
    assert digests0 == digests1 and digests0[0] != digests0[1]   # distinct batches per rank
    n, h, v = 256, 128, 1024
    assert abs(v0 - 2 * 6.0 * n * h * v * 5 / 0.025 / 1e12) < 1e-12
