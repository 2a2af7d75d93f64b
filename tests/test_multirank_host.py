"""The N > 1 path of bench.py on CPU: two gloo ranks, one replica each (the
path shards by independent batches, with no collective on the data path).
Checks the slowest-rank timing every rank agrees on, the whole-job value, that
every rank draws its own synthetic batch, and that the reference arm does its
work on rank 0 only."""
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


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import pd_inputs
        mine = [0.25, 0.75][rank]
        slowest = bench.rank_max(mine, world, "cpu")
        value = bench.whole_job_value(1000, 4, slowest, world)
        c = pd_inputs.qwen3_8b_decode(seed=rank)           # what bench.py gives rank r
        digest = float(c.q.float().sum()) + float(c.pool.context_lens.sum())
        t = torch.tensor([digest], dtype=torch.float64)
        got = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(got, t)

        class A:
            warmup, steps = 0, 0
        ref = bench.run_reference(A, rank, world) if rank != 0 else "skipped"
        out.put((rank, slowest, value, [float(x) for x in got], ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value, digests, ref in res:
        assert slowest == 0.75                        # the slower replica's time
        assert value == pytest.approx(2 * 1000 * 4 / 0.75 / 1e9)
        assert digests[0] != digests[1]               # each rank its own batch
    assert res[1][4] is None                          # reference arm: rank 1 does nothing


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.rank_max(0.5, 1, "cpu") == 0.5
    assert bench.whole_job_value(2e9, 10, 2.0, 1) == pytest.approx(10.0)
