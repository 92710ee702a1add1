"""The multi-process (replicas) path of bench.py on CPU: two gloo ranks on 127.0.0.1.
Each rank times its own token stream; the job reports the slowest rank's time and
the tokens of all ranks.  The reference arm runs on rank 0 only."""
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


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.slowest_rank_ms(10.0 + 5.0 * rank, world, "cpu")
    rate = bench.whole_job_rate(world, 5, 256, ms)
    ref = bench.run_reference(None) if rank != 0 else "rank0"
    dist.destroy_process_group()
    q.put((rank, ms, rate, ref))


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, ref in got:
        assert ms == 15.0                                   # the slowest rank's time
        assert rate == pytest.approx(2 * 5 * 256 / 0.015)   # both ranks' tokens
    assert got[1][3] is None                                # rank 1: no reference run


def test_single_process_path_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(12.5, 1, "cpu") == 12.5
    assert bench.whole_job_rate(1, 4, 256, 100.0) == pytest.approx(4 * 256 / 0.1)
