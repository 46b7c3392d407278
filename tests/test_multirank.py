"""The multi-rank host path of the benchmark on CPU: two gloo ranks.

The sampler shards by rows with no exchange step, so the only cross-rank logic is
the timing contract: every rank takes rows of its own, the timed region is the
slowest rank's, and the reported rate counts the rows of all ranks.  The reference
arm runs on rank 0 only.
"""
import contextlib
import io
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        times = {0: 12.5, 1: 30.0}
        slow = bench.slowest(times[rank])
        value = bench.weak_value(world, 64, 100, slow)
        # The reference arm: rank 0 alone prints its line, the others leave without work.
        out = io.StringIO()
        with contextlib.redirect_stdout(out):
            if rank != 0:
                bench.run_reference(bench.parse_args_from(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
        dist.barrier()
        q.put((rank, slow, value, bench.rank_seed(rank), out.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_timing_contract():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    for _ in procs:
        rank, slow, value, seed, out = q.get(timeout=120)
        results[rank] = (slow, value, seed, out)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # Both ranks see the slowest rank's time, and the rate counts both ranks' rows.
    assert results[0][0] == results[1][0] == 30.0
    assert results[0][1] == results[1][1] == pytest.approx(2 * 64 * 100 / 0.030)
    # Every rank samples its own rows.
    assert results[0][2] != results[1][2]
    # The reference arm prints nothing on rank 1.
    assert results[1][3] == ""


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest(7.0) == 7.0
    assert bench.weak_value(1, 64, 10, 1.0) == pytest.approx(640000.0)
