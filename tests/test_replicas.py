"""The bench's replica path (one process per GPU, no data-path collective) on CPU: two gloo ranks
exercise the max-over-ranks job time, the whole-job throughput and the rank-0-only reference
arm.  The collective is the timing's, never the layer's."""
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


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        job = bench.max_over_ranks(times[rank], world, device="cpu")
        value = bench.job_tokens_per_s(4, 100, world, job[0])
        out.put((rank, job, value))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_every_rank_tokens():
    world, port = 2, _free_port()
    times = [[10.0, 30.0], [12.5, 25.0]]      # per rank: device-timed ms, end-to-end ms
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job, value in res:
        assert job == [12.5, 30.0]                        # each value's max over the ranks
        assert value == pytest.approx(4 * 100 * 2 / 12.5e-3)   # both ranks' tokens over the slowest time


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
    assert bench.job_tokens_per_s(4, 10, 1, 2.0) == pytest.approx(4 * 10 / 2e-3)


def test_reference_arm_does_no_work_on_other_ranks(monkeypatch):
    """Under torchrun the reference arm runs on rank 0 alone; other ranks return at once."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    called = []
    monkeypatch.setattr(bench, "OracleRunner", lambda w: called.append(w))
    assert bench.run_reference(None, None) is None
    assert not called
