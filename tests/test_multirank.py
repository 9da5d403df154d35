"""Multi-rank logic of the benchmark on CPU: two gloo ranks (the GPU path runs
one replica per GPU with no collective on the data path; only the timing is
reduced), max-over-ranks timing and the whole-job weak-scaling value."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]
    worst = bench.max_over_ranks(ms, dist)
    value = bench.weak_scaling_value(world, 8192, worst)
    q.put((rank, worst, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, value in got:
        assert worst == 5.0
        assert value == pytest.approx(2 * 8192 / 5e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(4.5, None) == 4.5
    assert bench.weak_scaling_value(1, 8192, 2.0) == pytest.approx(8192 / 2e-3)
