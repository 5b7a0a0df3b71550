"""The benchmark's N>1 host logic on CPU: two gloo ranks on 127.0.0.1.

Each rank serves its own request (weak scaling, no data-path collective);
the only cross-rank step is the max of the per-rank timings."""
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


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    per_rank_ms = [12.5, 20.0][rank]
    mx = bench.max_over_ranks(per_rank_ms, dist)
    val = bench.weak_scaling_value(1e12, 10, world, mx)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, mx, val))


def test_two_gloo_ranks_max_and_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = [q.get(timeout=120) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, val in out:
        assert mx == 20.0                                  # slowest rank
        assert val == pytest.approx(2 * 1e12 * 10 / 20e-3 / 1e12)


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.weak_scaling_value(2e12, 5, 1, 10.0) == pytest.approx(1000.0)


def test_reference_arm_is_rank0_only(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")

    class A:
        steps, warmup, gpus, ref_budget = 1, 0, 2, 1.0
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
