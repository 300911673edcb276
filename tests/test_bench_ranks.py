"""The benchmark's multi-rank arithmetic on CPU with two gloo ranks.

With N GPUs every rank verifies its own batch (weak scaling, no data
exchange). The job is as slow as its slowest rank, so the timed region and
the end-to-end step are maxima over ranks, and the value counts every rank's
units. Two ranks report different timings here; both must agree on the
combined numbers.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as tdist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        region_ms = [800.0, 1000.0][rank]    # rank 1 is the slow one
        e2e_s = [0.002, 0.0015][rank]
        job = bench.combine_over_ranks(region_ms, e2e_s, steps=100, per_rank_units=224)
        results[rank] = job
    finally:
        tdist.destroy_process_group()


def test_two_ranks_take_the_slowest_and_count_all_units():
    world = 2
    with mp.Manager() as manager:
        results = manager.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
        jobs = dict(results)
    assert set(jobs) == {0, 1}
    for job in jobs.values():
        assert job["world"] == 2
        assert job["region_ms"] == 1000.0 and job["e2e_s"] == 0.002
        assert job["ms_per_step"] == pytest.approx(10.0)
        # 2 ranks x 100 steps x 224 positions in 1 s
        assert job["value"] == pytest.approx(2 * 100 * 224 / 1.0)
        assert job["e2e_value"] == pytest.approx(2 * 224 / 0.002)


def test_single_rank_without_a_process_group():
    import bench

    job = bench.combine_over_ranks(500.0, 0.001, steps=50, per_rank_units=224)
    assert job["world"] == 1 and job["value"] == pytest.approx(50 * 224 / 0.5)
