"""Multi-rank host logic of bench.py on CPU: two gloo ranks over 127.0.0.1.

A multi-GPU run is weak scaling with independent replicas (every rank runs
the whole verify step on its own GPU, no data-path collective); the only
collective is the max over ranks of the measured time, tested here without
a GPU."""
import importlib.util
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        bench = _bench()
        local_ms = [12.5, 20.0, 7.25, 3.0][rank]
        got = bench.max_over_ranks(local_ms)
        value = bench.whole_job_gbs(world, 10, 1152 * 1000, got)
        with open(os.path.join(out_dir, "rank%d.txt" % rank), "w") as f:
            f.write("%r %r\n" % (got, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_max_over_ranks_gloo(tmp_path, world):
    port = _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    expect_ms = max([12.5, 20.0, 7.25, 3.0][:world])
    expect_gbs = world * 10 * 1152 * 1000 / (expect_ms * 1e-3) / 1e9
    for r in range(world):
        got, value = map(float, open(tmp_path / ("rank%d.txt" % r)).read().split())
        assert got == expect_ms
        assert value == pytest.approx(expect_gbs, rel=1e-12)


def test_single_process_is_identity():
    bench = _bench()
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_gbs(1, 4, 2304, 2.0) == pytest.approx(4 * 2304 / 2e-3 / 1e9)


def test_reference_arm_non_zero_rank_does_no_work(monkeypatch):
    bench = _bench()
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"config": 2, "warmup": 3, "steps": 2, "gpus": 2})()
    assert bench.run_reference(args) == 0
