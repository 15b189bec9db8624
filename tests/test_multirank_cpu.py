"""Multi-rank host logic of the benchmark on CPU: two gloo ranks on 127.0.0.1.

FusedConv shards by batch with no exchange step, so N GPUs run N independent replicas:
the only cross-rank steps are the barrier, the max-over-ranks of the timed duration and
the whole-job throughput that rank 0 reports. These tests run exactly those steps with
the gloo backend in two processes (no GPU)."""
import importlib.util
import io
import os
import socket
import contextlib

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = load_bench()
        dist.barrier()
        slowest = bench.max_over_ranks(times[rank])
        out[rank] = (slowest, bench.job_tflops(1e12, world, 10, slowest))
    finally:
        dist.destroy_process_group()


def run_ranks(times):
    world = len(times)
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(rank_main, args=(world, free_port(), times, out), nprocs=world, join=True)
    return dict(out)


def test_every_rank_gets_the_slowest_time():
    res = run_ranks([3.0, 5.0])
    assert res[0][0] == 5.0 and res[1][0] == 5.0


def test_job_throughput_counts_all_replicas_over_the_slowest_time():
    res = run_ranks([2.0, 4.0])
    # 2 replicas x 10 steps x 1 TFLOP in 4 ms
    expected = 2 * 10 * 1e12 / 4e-3 / 1e12
    assert res[0][1] == pytest.approx(expected) and res[1][1] == pytest.approx(expected)


def test_single_rank_needs_no_process_group():
    bench = load_bench()
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_tflops(2e12, 1, 5, 10.0) == pytest.approx(1000.0)


def test_reference_arm_prints_only_on_rank_zero(monkeypatch):
    bench = load_bench()
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = type("A", (), {"steps": 1, "warmup": 0})()
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.run_reference(args) is None
    assert buf.getvalue() == ""
