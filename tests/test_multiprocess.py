"""CPU tests of the multi-rank bench logic with two gloo processes (no GPU): the job time is the
slowest rank's, throughput counts every rank's batch, and only rank 0 prints the reference line."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as tdist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 7.5 * rank                 # rank 1 is the slow replica
        got = bench.max_over_ranks(mine, "cpu")
        results[rank] = (got, bench.job_tokens_per_s(12288, world, got))
    finally:
        tdist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_worker, args=(world, port, results), nprocs=world, start_method="spawn")
        res = dict(results)
    assert res[0][0] == res[1][0] == 17.5           # every rank sees the slowest rank's time
    assert res[0][1] == pytest.approx(2 * 12288 / 0.0175)


def test_single_process_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_tokens_per_s(100, 1, 1000.0) == pytest.approx(100.0)


def test_launch_count_follows_chain_rows():
    """gpu_launches per step of the default path: the backward on the forward's workspace runs an E_c kernel
    while two 32-row chain CTAs per head fit the SMs (2 x heads <= SMs), and none with whole-head CTAs."""
    sys.path.insert(0, ROOT)
    import bench
    gen = bench.gen
    pth = bench.PATHS["operators"]
    assert bench.launches_per_step(pth, gen.WORKLOADS["debug_b12_t1024_h6"], 148) == 2 + 4      # 72 heads
    assert bench.launches_per_step(pth, gen.WORKLOADS["m100_b4_t512_h12"], 148) == 2 + 4        # 48 heads
    assert bench.launches_per_step(pth, gen.WORKLOADS["wide7b_b2_t4096_h64"], 148) == 2 + 3     # 128 heads
    assert bench.launches_per_step(bench.PATHS["operators-reform"], gen.WORKLOADS["wide7b_b2_t4096_h64"], 148) == 6


def test_reference_arm_only_rank0_prints():
    sys.path.insert(0, ROOT)
    import bench

    class A:  # the parsed arguments the reference arm reads
        workload = bench.WORKLOAD
        steps = 1
        warmup = 0

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, rank=1, world=2)
    assert buf.getvalue() == ""


def test_reference_arm_decode_workload_is_unavailable():
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload = "decode7b_b256_h2048"
        steps = 1
        warmup = 0

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, rank=0, world=1)
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and "unavailable" in line


def test_reference_arm_runs_the_oracle_over_a_process_pool():
    """The reference arm on the small oracle workload: one JSON line, value > 0, cores = pool size."""
    sys.path.insert(0, ROOT)
    import bench

    class A:
        workload = "oracle_b1_t128_h2"
        steps = 1
        warmup = 1

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, rank=0, world=1)
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["cores"] == min(os.cpu_count() or 1, 2)
    assert line["e2e"]["value"] == line["value"]


def test_cpu_baseline_reports_pool_and_single_thread():
    sys.path.insert(0, ROOT)
    import bench
    import wkv7_inputs as gen

    cb = bench.cpu_baseline(gen.WORKLOADS["oracle_b1_t128_h2"], 0.2)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert cb["single_thread"]["cores"] == 1 and cb["single_thread"]["value"] > 0


def test_reference_arm_config_is_the_workload_config():
    """Both arms print the same `config` object for the same workload."""
    sys.path.insert(0, ROOT)
    import bench
    import wkv7_inputs as gen

    class A:
        workload = "oracle_b1_t128_h2"
        steps = 1
        warmup = 0

    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(A, rank=0, world=1)
    line = json.loads(buf.getvalue())
    assert line["config"] == bench.workload_config(gen.WORKLOADS["oracle_b1_t128_h2"])


def test_bench_reads_no_markdown():
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert ".md" not in src
