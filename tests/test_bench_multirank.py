"""bench.py's multi-GPU host logic on the CPU: two gloo ranks (replicas) agree on the slowest rank's
time and report the whole-job throughput."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")   # rank 1 is the slow one
    v = bench.whole_job_tflops(world, 2e12, ms)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ms, v))


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, v in out:
        assert ms == 15.0
        assert v == pytest.approx(2 * 2e12 / 15e-3 / 1e12)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1, 1.5e12, 1.0) == pytest.approx(1500.0)


def _run_bench(args, env_extra):
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    env.update(env_extra)
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args, capture_output=True, text=True,
                       env=env, cwd=root, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_prints_one_contract_line():
    # the reference arm is the oracle on the host cores: one JSON line with the arm's own metric,
    # a cpu_baseline describing the run and an e2e object carrying the line's value
    (line,) = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "3", "--cpu-rows", "512"], {})
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["warmup"] >= 3 and line["steps"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert "workload" in line["config"]


def test_reference_arm_other_ranks_exit_quietly():
    # under torchrun only rank 0 runs and prints the reference line
    assert _run_bench(["--impl", "reference", "--steps", "1"], {"RANK": "1", "WORLD_SIZE": "2"}) == []
