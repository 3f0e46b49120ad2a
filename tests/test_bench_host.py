"""bench.py's contract on the host (no GPU): the reference arm's JSON line, argument checks,
the launch count per step, and the replicas' max-over-ranks step time over a two-rank gloo
group."""
import dataclasses
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402

REQUIRED = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
            "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"]


def _run(*args, env=None):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, cwd=ROOT, env=env, timeout=600)


def test_reference_arm_prints_one_contract_line():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in REQUIRED:
        assert key in d, key
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1 and d["steps_timed"] == 1
    assert d["config"]["workload"].startswith("decode1")
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] == 1 and cpu["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_is_bounded_in_time(monkeypatch):
    """Whatever --steps is, the oracle work stops at REF_BUDGET_S."""
    calls = []

    def fake_sample(cfg, budget_s, max_tokens):
        calls.append((budget_s, max_tokens))
        return max(1, min(max_tokens, 3)), 0.5

    monkeypatch.setattr(bench, "oracle_sample", fake_sample)

    class A:
        config, steps, warmup, ncopy, nbatch = "decode1", 40000, 10, 8, 8

    assert bench.run_reference(A) == 0
    assert calls[-1] == (bench.REF_BUDGET_S, 40000) and bench.REF_BUDGET_S <= 180


def test_warmup_below_three_is_refused():
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "2")
    assert r.returncode != 0 and "warmup" in r.stderr


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "3", env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_config_is_the_gpu_arms_config():
    """Both arms word the workload with the same function and the same defaults."""
    r = _run("--impl", "reference", "--steps", "1", "--warmup", "3")
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["config"] == bench.config_dict(workloads.CONFIGS["decode1"], 8, 8)
    assert "seed 1" in d["config"]["workload"]


@pytest.mark.parametrize("name,flags,n", [("decode1", 0, 3), ("tiny", 0, 10), ("decode32", 0, 10),
                                          ("prefill2048", 0, 10), ("decode32", 1, 3),
                                          ("decode1", 2, 10), ("decode1", 8, 1)])
def test_kernels_per_step(name, flags, n):
    assert bench.kernels_per_step(workloads.CONFIGS[name], flags) == n


@pytest.mark.parametrize("T,n", [(1, 3), (2, 3), (3, 10), (64, 10)])
def test_kernels_per_step_follows_the_crossover(T, n):
    """The GEMV chain (three launches) up to T = 2, the grouped path from T = 3."""
    cfg = dataclasses.replace(workloads.CONFIGS["decode1"], T=T)
    assert bench.kernels_per_step(cfg, 0) == n


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, values, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank])
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    values = [1.25, 3.5]
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(2, _free_port(), values, out), nprocs=2, join=True)
    assert out[0] == out[1] == max(values)


def test_max_over_ranks_without_a_group_is_the_value():
    assert bench.max_over_ranks(2.5) == 2.5
