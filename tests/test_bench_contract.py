"""The benchmark's reference arm (the oracle timed on the host cores) on CPU:
one JSON line with the contract's keys, on one process and under two gloo
ranks (rank 0 prints, the other exits 0 without work)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


def _run(cmd, env=None):
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def _check(line, n):
    assert KEYS <= set(line), KEYS - set(line)
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["n_gpus"] == n and line["steps"] == 3 and line["warmup"] == 3
    assert line["config"]["workload"] == "allreduce_bf16_n8_256MiB"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    assert isinstance(cb.get("cpu_model"), str) and cb["cpu_model"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_single_process():
    lines = _run([sys.executable, "bench.py", "--impl", "reference", "--steps", "3", "--warmup", "3",
                  "--ref-elems", "65536"])
    assert len(lines) == 1
    _check(lines[0], 1)


def test_reference_arm_two_ranks_rank0_only():
    pytest.importorskip("torch.distributed")
    env = dict(os.environ, MASTER_ADDR="127.0.0.1")
    lines = _run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                  "--master-addr", "127.0.0.1", "--master-port", "29631", "bench.py", "--impl", "reference",
                  "--gpus", "2", "--steps", "3", "--warmup", "3", "--ref-elems", "65536"], env=env)
    assert len(lines) == 1
    _check(lines[0], 2)


def test_timing_helpers_on_the_host():
    """The pure helpers of the bench: min / mean beside the median, and the CPU model."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.spread([3.0, 1.0, 2.0]) == {"min_ms": 1.0, "mean_ms": 2.0}
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_crossover_rule_minimises_summed_time():
    """The AUTO threshold the bench derives from a sweep: the cut that minimises
    the summed time, robust to one noisy point."""
    sys.path.insert(0, ROOT)
    import bench
    sizes = [4, 8, 16, 32, 64]
    assert bench.crossover_rule(sizes, [1, 1, 1, 1, 1], [2, 2, 2, 2, 2]) == 64   # one-shot always faster
    assert bench.crossover_rule(sizes, [2, 2, 2, 2, 2], [1, 1, 1, 1, 1]) == 0    # never
    assert bench.crossover_rule(sizes, [1, 1.1, 1, 2, 3], [1.5, 1.0, 1.5, 1.5, 1.5]) == 16  # one noisy loss at 8
    assert bench.crossover_rule(sizes, [1, 1, 1, 1, 1], [1, 1, 1, 1, 1]) == 0    # ties: the smaller threshold
