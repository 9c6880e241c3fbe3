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


def test_summary_keys_from_the_extras():
    """The compact summary the bench line ends with, built from extras of the
    shapes the GPU run produces: every key present, the AUTO table's cost 0
    when the sweep's best threshold is the compiled one, positive otherwise."""
    sys.path.insert(0, ROOT)
    import bench
    from driven_collective_communication_gb300 import build
    table = build.load_auto_table()
    sizes = [4096 << k for k in range(7)]

    def sweep(limit):  # one-shot faster up to `limit`, two-shot above
        return {"sizes": sizes, "one_shot_us": [1.0 if s <= limit else 2.0 for s in sizes],
                "two_shot_us": [1.5] * len(sizes), "one_shot_max_bytes": limit}
    other = {"c2_int32_inplace_one_shot": {"ms": 0.29, "hbm_gbs_2NS": 3700.0},
             "c2_int32_inplace_two_shot": {"ms": 0.16}, "c5_reduce_scatter": {"ms": 0.088},
             "c5_allgather": {"ms": 0.094}, "c5_ring_barrier": {"per_hop_us": 0.26},
             "linear_allreduce_bf16_n8_rows8192_kp1024": {"fused_us": 23.5, "fused_weight_gbs": 5700.0}}
    for t in (1, 16, 64, 128, 256):
        other["linear_tokens_bf16_n8_rows8192_kp1024_t%d" % t] = {"fused_tensor_us": 24.0 + t / 20,
                                                                   "gemm_then_allreduce_us": 37.0 + t / 10}
    matching = {"other": other, "crossover_n8": {t: sweep(table[8][t]) for t in table[8]}}
    s = bench.summary(None, matching)
    assert s["crossover_n8_matches_compiled_table"] is True
    assert all(v == 0 for v in s["crossover_n8_compiled_table_excess_pct"].values())
    assert set(s["linear_tokens_us"]) == {1, 16, 64, 128, 256} and s["fused_kp1024_us"] == 23.5
    other_limit = {t: (4096 if table[8][t] != 4096 else 262144) for t in table[8]}
    moved = {"other": other, "crossover_n8": {t: sweep(other_limit[t]) for t in table[8]}}
    s = bench.summary(None, moved)
    assert s["crossover_n8_matches_compiled_table"] is False
    assert all(v > 0 for v in s["crossover_n8_compiled_table_excess_pct"].values())
