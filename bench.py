"""Benchmark of the virtual-rank AllReduce on one GB300 (replicas on N GPUs).

A step is one sum AllReduce over N=8 virtual ranks of 134,217,728 bf16
elements (256 MiB) per rank, N(0,1)*(1+r) values, fp32 accumulation -- the
large-message workload -- through the C ABI with inputs resident in HBM.
Printed metric: algbw = per-rank bytes / step time (GB/s), plus the HBM
roofline fraction of the kernel (algorithmic traffic 2*N*S per launch).
Extra keys carry the decode-size sweep (16 KiB..4 MiB per rank, p50 us), the
ReduceScatter / AllGather and ring-barrier figures, the end-to-end number
through the host-buffer entry point, the oracle's CPU baseline and the SM
clocks sampled during the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun (N > 1) every rank runs an independent replica on its own GPU
("replicas only": the virtual-rank path has no exchange between GPUs); the
headline and the end-to-end number are timed on all replicas together, the
single-GPU extras (sweeps, other workloads, the CPU leg) run at N = 1 only.
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

# the PortChannel measurement waits on the proxy's stream: one hardware queue
# per stream (set before the CUDA context exists)
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from driven_collective_communication_gb300 import workloads as W  # noqa: E402
from driven_collective_communication_gb300.replicas import Dist  # noqa: E402

GB = 1e9
FALLBACK_HBM_GBS = 6800.0
# large messages (each launch >= tens of microseconds): warm-ups and timed launches per point
LARGE_WARMUP, LARGE_STEPS = 20, 50
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "allreduce_twoshot_bf16_n8.txt")
# what the timed kernel is made of: the roofline's measured traffic is reported
# only while these device sources hash to the value in the profile and the live
# launch shape (CTAs per rank x threads) equals the profiled one.  reduce_ops.cuh
# is left out on purpose: it holds only the MAX / MIN combiners, which the
# timed sum instance does not instantiate
KERNEL_SOURCES = ["collectives.cuh", "memory_channel.cuh", "instantiate.cuh", "coll_bf16.cu",
                  "dcc_internal.h"]


# ------------------------------------------------------------------ helpers
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "driven_collective_communication_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(blocks, threads):
    """DRAM bytes per launch of the timed kernel from the committed ncu summary,
    or None if the kernel or its launch shape changed since the counters were taken."""
    try:
        text = open(PROFILE_TRAFFIC).read()
    except OSError:
        return None
    m = re.search(r"^traffic_bytes_per_full_launch:\s*(\d+)", text, re.M)
    h = re.search(r"^kernel_source_hash:\s*(\w+)", text, re.M)
    sh = re.search(r"^launch_shape:\s*(\d+)\s*x\s*(\d+)", text, re.M)
    if not m or not h or not sh or h.group(1) != kernel_source_hash():
        return None
    if (int(sh.group(1)), int(sh.group(2))) != (blocks, threads):
        return None
    return int(m.group(1))


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="dcc_clocks_%d_" % self.gpu, suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        power = [float(r[3]) for r in rows if re.match(r"^[\d.]+$", r[3])]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(power) if power else None}


def spread(per):
    """min and mean of per-launch times (ms) beside the median a result reports as "ms"."""
    return {"min_ms": round(min(per), 4), "mean_ms": round(statistics.fmean(per), 4)}


def time_launches(fn, steps, stream):
    """Per-launch CUDA-event durations (ms) on `stream` and the whole span."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    t1.record(stream)
    t1.synchronize()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return per, t0.elapsed_time(t1)


def time_launches_queued(fn, steps, stream, batch=100, hold_cycles=5_000_000):
    """Per-launch CUDA-event durations (ms) with the host kept out of them: a
    bounded spin kernel (torch's sleep kernel, hold_cycles SM cycles, about
    2.4 ms at 2.07 GHz) holds the stream while the host queues a batch of
    (event, launch, event), so the launches then run back to back and each
    pair of events brackets one launch as the device runs it.  Also returns
    whether every batch was fully queued before its hold ended."""
    per, queued_ok = [], True
    for b0 in range(0, steps, batch):
        nb = min(batch, steps - b0)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(nb)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(nb)]
        h0 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            h0.record(stream)
            torch.cuda._sleep(hold_cycles)
            t = time.perf_counter()
            for i in range(nb):
                starts[i].record(stream)
                fn()
                ends[i].record(stream)
            host_ms = (time.perf_counter() - t) * 1e3
        ends[-1].synchronize()
        queued_ok &= host_ms < h0.elapsed_time(starts[0])
        per += [s_.elapsed_time(e) for s_, e in zip(starts, ends)]
    return per, queued_ok


def time_queued_span(fn, launches, stream, hold_cycles=5_000_000, rounds=5):
    """Device time per launch (us) of `launches` eager launches queued back to
    back behind the same hold as time_launches_queued, with one pair of events
    around the whole run instead of a pair per launch (an event between two
    launches makes the second wait for the first to drain).  Median over
    `rounds` runs."""
    out = []
    for _ in range(rounds):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(hold_cycles)
            e0.record(stream)
            for _ in range(launches):
                fn()
            e1.record(stream)
        e1.synchronize()
        out.append(e0.elapsed_time(e1) * 1e3 / launches)
    return statistics.median(out)


def eager_floor(stream):
    """The same per-launch measures for an empty kernel (torch's sleep kernel
    with a zero count): what an eager launch costs the device by itself."""
    empty = lambda: torch.cuda._sleep(0)  # noqa: E731
    with torch.cuda.stream(stream):
        for _ in range(50):
            empty()
        per, queued_ok = time_launches_queued(empty, 1000, stream)
    return {"event_bracketed_p50_us": round(statistics.median(per) * 1e3, 2),
            "event_bracketed_min_us": round(min(per) * 1e3, 2), "queued_ahead": bool(queued_ok),
            "back_to_back_us": round(time_queued_span(empty, 100, stream), 2)}


# ------------------------------------------------------------------ oracle CPU leg
def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform)."""
    import platform
    import subprocess
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


def oracle_sample_run(seconds, elems, threads=None):
    """Time the oracle (all host cores, or `threads`) on a prefix of `elems` elements
    per rank of the large-message workload.  Returns (GB/s algbw, threads, sample text,
    seconds per call)."""
    import oracle
    w = W.C4
    xs = [W.to_storage(t) for t in W.rank_inputs(w, device="cpu", count=elems)]
    threads = threads or os.cpu_count() or 1
    oracle.allreduce(xs, "bf16", nthreads=threads)  # warm
    n_calls, t_total = 0, 0.0
    while t_total < seconds:
        t = time.perf_counter()
        oracle.allreduce(xs, "bf16", nthreads=threads)
        t_total += time.perf_counter() - t
        n_calls += 1
    per_call = t_total / n_calls
    sample = ("oracle AllReduce, N=8 bf16, first %d elements (%d MiB) of each rank's 256 MiB "
              "buffer, %d calls, %.1f s" % (elems, elems * 2 >> 20, n_calls, t_total))
    return elems * 2 / per_call / GB, threads, sample, per_call


# ------------------------------------------------------------------ our arm
def run_ours(args, dist):
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc

    torch.cuda.set_device(dist.local)
    dev = torch.device("cuda", dist.local)
    stream = torch.cuda.Stream(device=dev)
    w = W.C4
    n = w.n_ranks
    S = w.bytes_per_rank

    with torch.cuda.stream(stream):
        xs = W.rank_inputs(w, device=dev)
        ys = [torch.empty_like(x) for x in xs]
    torch.cuda.synchronize()
    comm = dcc.Comm(n)
    comm.register_all("input", xs)
    comm.register_all("output", ys)
    h = comm.handle
    algo = "auto"
    blocks, threads = dcc.dcc_launch_shape(h, w.count, "bf16", algo)
    chosen = dcc.dcc_select_algo(h, w.count, "bf16")

    def step():
        dcc.dcc_allreduce(h, xs, ys, w.count, "bf16", algo, stream)

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    if comm.check(stream) != dcc.DCC_OK:
        raise RuntimeError("device failure during warm-up")

    clocks = ClockSampler(dist.local)
    clocks.start()
    dist.barrier()
    torch.cuda.synchronize()
    per, span_ms = time_launches(step, args.steps, stream)
    torch.cuda.synchronize()
    dist.barrier()
    clk = clocks.stop()
    rc = comm.check(stream)
    if rc != dcc.DCC_OK:
        raise RuntimeError("device failure in the timed region: " + dcc.dcc_error_string(rc))

    ms_per_step = dist.max(span_ms / args.steps)
    kernel_ms = sum(per) / len(per)
    # whole job: every replica processes one S-byte-per-rank AllReduce per step
    value = dist.ws * S / (ms_per_step / 1e3) / GB
    peak, peak_src = measured_peaks()
    algo_bytes = 2 * n * S
    achieved = algo_bytes / (kernel_ms / 1e3) / GB

    out = {
        "metric": "AllReduce algbw GB/s & % HBM roofline vs msg size at N=8 virtual ranks; p50 us @16KB",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": dist.ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "n_ranks": n, "elem": "bf16", "accumulate": "f32",
                   "count_per_rank": w.count, "bytes_per_rank": S, "algo": chosen,
                   "blocks_per_rank": blocks, "threads": threads,
                   "values": "N(0,1)*(1+r), seed 3+r", "l2": "inputs larger than L2 (2 GiB read per step)",
                   "parallelism": "replicas" if dist.ws > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": profiled_traffic(blocks, threads),
                     "algorithmic_bytes": algo_bytes, "peak_source": peak_src,
                     "kernel_ms": round(kernel_ms, 5)},
        "latency_us": {"p50": round(statistics.median(per) * 1e3, 2), "min": round(min(per) * 1e3, 2),
                       "mean": round(kernel_ms * 1e3, 2), "launches": len(per)},
        # NCCL-tests convention, for comparison with other reports only
        "busbw_gbs": round(value * 2 * (n - 1) / n, 2),
        "gpu_launches": args.steps,
        "clocks": clk,
    }

    if not args.quick:  # every replica, timed together
        out["e2e"] = e2e_host(dcc, comm, xs, ys, w, args, stream, dist)
    if dist.ws == 1 and not args.quick:  # single-GPU extras and the CPU leg (N = 1 only)
        out["sweep_c3"] = sweep_c3(dcc, dev, stream)
        # the AUTO crossover check runs here, in the state the tuning sweep
        # (--write-auto-table, a fresh process) measures in: later in this
        # process, after the other workloads, the same sweep read 0.1-0.2 us
        # less at 4-16 KiB and 0.3 us more for one-shot at 64 KiB, a shift no
        # single workload reproduced on its own
        crossover = crossover_sweep(dcc, dev, stream)[8]
        out["graph_node_floor_us"] = graph_node_floor(stream)
        out["eager_launch_floor"] = eager_floor(stream)
        out["sweep_large"] = sweep_large(dcc, dev, stream)
        out["other"] = other_workloads(dcc, dev, stream)
        gbs, cores, sample, _ = oracle_sample_run(args.cpu_seconds, args.cpu_elems)
        gbs1, _, sample1, _ = oracle_sample_run(3.0, args.cpu_elems // 8, threads=1)
        out["cpu_baseline"] = {"value": round(gbs, 3), "unit": "GB/s", "cores": cores,
                               "kind": "oracle", "sample": sample, "cpu_model": cpu_model(),
                               "single_thread": {"value": round(gbs1, 4), "unit": "GB/s",
                                                 "cores": 1, "sample": sample1}}
        out["crossover_n8"] = crossover
        # compact figures last, so that a reader keeping only the end of the line has them
        out["summary"] = summary(dcc, out)
        out["latency_16KiB_us"] = latency_16k(dcc, out)
    comm.close()
    return out


def latency_16k(dcc, out):
    """The metric's latency half: 8 ranks x 16 KiB bf16 (1 token x 8192) under AUTO."""
    row = next(r for r in out["sweep_c3"] if r["tokens"] == 1)
    algo = row["auto_algo"]
    m = row[algo]
    return {"algo": algo, "p50_event": m["p50_us"], "min_event": m["min_us"],
            "back_to_back": m["back_to_back_us"], "graph": m["graph_us"],
            "host_us_per_call": m["host_us_per_call"],
            "graph_node_floor": out["graph_node_floor_us"],
            "eager_floor_p50_event": out["eager_launch_floor"]["event_bracketed_p50_us"],
            "eager_floor_back_to_back": out["eager_launch_floor"]["back_to_back_us"]}


def summary(dcc, out):
    """Short figures of the extras (the detail is in the keys before)."""
    from driven_collective_communication_gb300 import build
    o = out["other"]
    table = build.load_auto_table()
    cross = {t: v["one_shot_max_bytes"] for t, v in out["crossover_n8"].items()}

    def summed(v, limit):  # the sweep's summed time with one-shot up to `limit` bytes
        return sum(a if size <= limit else b for size, a, b in zip(v["sizes"], v["one_shot_us"], v["two_shot_us"]))
    # what the compiled table costs over this sweep against the sweep's own best threshold, %:
    # near the crossover the schedules differ by hundredths of a microsecond, so the best
    # threshold itself moves between boxes while the cost of either stays small
    excess = {t: round(100.0 * (summed(v, table[8][t]) / summed(v, cross[t]) - 1.0), 2)
              for t, v in out["crossover_n8"].items()}
    return {
        "crossover_n8_bytes": cross,
        "crossover_n8_matches_compiled_table": all(table[8][t] == b for t, b in cross.items()),
        "crossover_n8_compiled_table_excess_pct": excess,
        "c2_int32_inplace_ms": {"one_shot": o["c2_int32_inplace_one_shot"]["ms"],
                                "two_shot": o["c2_int32_inplace_two_shot"]["ms"]},
        "c2_one_shot_roofline_frac": round(o["c2_int32_inplace_one_shot"]["hbm_gbs_2NS"]
                                           / measured_peaks()[0], 3),
        "c5_rs_ag_ms": [o["c5_reduce_scatter"]["ms"], o["c5_allgather"]["ms"]],
        "ring_barrier_per_hop_us": o["c5_ring_barrier"]["per_hop_us"],
        "fused_kp1024_us": o["linear_allreduce_bf16_n8_rows8192_kp1024"]["fused_us"],
        "fused_kp1024_weight_frac": round(o["linear_allreduce_bf16_n8_rows8192_kp1024"]["fused_weight_gbs"]
                                          / measured_peaks()[0], 3),
        # the tensor-core layer over 1 / 16 / 64 / 128 / 256 tokens (8 x 8192 x 1024 bf16) and
        # per-rank cuBLAS GEMM then the AllReduce on the same shapes, us
        "linear_tokens_us": {t: o["linear_tokens_bf16_n8_rows8192_kp1024_t%d" % t]["fused_tensor_us"]
                             for t in (1, 16, 64, 128, 256)},
        "gemm_then_allreduce_us": {t: o["linear_tokens_bf16_n8_rows8192_kp1024_t%d" % t]["gemm_then_allreduce_us"]
                                   for t in (1, 16, 64, 128, 256)},
    }


def e2e_host(dcc, comm, xs, ys, w, args, stream, dist):
    """The same AllReduce through dcc_allreduce_from_host: pinned host inputs
    copied in, the collective, outputs copied back -- all inside the timing.
    Every replica runs it between barriers; the job takes the slowest."""
    hin = [x.cpu().pin_memory() for x in xs]
    hout = [torch.empty_like(t).pin_memory() for t in hin]
    h = comm.handle

    def step():
        dcc.dcc_allreduce_from_host(h, hin, hout, xs, ys, w.count, "bf16", "auto", stream)

    for _ in range(2):
        step()
    stream.synchronize()
    steps = max(3, min(10, args.steps // 100))
    dist.barrier()
    t0 = time.perf_counter()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        step()
    ev1.record(stream)
    ev1.synchronize()
    wall = (time.perf_counter() - t0) / steps
    dist.barrier()
    ms = dist.max(ev0.elapsed_time(ev1) / steps)
    wall = dist.max(wall)
    nbytes = dist.ws * w.n_ranks * w.bytes_per_rank  # every replica's inputs in and outputs out
    return {"value": round(dist.ws * w.bytes_per_rank / (ms / 1e3) / GB, 3), "unit": "GB/s",
            "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": nbytes,
            "ms_per_step": round(ms, 3), "wall_ms_per_step": round(wall * 1e3, 3), "steps": steps}


def sweep_large(dcc, dev, stream):
    """algbw and fraction of the HBM roofline vs message size above L2: the
    8-rank bf16 AllReduce (AUTO) at 16 MiB .. 1 GiB per rank, inputs N(0,1)*(1+r)."""
    peak, _ = measured_peaks()
    res = []
    for mib in (16, 64, 256, 1024):
        count = (mib << 20) // 2
        w = W.with_count(W.C4, count)
        with torch.cuda.stream(stream):
            xs = W.rank_inputs(w, device=dev)
            ys = [torch.empty_like(x) for x in xs]
        torch.cuda.synchronize()
        with dcc.Comm(8) as c:
            c.register_all("input", xs)
            c.register_all("output", ys)
            step = dcc.prepare_allreduce(c.handle, xs, ys, count, "bf16", "auto", stream)
            for _ in range(LARGE_WARMUP):
                step()
            per, _ = time_launches(step, LARGE_STEPS, stream)
            # launches queued back to back (no event in between, so consecutive
            # launches overlap through programmatic dependent launch)
            b2b_ms = time_queued_span(step, 20, stream) / 1e3
            assert c.check(stream) == dcc.DCC_OK
        ms = statistics.median(per)
        hbm = 2 * 8 * (mib << 20) / ms / 1e6
        res.append({"bytes_per_rank": mib << 20, "ms": round(ms, 4), **spread(per),
                    "algbw_gbs": round((mib << 20) / ms / 1e6, 1), "hbm_gbs_2NS": round(hbm, 1),
                    "roofline_frac": round(hbm / peak, 4), "back_to_back_ms": round(b2b_ms, 4),
                    "back_to_back_roofline_frac": round(2 * 8 * (mib << 20) / b2b_ms / 1e6 / peak, 4)})
        del xs, ys
    return res


def graph_node_floor(stream, reps=100):
    """Time per node of a CUDA graph of near-empty kernels (torch's spin kernel
    with a zero count): the launch floor under the graph-amortised latencies."""
    for _ in range(10):
        torch.cuda._sleep(0)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            torch.cuda._sleep(0)
    with torch.cuda.stream(stream):
        g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(10):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return round(e0.elapsed_time(e1) * 1e3 / (10 * reps), 3)


def alternate(sets):
    """A callable returning sets[0], sets[1], ... in turn (the weights of
    consecutive layers)."""
    k = [0]

    def nxt():
        k[0] += 1
        return sets[(k[0] - 1) % len(sets)]
    return nxt


def graph_us(step, stream, reps=100, replays=10):
    """Device time per call of `step` inside a CUDA graph of `reps` calls,
    replayed `replays` times after one untimed replay (steady state)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            step()
    with torch.cuda.stream(stream):  # replay() launches on the current stream
        g.replay()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) * 1e3 / (replays * reps)


CROSSOVER_SIZES = tuple(k << 10 for k in (4, 8, 16, 32, 64, 128, 256))
DTYPE_RECIPES = {"int32": W.C2, "fp32": W.C1, "fp16": W.C5, "bf16": W.C4}


def crossover_rule(sizes, t_one, t_two):
    """The threshold (0 or a measured size) that minimises the summed time over
    the measured sizes when every size up to it runs one-shot and every larger
    one two-shot; ties go to the smaller threshold.  Summing over the sizes
    keeps one noisy point from moving the threshold the way a first-loss rule
    would."""
    best, best_gain, gain = 0, 0.0, 0.0
    for s, a, b in zip(sizes, t_one, t_two):
        gain += b - a  # time saved by running every size up to s one-shot
        if gain > best_gain + 1e-9:
            best, best_gain = s, gain
    return best


def crossover_sweep(dcc, dev, stream, ranks=(8,), dtypes=("int32", "fp32", "fp16", "bf16"),
                    sizes=CROSSOVER_SIZES, repeats=5):
    """Out-of-place AllReduce, one-shot vs two-shot, CUDA-graph-amortised us per
    call (median of `repeats` graphs) at each size, per rank count and dtype;
    returns {n: {dtype: {"sizes", "one_shot_us", "two_shot_us", "one_shot_max_bytes"}}}."""
    res = {}
    for n in ranks:
        res[n] = {}
        for dtype in dtypes:
            eb = W.ELEM_BYTES[dtype]
            w = W.with_count(DTYPE_RECIPES[dtype], max(sizes) // eb, n_ranks=n)
            with torch.cuda.stream(stream):
                xs = W.rank_inputs(w, device=dev)
                ys = [torch.empty_like(x) for x in xs]
            torch.cuda.synchronize()
            t = {"one_shot": [], "two_shot": []}
            with dcc.Comm(n) as c:
                c.register_all("input", xs)
                c.register_all("output", ys)
                for size in sizes:
                    count = size // eb
                    for algo in ("one_shot", "two_shot"):
                        step = dcc.prepare_allreduce(c.handle, xs, ys, count, dtype, algo, stream)
                        for _ in range(20):
                            step()
                        t[algo].append(statistics.median(graph_us(step, stream) for _ in range(repeats)))
                assert c.check(stream) == dcc.DCC_OK
            res[n][dtype] = {"sizes": list(sizes),
                             "one_shot_us": [round(v, 3) for v in t["one_shot"]],
                             "two_shot_us": [round(v, 3) for v in t["two_shot"]],
                             "one_shot_max_bytes": crossover_rule(sizes, t["one_shot"], t["two_shot"])}
            del xs, ys
    return res


def combine_sweeps(paths):
    """Mean timings of several sweeps (tuning JSONs written by --write-auto-table)
    and the thresholds the rule gives for the mean: single sweeps differ by a
    few hundredths of a microsecond, as much as one-shot and two-shot differ
    near the crossover."""
    docs = [json.load(open(p)) for p in paths]
    sweep = {}
    for n in docs[0]["timings_us"]:
        sweep[int(n)] = {}
        for t, r in docs[0]["timings_us"][n].items():
            rows = [d["timings_us"][n][t] for d in docs]
            one = [statistics.fmean(v) for v in zip(*[x["one_shot_us"] for x in rows])]
            two = [statistics.fmean(v) for v in zip(*[x["two_shot_us"] for x in rows])]
            sweep[int(n)][t] = {"sizes": r["sizes"], "one_shot_us": [round(v, 3) for v in one],
                                "two_shot_us": [round(v, 3) for v in two],
                                "one_shot_max_bytes": crossover_rule(r["sizes"], one, two)}
    return sweep, "mean of %d sweeps: %s" % (len(docs), "; ".join(d["source"] for d in docs))


def warm_up_gpu(dcc, dev, stream, seconds):
    """Back-to-back 8 x 64 MiB bf16 AllReduces for about `seconds`."""
    with torch.cuda.stream(stream):
        xs = [torch.ones(32 << 20, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        ys = [torch.empty_like(x) for x in xs]
    torch.cuda.synchronize()
    with dcc.Comm(8) as c:
        c.register_all("input", xs)
        c.register_all("output", ys)
        step = dcc.prepare_allreduce(c.handle, xs, ys, xs[0].numel(), "bf16", "two_shot", stream)
        t0 = time.time()
        while time.time() - t0 < seconds:
            for _ in range(50):
                step()
            torch.cuda.synchronize()
        assert c.check(stream) == dcc.DCC_OK
    del xs, ys


def write_auto_table(args):
    """Measure the crossover for every rank count 2..16 and dtype (or combine
    earlier sweeps, --combine) and write the tuning JSON that the library
    build compiles in (1 rank: no choice, 0)."""
    from driven_collective_communication_gb300 import build
    if args.combine:
        sweep, source = combine_sweeps(args.combine)
    else:
        build.build()
        from driven_collective_communication_gb300 import dcc
        torch.cuda.set_device(0)
        dev = torch.device("cuda", 0)
        stream = torch.cuda.Stream(device=dev)
        # the same state the bench's own crossover sweep meets: a GPU that has
        # been busy for a while (a cold start measured small messages 0.1-0.2 us
        # slower)
        warm_up_gpu(dcc, dev, stream, seconds=3.0)
        clocks = ClockSampler(0)
        clocks.start()
        sweep = crossover_sweep(dcc, dev, stream, ranks=tuple(range(2, 17)))
        ck = clocks.stop()
        props = torch.cuda.get_device_properties(dev)
        source = "python bench.py --write-auto-table on %s (%d SMs), %s, SM clock median %s MHz" % (
            props.name, props.multi_processor_count, time.strftime("%Y-%m-%d"), ck.get("sm_mhz"))
    table = {"1": {t: 0 for t in build.DTYPE_ORDER}}
    for n, per in sweep.items():
        table[str(n)] = {t: per[t]["one_shot_max_bytes"] for t in build.DTYPE_ORDER}
    doc = {
        "what": "largest out-of-place AllReduce message, in bytes per rank, that DCC_ALGO_AUTO runs "
                "one-shot (above it: two-shot), per rank count and element type",
        "rule": "the threshold (0 or a measured size) that minimises the time summed over the measured "
                "sizes when every size up to it runs one-shot and every larger one two-shot "
                "(CUDA-graph-amortised time per AllReduce, median of repeats)",
        "source": source,
        "one_shot_max_bytes": table,
        "timings_us": {str(n): per for n, per in sweep.items()},
    }
    with open(args.write_auto_table, "w") as f:
        json.dump(doc, f, indent=1)
    print(json.dumps({"auto_table": args.write_auto_table,
                      "one_shot_max_bytes": {n: table[n] for n in sorted(table, key=int)}}))


def sweep_c3(dcc, dev, stream):
    """Decode-shaped sizes, per algorithm: per-launch p50 / min / mean (CUDA
    events, launches queued ahead of the device so the host's submission time
    is not inside them), the same host-paced (one launch at a time from
    Python), the host cost per call, and the CUDA-graph-amortised us.  Steady
    state: the 8 x 16 KiB..4 MiB inputs stay in L2."""
    res = []
    for tokens in W.C3_TOKENS:
        w = W.c3(tokens)
        with torch.cuda.stream(stream):
            xs = W.rank_inputs(w, device=dev)
            ys = [torch.empty_like(x) for x in xs]
        torch.cuda.synchronize()
        comm = dcc.Comm(8)
        comm.register_all("input", xs)
        comm.register_all("output", ys)
        h = comm.handle
        # a working set (2 N S) that fits in L2 is a latency case, not an HBM-roofline one
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        row = {"tokens": tokens, "bytes_per_rank": w.bytes_per_rank,
               "working_set_in_l2": 2 * 8 * w.bytes_per_rank <= l2, "l2_bytes": l2,
               "auto_algo": dcc.dcc_select_algo(h, w.count, "bf16")}
        for algo in ("one_shot", "two_shot"):
            step = dcc.prepare_allreduce(h, xs, ys, w.count, "bf16", algo, stream)
            for _ in range(50):
                step()
            per, queued_ok = time_launches_queued(step, 1000, stream)
            p50 = statistics.median(per) * 1e3
            p_min, p_mean = min(per) * 1e3, statistics.mean(per) * 1e3
            eager, _ = time_launches(step, 1000, stream)
            span_us = time_queued_span(step, 100, stream)
            # host cost of one call (launch included), no device wait in between
            stream.synchronize()
            t = time.perf_counter()
            for _ in range(1000):
                step()
            host_us = (time.perf_counter() - t) * 1e3
            stream.synchronize()
            g_us = graph_us(step, stream)
            row[algo] = {"p50_us": round(p50, 2), "min_us": round(p_min, 2), "mean_us": round(p_mean, 2),
                         "queued_ahead": bool(queued_ok),
                         "host_paced_p50_us": round(statistics.median(eager) * 1e3, 2),
                         "back_to_back_us": round(span_us, 2),
                         "host_us_per_call": round(host_us, 2),
                         "graph_us": round(g_us, 2),
                         "algbw_gbs_graph": round(w.bytes_per_rank / (g_us * 1e-6) / GB, 2)}
        if w.bytes_per_rank <= dcc.DCC_LL_MAX_BYTES:  # in place: barrier one-shot vs LL
            for algo in ("one_shot", "one_shot_ll"):
                step = dcc.prepare_allreduce(h, xs, xs, w.count, "bf16", algo, stream)
                for _ in range(20):
                    step()
                row[algo + "_inplace"] = {"graph_us": round(graph_us(step, stream), 2)}
        assert comm.check(stream) == dcc.DCC_OK
        comm.close()
        res.append(row)
    return res


def other_workloads(dcc, dev, stream):
    """C2 (int32 in-place, both algorithms), C5 (ReduceScatter, AllGather,
    ring barrier): device-event timings."""
    out = {}
    # every AllReduce schedule on the headline size
    w = W.C4
    with torch.cuda.stream(stream):
        xs = W.rank_inputs(w, device=dev)
        ys = [torch.empty_like(x) for x in xs]
        scr = [torch.empty_like(x) for x in xs]
    torch.cuda.synchronize()
    comm = dcc.Comm(8)
    comm.register_all("input", xs)
    comm.register_all("output", ys)
    comm.register_all("scratch", scr)
    for algo in ("two_shot", "two_shot_bulk", "two_shot_scratch", "one_shot"):
        step = dcc.prepare_allreduce(comm.handle, xs, ys, w.count, "bf16", algo, stream)
        for _ in range(LARGE_WARMUP):
            step()
        per, _ = time_launches(step, LARGE_STEPS, stream)
        ms = statistics.median(per)
        out["c4_bf16_" + algo] = {"ms": round(ms, 4), **spread(per),
                                  "hbm_gbs_2NS": round(2 * 8 * w.bytes_per_rank / ms / 1e6, 1)}
    # MAX / MIN on the headline size (AUTO: the two-shot push kernels, raw-bit combines)
    for op in ("max", "min"):
        def step(op=op):
            dcc.dcc_allreduce_op(comm.handle, xs, ys, w.count, "bf16", op, "auto", stream)
        for _ in range(LARGE_WARMUP):
            step()
        per, _ = time_launches(step, LARGE_STEPS, stream)
        ms = statistics.median(per)
        out["c4_bf16_" + op] = {"ms": round(ms, 4), **spread(per),
                                "hbm_gbs_2NS": round(2 * 8 * w.bytes_per_rank / ms / 1e6, 1)}
    # the optional entry barrier: its cost on the headline size (one co-resident wave)
    dcc.dcc_set_entry_barrier(comm.handle, True)
    step = dcc.prepare_allreduce(comm.handle, xs, ys, w.count, "bf16", "two_shot", stream)
    for _ in range(LARGE_WARMUP):
        step()
    per, _ = time_launches(step, LARGE_STEPS, stream)
    dcc.dcc_set_entry_barrier(comm.handle, False)
    out["c4_bf16_two_shot_entry_barrier"] = {"ms": round(statistics.median(per), 4), **spread(per)}
    assert comm.check(stream) == dcc.DCC_OK
    comm.close()
    # the 2-rank fp32 1 MiB one-shot (a latency case: 4 MiB of traffic sits in L2)
    w1 = W.C1
    with torch.cuda.stream(stream):
        xs1 = W.rank_inputs(w1, device=dev)
        ys1 = [torch.empty_like(x) for x in xs1]
    torch.cuda.synchronize()
    with dcc.Comm(2) as c1:
        c1.register_all("input", xs1)
        c1.register_all("output", ys1)
        step = dcc.prepare_allreduce(c1.handle, xs1, ys1, w1.count, "fp32", "one_shot", stream)
        for _ in range(20):
            step()
        per, _ = time_launches(step, 200, stream)
        b2b_us = time_queued_span(step, 100, stream)
        assert c1.check(stream) == dcc.DCC_OK
        out["c1_fp32_n2_1MiB_one_shot"] = {"p50_us": round(statistics.median(per) * 1e3, 2),
                                           "min_us": round(min(per) * 1e3, 2),
                                           "mean_us": round(statistics.fmean(per) * 1e3, 2),
                                           "back_to_back_us": round(b2b_us, 2)}
    # ... and on the 16 KiB decode size, CUDA-graph amortised
    w16 = W.c3(1)
    with torch.cuda.stream(stream):
        xs16 = W.rank_inputs(w16, device=dev)
        ys16 = [torch.empty_like(x) for x in xs16]
    torch.cuda.synchronize()
    with dcc.Comm(8) as c16:
        c16.register_all("input", xs16)
        c16.register_all("output", ys16)
        res = {}
        for on in (False, True):
            dcc.dcc_set_entry_barrier(c16.handle, on)
            step = dcc.prepare_allreduce(c16.handle, xs16, ys16, w16.count, "bf16", "two_shot", stream)
            for _ in range(20):
                step()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(100):
                    step()
            with torch.cuda.stream(stream):
                g.replay()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(10):
                    g.replay()
                e1.record(stream)
            e1.synchronize()
            res["with_barrier_us" if on else "without_us"] = round(e0.elapsed_time(e1) * 1e3 / 1000, 2)
        assert c16.check(stream) == dcc.DCC_OK
        out["c3_16KiB_two_shot_entry_barrier_graph"] = res
    # the allocation-free entry point on the same 16 KiB decode size (two-shot
    # via its static array, cooperative launch): per launch and back to back
    ys16n = [torch.empty_like(x) for x in xs16]
    na = lambda: dcc.dcc_allreduce_noalloc(8, xs16, ys16n, w16.count, "bf16", stream)  # noqa: E731
    for _ in range(20):
        na()
    per, _ = time_launches(na, 200, stream)
    out["c3_16KiB_noalloc"] = {"p50_event_us": round(statistics.median(per) * 1e3, 2),
                               "back_to_back_us": round(time_queued_span(na, 100, stream), 2)}
    assert dcc.dcc_noalloc_check(stream)[0] == dcc.DCC_OK
    del xs, ys, scr
    # more ranks and another dtype at the large size (two-shot push, 256 MiB per rank)
    for n_ranks, dtype in ((2, "bf16"), (4, "bf16"), (16, "bf16"), (8, "fp32")):
        recipe = W.C4 if dtype == "bf16" else W.C1
        count = (256 << 20) // W.ELEM_BYTES[dtype]
        wk = W.with_count(recipe, count, n_ranks=n_ranks)
        with torch.cuda.stream(stream):
            xs = W.rank_inputs(wk, device=dev)
            ys = [torch.empty_like(x) for x in xs]
        torch.cuda.synchronize()
        with dcc.Comm(n_ranks) as cn:
            cn.register_all("input", xs)
            cn.register_all("output", ys)
            step = dcc.prepare_allreduce(cn.handle, xs, ys, count, dtype, "auto", stream)
            for _ in range(LARGE_WARMUP):
                step()
            per, _ = time_launches(step, LARGE_STEPS, stream)
            assert cn.check(stream) == dcc.DCC_OK
        ms = statistics.median(per)
        out["allreduce_%s_n%d_256MiB" % (dtype, n_ranks)] = {
            "ms": round(ms, 4), **spread(per), "algbw_gbs": round((256 << 20) / ms / 1e6, 1),
            "hbm_gbs_2NS": round(2 * n_ranks * (256 << 20) / ms / 1e6, 1)}
        del xs, ys
    w = W.C2
    with torch.cuda.stream(stream):
        xs = W.rank_inputs(w, device=dev)
    torch.cuda.synchronize()
    comm = dcc.Comm(8)
    comm.register_all("input", xs)
    for algo in ("one_shot", "two_shot"):
        def step():
            dcc.dcc_allreduce(comm.handle, xs, xs, w.count, "int32", algo, stream)
        for _ in range(LARGE_WARMUP):
            step()
        per, _ = time_launches(step, LARGE_STEPS, stream)
        ms = statistics.median(per)
        out["c2_int32_inplace_" + algo] = {"ms": round(ms, 4), **spread(per),
                                           "algbw_gbs": round(w.bytes_per_rank / ms / 1e6, 2),
                                           "hbm_gbs_2NS": round(2 * 8 * w.bytes_per_rank / ms / 1e6, 1)}
    assert comm.check(stream) == dcc.DCC_OK
    comm.close()
    del xs
    w = W.C5
    m = w.count // 8
    with torch.cuda.stream(stream):
        xs = W.rank_inputs(w, device=dev)
        rs = [torch.empty(m, dtype=torch.float16, device=dev) for _ in range(8)]
        ag = [torch.empty(w.count, dtype=torch.float16, device=dev) for _ in range(8)]
    torch.cuda.synchronize()
    comm = dcc.Comm(8)
    comm.register_all("input", xs)
    comm.register_all("output", rs)
    comm.register_all("output", ag)
    for name, fn, nbytes in (
            ("c5_reduce_scatter", lambda: dcc.dcc_reduce_scatter(comm.handle, xs, rs, m, "fp16", stream),
             8 * w.bytes_per_rank + w.bytes_per_rank),
            ("c5_allgather", lambda: dcc.dcc_allgather(comm.handle, rs, ag, m, "fp16", stream),
             w.bytes_per_rank + 8 * w.bytes_per_rank)):
        for _ in range(LARGE_WARMUP):
            fn()
        per, _ = time_launches(fn, LARGE_STEPS, stream)
        b2b_ms = time_queued_span(fn, 50, stream) / 1e3
        ms = statistics.median(per)
        out[name] = {"ms": round(ms, 4), **spread(per), "hbm_gbs": round(nbytes / ms / 1e6, 1),
                     "algorithmic_bytes": nbytes, "back_to_back_ms": round(b2b_ms, 4),
                     "back_to_back_hbm_gbs": round(nbytes / b2b_ms / 1e6, 1)}
    # the two halves as one stream-ordered pair (RS then AG of its output), back to back
    def rs_ag():
        dcc.dcc_reduce_scatter(comm.handle, xs, rs, m, "fp16", stream)
        dcc.dcc_allgather(comm.handle, rs, ag, m, "fp16", stream)
    b2b_ms = time_queued_span(rs_ag, 50, stream) / 1e3
    out["c5_reduce_scatter_then_allgather_back_to_back"] = {
        "ms": round(b2b_ms, 4), "hbm_gbs": round(2 * 9 * w.bytes_per_rank / b2b_ms / 1e6, 1)}
    assert comm.check(stream) == dcc.DCC_OK
    comm.close()
    # the same AllGather through PortChannels: the host proxy drives copy engines
    with dcc.Comm(8) as pc:
        pc.register_all("input", rs)
        pc.register_all("output", ag)
        dcc.dcc_proxy_start(pc.handle)
        fn = lambda: dcc.dcc_port_allgather(pc.handle, rs, ag, m, "fp16", stream)  # noqa: E731
        for _ in range(LARGE_WARMUP):
            fn()
        per, _ = time_launches(fn, LARGE_STEPS, stream)
        assert pc.check(stream) == dcc.DCC_OK
        assert dcc.dcc_proxy_stop(pc.handle) == dcc.DCC_OK
        ms = statistics.median(per)
        out["c5_allgather_port_channel"] = {"ms": round(ms, 4), **spread(per), "hbm_gbs": round(
            (w.bytes_per_rank + 8 * w.bytes_per_rank) / ms / 1e6, 1)}
    # fused row-parallel linear + AllReduce vs per-rank GEMV (cuBLAS) then AllReduce,
    # tensor-parallel decode shapes: hidden 8192 rows, 8 ranks, kp = 1024, 3584, 8192
    # (kp >= 3584 runs the bulk-copy kernel)
    for kp in (1024, 3584, 8192):
        rows = 8192
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        # two weight sets, layer i of a graph taking set i % 2 (as consecutive
        # layers of a model do): 2 x 134 MB at kp 1024 is more than L2, so no
        # layer finds its weights left in L2 by the one before
        wsets = [[(torch.randn(rows, kp, generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(8)]
                 for _ in range(2)]
        wts = wsets[0]
        nxt = alternate(wsets)
        xin = [torch.randn(kp, generator=g, device=dev).to(torch.bfloat16) for _ in range(8)]
        yf = [torch.empty(rows, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        part = [torch.empty(rows, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        ysep = [torch.empty(rows, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        hres = [torch.zeros(rows, dtype=torch.bfloat16, device=dev) for _ in range(8)]  # residual stream
        with dcc.Comm(8) as lc:
            for ws in wsets:
                lc.register_all("input", ws)
            lc.register_all("input", xin)
            lc.register_all("output", yf)
            lc.register_all("input", part)
            lc.register_all("output", ysep)
            lc.register_all("output", hres)
            fused = lambda: dcc.dcc_linear_allreduce(lc.handle, nxt(), xin, yf, rows, kp, "bf16", stream)  # noqa
            fused_res = lambda: dcc.dcc_linear_allreduce_residual(  # noqa: E731  h <- h + layer, in place
                lc.handle, nxt(), xin, hres, hres, rows, kp, "bf16", stream)
            ar = dcc.prepare_allreduce(lc.handle, part, ysep, rows, "bf16", "auto", stream)

            def unfused():
                ws = nxt()
                with torch.cuda.stream(stream):
                    for r in range(8):
                        torch.matmul(ws[r], xin[r], out=part[r])
                ar()
            res = {}
            for name, fn in (("fused", fused), ("fused_residual_inplace", fused_res),
                             ("gemv_then_allreduce", unfused)):
                for _ in range(5):
                    fn()
                g2 = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g2, stream=stream):
                    for _ in range(20):
                        fn()
                with torch.cuda.stream(stream):
                    g2.replay()
                    e0 = torch.cuda.Event(enable_timing=True)
                    e1 = torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    for _ in range(5):
                        g2.replay()
                    e1.record(stream)
                e1.synchronize()
                us = e0.elapsed_time(e1) * 1e3 / 100
                res[name + "_us"] = round(us, 2)
                res[name + "_weight_gbs"] = round(8 * rows * kp * 2 / (us * 1e-6) / GB, 1)
            assert lc.check(stream) == dcc.DCC_OK
        out["linear_allreduce_bf16_n8_rows8192_kp%d" % kp] = res
        del wsets, wts, xin, yf, part, ysep, hres
    # the row-parallel layer over a batch of tokens on the tensor cores vs
    # per-rank cuBLAS GEMM then the AllReduce (8 ranks x 8192 rows x kp 1024)
    for tokens in (1, 16, 64, 128, 256):
        rows, kp = 8192, 1024
        g = torch.Generator(device=dev)
        g.manual_seed(6)
        wsets = [[(torch.randn(rows, kp, generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(8)]
                 for _ in range(2)]  # alternating weight sets, as above
        wts = wsets[0]
        nxt = alternate(wsets)
        xin = [torch.randn(tokens, kp, generator=g, device=dev).to(torch.bfloat16) for _ in range(8)]
        yt = [torch.empty(tokens, rows, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        part = [torch.empty(tokens, rows, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        ysep = [torch.empty(tokens, rows, dtype=torch.bfloat16, device=dev) for _ in range(8)]
        hres = [torch.randn(tokens, rows, generator=g, device=dev).to(torch.bfloat16) for _ in range(8)]
        with dcc.Comm(8) as tc:
            for bufs, kind in ((wsets[0], "input"), (wsets[1], "input"), (xin, "input"), (part, "input"),
                               (yt, "output"), (ysep, "output"), (hres, "output")):
                tc.register_all(kind, bufs)
            fused = lambda: dcc.dcc_linear_allreduce_tokens(tc.handle, nxt(), xin, yt, tokens, rows, kp,  # noqa
                                                            "bf16", stream)
            fused_res = lambda: dcc.dcc_linear_allreduce_tokens_residual(  # noqa: E731 (h <- h + layer, in place)
                tc.handle, nxt(), xin, hres, hres, tokens, rows, kp, "bf16", stream)
            ar = dcc.prepare_allreduce(tc.handle, part, ysep, tokens * rows, "bf16", "auto", stream)

            def unfused():
                ws = nxt()
                with torch.cuda.stream(stream):
                    for r in range(8):
                        torch.matmul(xin[r], ws[r].t(), out=part[r])
                ar()
            res = {}
            # host cost of one eager call (argument checks, the cached launch
            # plan, the launch), arguments marshalled once, no device wait
            step = dcc.prepare_linear_allreduce_tokens(tc.handle, wts, xin, yt, tokens, rows, kp, "bf16", stream)
            for _ in range(3):
                step()
            stream.synchronize()
            t0 = time.perf_counter()
            for _ in range(200):
                step()
            res["fused_tensor_host_us_per_call"] = round((time.perf_counter() - t0) * 1e6 / 200, 2)
            stream.synchronize()
            for name, fn in (("fused_tensor", fused), ("fused_tensor_residual_inplace", fused_res),
                             ("gemm_then_allreduce", unfused)):
                for _ in range(3):
                    fn()
                us = graph_us(fn, stream, reps=20, replays=5)
                res[name + "_us"] = round(us, 2)
                res[name + "_tflops"] = round(2 * 8 * rows * kp * tokens / (us * 1e-6) / 1e12, 1)
                res[name + "_weight_gbs"] = round(8 * rows * kp * 2 / (us * 1e-6) / GB, 1)
            assert tc.check(stream) == dcc.DCC_OK
        out["linear_tokens_bf16_n8_rows8192_kp1024_t%d" % tokens] = res
        del wsets, wts, xin, yt, part, ysep, hres
    # the ring barrier: default transport (8 ranks: one cluster, distributed
    # shared memory) and the global-memory semaphores (DCC_RING_CLUSTER=0)
    for key, env in (("c5_ring_barrier", None), ("c5_ring_barrier_l2_semaphores", "0")):
        if env is not None:
            os.environ["DCC_RING_CLUSTER"] = env
        try:
            with dcc.Comm(8, connect="ring") as ring:
                ring.ring_barrier(100, stream)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                ring.ring_barrier(W.BARRIER_ITERS, stream)
                e1.record(stream)
                e1.synchronize()
                assert ring.check(stream) == dcc.DCC_OK
        finally:
            os.environ.pop("DCC_RING_CLUSTER", None)
        us = e0.elapsed_time(e1) * 1e3 / W.BARRIER_ITERS
        out[key] = {"iters": W.BARRIER_ITERS, "round_trip_us": round(us, 3), "per_hop_us": round(us / 8, 3)}
    return out


# ------------------------------------------------------------------ reference arm
def run_reference(args, dist):
    """The oracle timed as the reference arm on the host cores (rank 0 only)."""
    if dist.rank != 0:
        return None
    per_step_s = []
    threads = os.cpu_count() or 1
    import oracle
    w = W.C4
    elems = args.ref_elems
    xs = [W.to_storage(t) for t in W.rank_inputs(w, device="cpu", count=elems)]
    for _ in range(args.warmup):
        oracle.allreduce(xs, "bf16", nthreads=threads)
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.allreduce(xs, "bf16", nthreads=threads)
        per_step_s.append(time.perf_counter() - t)
    t_step = sum(per_step_s) / len(per_step_s)
    value = elems * 2 / t_step / GB
    sample = ("oracle AllReduce, N=8 bf16, first %d elements (%d MiB) of each rank's 256 MiB "
              "buffer per step" % (elems, elems * 2 >> 20))
    return {
        "impl": "reference",
        "metric": "AllReduce algbw GB/s & % HBM roofline vs msg size at N=8 virtual ranks; p50 us @16KB",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": dist.ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "n_ranks": 8, "elem": "bf16", "accumulate": "f32",
                   "count_per_rank": w.count, "sample_elems_per_rank": elems},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ profiling cases
PROFILE_CASES = ("allreduce_two_shot", "allreduce_two_shot_bulk", "allreduce_one_shot",
                 "allreduce_one_shot_inplace", "allreduce_two_shot_scratch", "allreduce_one_shot_ll",
                 "allreduce_two_shot_max", "reduce_scatter",
                 "allgather", "ring_barrier", "linear_allreduce", "linear_tokens")


def run_profile_case(args):
    """One operation, `warmup` + `steps` launches, on a reduced size: the
    command that Nsight Compute captures (a few hundred MB on the device)."""
    from driven_collective_communication_gb300 import build
    build.build()
    from driven_collective_communication_gb300 import dcc
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    recipe = {"bf16": W.C4, "fp16": W.C5, "int32": W.C2, "fp32": W.C1}[args.dtype]
    n = 8
    w = W.with_count(recipe, args.count, n_ranks=n)
    case = args.profile_case
    if case == "linear_allreduce":  # --count is kp; 8192 rows per rank, bf16
        rows, kp = 8192, args.count
        g = torch.Generator(device=dev)
        g.manual_seed(5)
        wts = [(torch.randn(rows, kp, generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(n)]
        xin = [torch.randn(kp, generator=g, device=dev).to(torch.bfloat16) for _ in range(n)]
        yf = [torch.empty(rows, dtype=torch.bfloat16, device=dev) for _ in range(n)]
        with dcc.Comm(n) as lc:
            lc.register_all("input", wts)
            lc.register_all("input", xin)
            lc.register_all("output", yf)
            for _ in range(args.warmup + args.steps):
                dcc.dcc_linear_allreduce(lc.handle, wts, xin, yf, rows, kp, "bf16")
            torch.cuda.synchronize()
            rc = lc.check()
        if rc != dcc.DCC_OK:
            raise RuntimeError(dcc.dcc_error_string(rc))
        print(json.dumps({"profile_case": case, "rows": rows, "kp": kp, "launches": args.warmup + args.steps}))
        return
    if case == "linear_tokens":  # --count is the number of tokens; 8192 rows x kp 1024 per rank, bf16
        tokens, rows, kp = args.count, 8192, 1024
        g = torch.Generator(device=dev)
        g.manual_seed(6)
        wts = [(torch.randn(rows, kp, generator=g, device=dev) * 0.02).to(torch.bfloat16) for _ in range(n)]
        xin = [torch.randn(tokens, kp, generator=g, device=dev).to(torch.bfloat16) for _ in range(n)]
        yt = [torch.empty(tokens, rows, dtype=torch.bfloat16, device=dev) for _ in range(n)]
        with dcc.Comm(n) as tc:
            tc.register_all("input", wts)
            tc.register_all("input", xin)
            tc.register_all("output", yt)
            for _ in range(args.warmup + args.steps):
                dcc.dcc_linear_allreduce_tokens(tc.handle, wts, xin, yt, tokens, rows, kp, "bf16")
            torch.cuda.synchronize()
            rc = tc.check()
        if rc != dcc.DCC_OK:
            raise RuntimeError(dcc.dcc_error_string(rc))
        print(json.dumps({"profile_case": case, "tokens": tokens, "rows": rows, "kp": kp,
                          "launches": args.warmup + args.steps}))
        return
    xs = W.rank_inputs(w, device=dev)
    comm = dcc.Comm(n, connect="ring" if case == "ring_barrier" else "all")
    if case == "reduce_scatter":
        m = w.count // n
        ys = [torch.empty(m, dtype=xs[0].dtype, device=dev) for _ in range(n)]
        fn = lambda: dcc.dcc_reduce_scatter(comm.handle, xs, ys, m, args.dtype)  # noqa: E731
    elif case == "allgather":
        m = w.count // n
        xs = [x[:m].clone() for x in xs]
        ys = [torch.empty(w.count, dtype=xs[0].dtype, device=dev) for _ in range(n)]
        fn = lambda: dcc.dcc_allgather(comm.handle, xs, ys, m, args.dtype)  # noqa: E731
    elif case == "ring_barrier":
        ys = []
        fn = lambda: dcc.dcc_ring_barrier(comm.handle, W.BARRIER_ITERS)  # noqa: E731
    else:
        algo = case[len("allreduce_"):]
        inplace = algo.endswith("_inplace")
        algo = algo.replace("_inplace", "")
        op = "sum"
        for o in ("max", "min"):
            if algo.endswith("_" + o):
                op, algo = o, algo[: -len(o) - 1]
        ys = xs if inplace else [torch.empty_like(x) for x in xs]
        if algo == "two_shot_scratch":
            comm.register_all("scratch", [torch.empty_like(x) for x in xs])
        fn = lambda: dcc.dcc_allreduce_op(comm.handle, xs, ys, w.count, args.dtype, op, algo)  # noqa: E731
    if case != "ring_barrier":
        comm.register_all("input", xs)
        if ys is not xs:
            comm.register_all("output", ys)
    for _ in range(args.warmup + args.steps):
        fn()
    torch.cuda.synchronize()
    rc = comm.check()
    comm.close()
    if rc != dcc.DCC_OK:
        raise RuntimeError(dcc.dcc_error_string(rc))
    print(json.dumps({"profile_case": case, "dtype": args.dtype, "count_per_rank": w.count,
                      "launches": args.warmup + args.steps}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--profile-case", choices=PROFILE_CASES, default=None,
                    help="run one operation for an Nsight Compute capture (no timing)")
    ap.add_argument("--count", type=int, default=1 << 24, help="elements per rank (profile case)")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "fp16", "int32", "fp32"])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--quick", action="store_true", help="headline only (no sweep, e2e, CPU leg)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--cpu-elems", type=int, default=1 << 24)
    ap.add_argument("--ref-elems", type=int, default=1 << 22)
    ap.add_argument("--write-auto-table", default=None, metavar="PATH",
                    help="measure the one-shot/two-shot crossover for 2..16 ranks and write the tuning JSON")
    ap.add_argument("--combine", nargs="+", default=None, metavar="SWEEP",
                    help="with --write-auto-table: average earlier sweeps instead of measuring")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile_case:
        run_profile_case(args)
        return
    if args.write_auto_table:
        write_auto_table(args)
        return
    dist = Dist()
    try:
        out = run_reference(args, dist) if args.impl == "reference" else run_ours(args, dist)
        if out is not None and dist.rank == 0:
            print(json.dumps(out), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
