"""The multi-GPU (replica) path of the benchmark on CPU: two gloo ranks run the
barrier / max / sum steps bench.py uses around its timed region."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from driven_collective_communication_gb300.replicas import Dist
    d = Dist()
    try:
        d.barrier()
        # per-replica step time: rank r took (r + 1) ms; the job takes the slowest
        mx = d.max(float(rank + 1))
        sm = d.sum(float(rank + 1))
        q.put((rank, d.ws, d.rank, d.local, mx, sm))
    finally:
        d.close()


def test_two_gloo_replicas_agree_on_max_and_sum():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ws, r, local, mx, sm in res:
        assert ws == world and r == rank and local == rank
        assert mx == 2.0 and sm == 3.0


def test_single_process_needs_no_process_group(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    from driven_collective_communication_gb300.replicas import Dist
    d = Dist()
    assert (d.ws, d.rank, d.local) == (1, 0, 0)
    assert d.max(3.5) == 3.5 and d.sum(2.0) == 2.0
    d.barrier()
    d.close()
