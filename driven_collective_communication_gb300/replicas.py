"""Replica bookkeeping for running the benchmark on several GPUs of one node.

The virtual-rank collectives run all N ranks inside one kernel on one GPU, so
there is nothing to exchange between GPUs: under torchrun every process runs
an independent replica on its own GPU ("replicas only").  This module holds
the only cross-process steps -- a barrier around the timed region and the
max / sum of the per-replica figures -- over the gloo backend (CPU), reading
RANK / LOCAL_RANK / WORLD_SIZE / MASTER_* from the environment.
"""
import os

import torch


def dist_env():
    """(world size, rank, local rank) from the torchrun environment (1, 0, 0 without it)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Dist:
    def __init__(self):
        self.ws, self.rank, self.local = dist_env()
        self.pg = None
        if self.ws > 1:
            import torch.distributed as td
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            td.init_process_group("gloo", rank=self.rank, world_size=self.ws)
            self.pg = td

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x):
        if not self.pg:
            return x
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x):
        if not self.pg:
            return x
        t = torch.tensor([float(x)], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


