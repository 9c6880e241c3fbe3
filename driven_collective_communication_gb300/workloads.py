"""Seeded synthetic inputs for the virtual-rank collectives.

This module holds the input recipes only -- shapes, value distributions and
seeds -- and none of the collectives' arithmetic.  Both the CUDA path's tests
and the oracle's tests draw their rank buffers from here, so the two sides
always see the same bytes.

Each rank's buffer comes from its own ``torch.Generator`` seeded with
``seed0 + rank`` on the device the buffer is made on (CPU and CUDA generators
give different streams; a caller that compares two sides generates once and
copies).  The pages name no dataset or benchmark suite; every workload is
synthetic by construction, shaped like the five configurations below.
"""
from dataclasses import dataclass, field

import torch

TORCH_DTYPES = {"int32": torch.int32, "fp32": torch.float32,
                "fp16": torch.float16, "bf16": torch.bfloat16}
ELEM_BYTES = {"int32": 4, "fp32": 4, "fp16": 2, "bf16": 2}


@dataclass(frozen=True)
class Workload:
    name: str
    n_ranks: int
    dtype: str
    count: int                 # elements per rank buffer
    dist: str                  # "randint" | "normal" | "normal_scaled" | "uniform"
    seed0: int
    lo: int = 0                # randint bounds, inclusive
    hi: int = 0
    inplace: bool = False
    algos: tuple = field(default=("two_shot",))

    @property
    def bytes_per_rank(self) -> int:
        return self.count * ELEM_BYTES[self.dtype]


# Sizes, value ranges and seeds of the five workloads.  C3 is a family: message
# = tokens x 8192 hidden bf16 elements per rank (tensor-parallel decode shapes).
C1 = Workload("allreduce_fp32_n2_1MiB", 2, "fp32", 262144, "randint", 0, -8, 8,
              inplace=False, algos=("one_shot",))
C2 = Workload("allreduce_int32_n8_64MiB_inplace", 8, "int32", 16777216, "randint", 1,
              -(2 ** 20), 2 ** 20, inplace=True, algos=("one_shot", "two_shot"))
C3_TOKENS = (1, 2, 4, 8, 16, 32, 64, 128, 256)
C3_HIDDEN = 8192
C4 = Workload("allreduce_bf16_n8_256MiB", 8, "bf16", 134217728, "normal_scaled", 3,
              algos=("two_shot",))
C5 = Workload("rs_ag_fp16_n8_64MiB", 8, "fp16", 33554432, "uniform", 4)
BARRIER_ITERS = 10000


def c3(tokens: int) -> Workload:
    return Workload("allreduce_bf16_n8_decode_t%d" % tokens, 8, "bf16", tokens * C3_HIDDEN,
                    "normal", 2, algos=("one_shot", "two_shot"))


def with_count(w: Workload, count: int, n_ranks: int = None) -> Workload:
    """The same recipe at another size (and optionally another rank count)."""
    return Workload(w.name + "_count%d" % count, n_ranks or w.n_ranks, w.dtype, count, w.dist,
                    w.seed0, w.lo, w.hi, w.inplace, w.algos)


def rank_input(w: Workload, rank: int, device="cpu", count: int = None) -> torch.Tensor:
    """Rank ``rank``'s input buffer for workload ``w`` (seed = seed0 + rank)."""
    n = w.count if count is None else count
    g = torch.Generator(device=device)
    g.manual_seed(w.seed0 + rank)
    if w.dist == "randint":
        x = torch.randint(w.lo, w.hi + 1, (n,), generator=g, device=device, dtype=torch.int64)
        return x.to(TORCH_DTYPES[w.dtype])
    if w.dist == "normal":
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        return x.to(TORCH_DTYPES[w.dtype])
    if w.dist == "normal_scaled":
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        x.mul_(float(1 + rank))
        return x.to(TORCH_DTYPES[w.dtype])
    if w.dist == "uniform":
        x = torch.rand(n, generator=g, device=device, dtype=torch.float32)
        x.mul_(2.0).sub_(1.0)
        return x.to(TORCH_DTYPES[w.dtype])
    raise ValueError("unknown distribution %r" % (w.dist,))


def rank_inputs(w: Workload, device="cpu", count: int = None):
    return [rank_input(w, r, device=device, count=count) for r in range(w.n_ranks)]


def to_storage(t: torch.Tensor):
    """A CPU tensor as the numpy raw-storage array the oracle takes
    (16-bit floats as uint16 bit patterns)."""
    t = t.detach().cpu().contiguous()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()


def from_storage(a, dtype: str) -> torch.Tensor:
    """Inverse of ``to_storage``."""
    import numpy as np
    if dtype in ("fp16", "bf16"):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(TORCH_DTYPES[dtype])
    return torch.from_numpy(np.ascontiguousarray(a))
