"""GB300-native virtual-rank collectives: sum AllReduce (one-shot, two-shot),
ReduceScatter, AllGather and a signal/wait ring barrier, built on a device-side
MemoryChannel (put/get/signal/wait/flush) in hand-written sm_103a kernels.

The CUDA library is loaded by ``driven_collective_communication_gb300.dcc``;
importing that module fails loudly when the library has not been built.
"""
__all__ = ["dcc", "workloads"]
