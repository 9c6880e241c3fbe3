// sync_kernels.cu -- ring barrier and the stand-alone MemoryChannel primitives.
//
// MSCCL++ README, "On-GPU Communication Interfaces: Channels": one thread
// suffices for the barrier (signal, optional flush, wait), and put copies from
// the local GPU's memory to the remote's.  The ring barrier chains that
// two-rank barrier around all N ranks so one iteration is a token passed
// rank 0 -> 1 -> ... -> N-1 -> 0.
#include <cuda_runtime.h>

#include "memory_channel.cuh"
#include "sync_kernels.cuh"

namespace dcc {

// One CTA (one active thread) per rank.  Block slot 0 of the semaphores.
__global__ void k_ring_barrier(DevComm dc, int iters) {
  if (threadIdx.x != 0) return;
  const int n = dc.n, rank = blockIdx.x;
  const int next = (rank + 1) % n, prev = (rank + n - 1) % n;
  const MemoryChannel to_next = MemoryChannel::make(dc, rank, next, 0, nullptr, nullptr);
  const MemoryChannel from_prev = MemoryChannel::make(dc, rank, prev, 0, nullptr, nullptr);
  unsigned long long expected = *from_prev.local_expect;
  for (int it = 0; it < iters; ++it) {
    if (rank == 0) {
      to_next.signal(dc, rank);
      if (!from_prev.wait(dc, expected, rank, prev, 0)) break;
    } else {
      if (!from_prev.wait(dc, expected, rank, prev, 0)) break;
      to_next.signal(dc, rank);
    }
  }
  *from_prev.local_expect = expected;
}

// CTA 0 plays src: put, then (optionally) flush + signal.  CTA 1 plays dst:
// waits for that signal on its own channel to src.
__global__ void k_channel_put(DevComm dc, PrimArgs pa) {
  const DevChannel& c = pa.table[pa.src * DCC_MAX_RANKS + pa.dst];
  if (blockIdx.x == 0) {
    const MemoryChannel ch = MemoryChannel::make(dc, pa.src, pa.dst, 0, c.remote_in, c.remote_out);
    ch.put(pa.remote_off, c.local_in, pa.local_off, pa.bytes, threadIdx.x, blockDim.x);
    if (pa.signal) {
      __syncthreads();
      if (threadIdx.x == 0) {
        ch.flush();
        ch.signal(dc, pa.src);
      }
    }
  } else if (pa.signal && threadIdx.x == 0) {
    const MemoryChannel back = MemoryChannel::make(dc, pa.dst, pa.src, 0, nullptr, nullptr);
    unsigned long long expected = *back.local_expect;
    back.wait(dc, expected, pa.dst, pa.src, 0);
    *back.local_expect = expected;
  }
}

__global__ void k_channel_get(DevComm dc, PrimArgs pa) {
  const DevChannel& c = pa.table[pa.src * DCC_MAX_RANKS + pa.dst];
  const MemoryChannel ch = MemoryChannel::make(dc, pa.src, pa.dst, 0, c.remote_in, c.remote_out);
  ch.get(pa.remote_off, c.local_out, pa.local_off, pa.bytes, threadIdx.x, blockDim.x);
}

const void* ring_barrier_kernel() { return reinterpret_cast<const void*>(&k_ring_barrier); }
const void* channel_put_kernel() { return reinterpret_cast<const void*>(&k_channel_put); }
const void* channel_get_kernel() { return reinterpret_cast<const void*>(&k_channel_get); }

}  // namespace dcc
