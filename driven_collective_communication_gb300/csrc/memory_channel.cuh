// memory_channel.cuh -- device side of a MemoryChannel between two virtual ranks.
//
// MSCCL++ README, "PortChannel and MemoryChannel": with a MemoryChannel the
// calling GPU threads themselves load from and store to the peer's memory, so
// bandwidth takes many threads.  "On-GPU Communication Interfaces: Channels"
// gives the method set -- put (local memory into the peer's), signal (tell the
// peer this point is reached with earlier memory operations finished), flush
// (earlier channel operations finished as seen from this GPU) and wait (until
// the peer has signalled) -- and a barrier made of them.  get is listed with put in the
// project summary ("How It Works").
//
// GB300 reading, one GPU, N virtual ranks:
//  * the peer's memory is another allocation in the same HBM, so put/get are
//    16-byte vector stores/loads by many threads (warp-cooperative, one
//    vector per lane per step);
//  * signal is a release-ordered atomic increment at GPU scope on the peer's
//    inbound counter for this channel; wait is an acquire-ordered spin until
//    the inbound counter reaches the waiter's own count of completed waits;
//    flush is a GPU-scope fence (stores to HBM are synchronous, so nothing
//    else is outstanding);
//  * counters only grow (64-bit, no reset), and the waiter keeps its count in
//    device memory, so repeated calls and CUDA-graph replays never need a
//    reset and never reuse a stale epoch;
//  * every wait is bounded: after the communicator's limit it records the
//    failure in the status word and returns false; a wait also gives up as
//    soon as any other wait has failed, so a kernel always ends.
#pragma once
#include <cstdint>

#include "dcc_internal.h"

namespace dcc {

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long ld_relaxed_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned long long* p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may begin launching while the kernel before it on the stream
// is still finishing; griddepcontrol.wait then blocks until that kernel has
// completed and its memory operations are visible, so it must come before
// any access to global memory.  launch_dependents lets the next such kernel
// begin launching (it waits in turn).  Both are no-ops in a launch without
// the attribute.  Only kernels whose CTAs never wait on one another take it.
__device__ __forceinline__ void pdl_prologue() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte vector accesses.  Peer data that another CTA wrote in this kernel is
// read at L2 (ld.global.cg) so that no stale L1 line can be returned.
__device__ __forceinline__ uint4 ld_vec(const uint4* p) { return *p; }
__device__ __forceinline__ uint4 ld_vec_l2(const uint4* p) { return __ldcg(p); }
__device__ __forceinline__ void st_vec(uint4* p, uint4 v) { *p = v; }

// Bounds check of one data access (bounds-checked build only; otherwise a
// constant true that the compiler removes): [off, off + bytes) from the
// pointer of buffer `kind` of `rank` must lie inside the extent the host put
// in a.ext.  On a violation the first one is recorded in the status word and
// the caller skips the access, so the kernel's control flow (and every
// barrier in it) stays the same and the kernel ends normally.
template <typename A>
__device__ __forceinline__ bool in_bounds(const DevComm& dc, const A& a, int kind, int rank, size_t off,
                                          size_t bytes) {
#if DCC_CHECK_BOUNDS
  const size_t e = a.ext[kind][rank];
  if (off <= e && bytes <= e - off) return true;
  atomicCAS(dc.status, 0ull, pack_bounds(rank, kind, off));
  return false;
#else
  (void)dc; (void)a; (void)kind; (void)rank; (void)off; (void)bytes;
  return true;
#endif
}

// ---------------------------------------------------------------- channel
struct MemoryChannel {
  const char* remote_src;                 // peer memory this rank gets from
  char* remote_dst;                       // peer memory this rank puts into
  unsigned long long* remote_inbound;     // peer's counter of this rank's signals
  const unsigned long long* local_inbound;  // this rank's counter of the peer's signals
  unsigned long long* local_expect;       // this rank's count of completed waits on the peer

  __device__ static MemoryChannel make(const DevComm& dc, int self, int peer, int blk,
                                       const void* peer_src, void* peer_dst) {
    MemoryChannel ch;
    ch.remote_src = static_cast<const char*>(peer_src);
    ch.remote_dst = static_cast<char*>(peer_dst);
    ch.remote_inbound = dc.sem + sem_slot(peer, self, blk) * kSemWords;
    ch.local_inbound = dc.sem + sem_slot(self, peer, blk) * kSemWords;
    ch.local_expect = dc.expect + sem_slot(self, peer, blk);
    return ch;
  }

  // get / put of one 16-byte vector at vector index i of the peer's memory
  __device__ __forceinline__ uint4 read(size_t i) const {
    return ld_vec(reinterpret_cast<const uint4*>(remote_src) + i);
  }
  __device__ __forceinline__ void write(size_t i, uint4 v) const {
    st_vec(reinterpret_cast<uint4*>(remote_dst) + i, v);
  }

  // put: remote_dst[remote_off, +bytes) <- local[local_off, +bytes), 16-byte
  // vectors, lanes lane, lane+nlanes, ... of the calling group.  Offsets and
  // bytes are multiples of 16 (checked on the host).
  __device__ __forceinline__ void put(size_t remote_off, const char* local, size_t local_off,
                                      size_t bytes, unsigned lane, unsigned nlanes) const {
    const uint4* s = reinterpret_cast<const uint4*>(local + local_off);
    uint4* d = reinterpret_cast<uint4*>(remote_dst + remote_off);
    for (size_t i = lane; i < bytes / 16; i += nlanes) st_vec(d + i, ld_vec(s + i));
  }

  // get: local[local_off, +bytes) <- remote_src[remote_off, +bytes)
  __device__ __forceinline__ void get(size_t remote_off, char* local, size_t local_off,
                                      size_t bytes, unsigned lane, unsigned nlanes) const {
    const uint4* s = reinterpret_cast<const uint4*>(remote_src + remote_off);
    uint4* d = reinterpret_cast<uint4*>(local + local_off);
    for (size_t i = lane; i < bytes / 16; i += nlanes) st_vec(d + i, ld_vec_l2(s + i));
  }

  // flush: every memory operation this thread has issued (and, through a
  // preceding __syncthreads, its CTA's) is ordered before what follows at GPU
  // scope.
  __device__ __forceinline__ void flush() const { fence_acq_rel_gpu(); }

  // signal: one thread.  Release: all memory operations ordered before it
  // (this thread's, and the CTA's through a preceding __syncthreads) become
  // visible to the peer before the peer's wait returns.
  __device__ __forceinline__ void signal(const DevComm& dc, int self) const {
    if (dc.skip_signal_rank == self) return;  // test knob: a lost signal
    red_release_gpu_add(remote_inbound, 1ull);
  }

  // wait: one thread.  `expected` is the caller's register copy of
  // *local_expect; it is advanced by one and the call spins until the peer's
  // signals reach it.  Returns false if the wait gave up (time limit, or
  // another wait of this launch already failed).
  // Each poll is an acquire load (measured on GB300 faster than relaxed polls
  // followed by one acquire fence: 4.8 vs 6.5 us for an in-place 8-rank 16 KiB
  // one-shot, whose chunk barrier is one signal/wait round).
  __device__ __forceinline__ bool wait(const DevComm& dc, unsigned long long& expected, int self,
                                       int peer, int blk) const {
    expected += 1;
    if (ld_acquire_gpu(local_inbound) >= expected) return true;
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 1;; ++it) {
      if (ld_acquire_gpu(local_inbound) >= expected) return true;
      if ((it & 31u) == 0) {
        if (ld_relaxed_gpu(dc.status) != 0ull) return false;
        if (global_timer_ns() - t0 > dc.timeout_ns) {
          atomicCAS(dc.status, 0ull, pack_status(kStatusTimeout, self, peer, blk));
          return false;
        }
      }
    }
  }
};

// Barrier among the N CTAs that share block slot `blk` (one per rank): every
// thread's prior memory operations are complete for all N ranks when it
// returns true.  Thread p < N (p != self) owns the channel to peer p: it
// signals p (the release covers what a flush would) and waits for p's signal, holding its completed-wait
// count in `expected` (loaded by the caller from the channel's local_expect
// and stored back at kernel end).  All threads of the CTA must call it.
__device__ __forceinline__ bool group_barrier(const DevComm& dc, int self, int n, int blk,
                                              unsigned long long& expected) {
  __syncthreads();
  bool ok = true;
  const int p = threadIdx.x;
  if (p < n && p != self) {
    MemoryChannel ch = MemoryChannel::make(dc, self, p, blk, nullptr, nullptr);
    ch.signal(dc, self);
    ok = ch.wait(dc, expected, self, p, blk);
  }
  return __syncthreads_and(ok) != 0;
}

// The two halves of group_barrier, for a pipelined caller: group_signal
// tells every peer that this CTA has finished reading (its threads' loads are
// consumed before the block barrier), group_wait waits for every peer's
// matching signal.
__device__ __forceinline__ void group_signal(const DevComm& dc, int self, int n, int blk) {
  __syncthreads();
  const int p = threadIdx.x;
  if (p < n && p != self) {
    MemoryChannel ch = MemoryChannel::make(dc, self, p, blk, nullptr, nullptr);
    ch.signal(dc, self);
  }
}
__device__ __forceinline__ bool group_wait(const DevComm& dc, int self, int n, int blk,
                                           unsigned long long& expected) {
  bool ok = true;
  const int p = threadIdx.x;
  if (p < n && p != self) {
    MemoryChannel ch = MemoryChannel::make(dc, self, p, blk, nullptr, nullptr);
    ok = ch.wait(dc, expected, self, p, blk);
  }
  return __syncthreads_and(ok) != 0;
}

}  // namespace dcc
