// port_channel.cuh -- device side of a PortChannel: one GPU thread hands
// operations to a host-side proxy through a FIFO of triggers.
//
// MSCCL++ README, "PortChannel and MemoryChannel": a PortChannel call hands
// the work to a helper on the host, which performs the transfer (cudaMemcpy*
// here) or the synchronisation, so a single GPU thread can drive it.
// "Host-Side Communication Proxy": that helper is a host thread that keeps
// polling a FIFO into which GPU threads place triggers (FifoDeviceHandle::push
// of a ProxyTrigger with fields fst/snd); applications may replace its trigger
// handling with their own.
//
// Layout and protocol (both sides):
//  * the FIFO is a ring of 16-byte triggers {fst, snd} in pinned, mapped host
//    memory; fst == 0 marks a free slot.  A pusher claims slot k with an
//    atomic increment of the device-side head, waits (bounded) until
//    k - tail < capacity, writes snd, then publishes fst with a system-scope
//    release store.  The proxy reads fst with acquire, handles the trigger,
//    clears fst and advances tail (release).
//  * built-in triggers have bit 63 of fst set: bits 59..61 are the PUT /
//    SIGNAL / FLUSH flags, bits 48..55 the destination rank, 40..47 the source
//    rank, 0..39 the byte count; snd holds the destination offset (low 32 bits)
//    and the source offset (high 32 bits) in 16-byte units, relative to the
//    destination's first OUTPUT window and the source's first INPUT window.
//    Any other non-zero fst is a custom trigger for the user's handler.
//  * SIGNAL: the proxy bumps its count of (src -> dst) signals and writes the
//    new count into port_sem[dst][src] in stream order after the copies it
//    issued before; the destination waits until that count reaches its own
//    number of completed waits (reset-free, like the MemoryChannel epochs).
//  * FLUSH: the proxy writes the trigger's sequence number + 1 into `done`
//    in stream order; the pusher waits until done passes its sequence number.
#pragma once
#include "memory_channel.cuh"

namespace dcc {

struct ProxyTrigger {
  unsigned long long fst;
  unsigned long long snd;
};

constexpr unsigned long long kTrigBuiltin = 1ull << 63;
constexpr unsigned long long kTrigPut = 1ull << 59;
constexpr unsigned long long kTrigSignal = 1ull << 60;
constexpr unsigned long long kTrigFlush = 1ull << 61;
constexpr unsigned long long kTrigSizeMask = (1ull << 40) - 1;

__host__ __device__ inline unsigned long long trig_fst(unsigned long long flags, int src, int dst,
                                                       unsigned long long bytes) {
  return kTrigBuiltin | flags | ((unsigned long long)(dst & 0xFF) << 48) |
         ((unsigned long long)(src & 0xFF) << 40) | (bytes & kTrigSizeMask);
}
__host__ __device__ inline unsigned long long trig_snd(size_t dst_off, size_t src_off) {
  return (unsigned long long)(dst_off / 16) | ((unsigned long long)(src_off / 16) << 32);
}

// Device view of the proxy's FIFO and completion words.
struct PortDev {
  ProxyTrigger* slots;                 // host-mapped ring
  unsigned long long* tail;            // host-mapped: triggers the proxy has taken
  unsigned long long* head;            // device: next slot to claim
  unsigned long long* done;            // device: flushed sequence + 1 (written by the proxy's stream)
  unsigned long long* sem;             // device: [dst][src] signal counts (kSemWords apart)
  unsigned long long* expect;          // device: [dst][src] completed waits
  unsigned long long capacity;
};

__device__ __forceinline__ unsigned long long ld_acquire_sys(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.sys.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed_sys(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_release_sys(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.sys.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Bounded spin until *p >= target (p written by the host or by a stream memory
// operation); records a timeout for (rank, peer).
__device__ __forceinline__ bool port_spin_ge(const unsigned long long* p, unsigned long long target,
                                             const DevComm& dc, int rank, int peer) {
  const unsigned long long t0 = global_timer_ns();
  for (unsigned it = 0;; ++it) {
    if (ld_acquire_sys(p) >= target) return true;
    if ((it & 31u) == 31u) {
      if (ld_relaxed_gpu(dc.status) != 0ull) return false;
      if (global_timer_ns() - t0 > dc.timeout_ns) {
        atomicCAS(dc.status, 0ull, pack_status(kStatusTimeout, rank, peer, 0));
        return false;
      }
    }
  }
}

// FifoDeviceHandle::push: returns false (status recorded) if the FIFO stayed
// full past the wait limit.  `seq` receives the trigger's sequence number.
__device__ __forceinline__ bool fifo_push(const PortDev& pd, ProxyTrigger t, unsigned long long& seq,
                                          const DevComm& dc, int rank) {
  seq = atomicAdd(pd.head, 1ull);
  if (seq >= pd.capacity && !port_spin_ge(pd.tail, seq - pd.capacity + 1, dc, rank, rank)) return false;
  ProxyTrigger* s = pd.slots + (seq % pd.capacity);
  st_relaxed_sys(&s->snd, t.snd);
  st_release_sys(&s->fst, t.fst);
  return true;
}

struct PortChannel {
  PortDev pd;
  int src, dst;

  __device__ bool put(size_t dst_off, size_t src_off, size_t bytes, unsigned long long flags,
                      unsigned long long& seq, const DevComm& dc) const {
    if (dc.skip_signal_rank == src) flags &= ~kTrigSignal;  // test knob: a lost signal
    return fifo_push(pd, ProxyTrigger{trig_fst(kTrigPut | flags, src, dst, bytes), trig_snd(dst_off, src_off)},
                     seq, dc, src);
  }
  __device__ bool signal(unsigned long long& seq, const DevComm& dc) const {
    if (dc.skip_signal_rank == src) return true;  // test knob: a lost signal
    return fifo_push(pd, ProxyTrigger{trig_fst(kTrigSignal, src, dst, 0), 0}, seq, dc, src);
  }
  // flush: every trigger this thread pushed so far has been carried out
  __device__ bool flush(const DevComm& dc) const {
    unsigned long long seq;
    if (!fifo_push(pd, ProxyTrigger{trig_fst(kTrigFlush, src, dst, 0), 0}, seq, dc, src)) return false;
    return port_spin_ge(pd.done, seq + 1, dc, src, dst);
  }
  // wait (called on the destination side of this channel's pair): one more
  // signal from `src` has arrived at `dst`
  __device__ bool wait(const DevComm& dc) const {
    unsigned long long* e = pd.expect + sem_slot(dst, src, 0);
    const unsigned long long target = *e + 1;
    if (!port_spin_ge(pd.sem + sem_slot(dst, src, 0) * kSemWords, target, dc, dst, src)) return false;
    *e = target;
    return true;
  }
};

}  // namespace dcc
