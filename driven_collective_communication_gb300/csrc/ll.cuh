// ll.cuh -- one-shot AllReduce with a low-latency (LL) packet protocol.
//
// The MSCCL++ README ("PortChannel and MemoryChannel") presents the
// MemoryChannel as the channel for latency-sensitive transfers; the project
// summary ("How It Works") adds custom collectives that cannot deadlock.  LL takes the synchronisation out of a separate signal/wait
// round trip and puts it into the data: every 8-byte half of a 16-byte packet
// holds 4 bytes of payload and a 4-byte flag, written with one 16-byte store
// of two 8-byte elements, and a reader accepts a packet only when both flags
// carry the current epoch.
// Packets are written and polled with relaxed GPU-scope accesses: only GPU
// threads read them, and on GB300 (whose host CPU may cache GPU memory
// coherently) the system-scope volatile forms measured 4.6 us per 16 KiB
// AllReduce against 3.8 us (3.4 us once missing packets are re-polled in one
// round rather than peer by peer, with 8-byte-element accesses).
//
// Rank r first publishes its input as packets into its own LL buffer (a
// library-owned allocation, so no caller data can look like a flag), then gets
// every rank's packets for its vectors, spinning (bounded) on the flags, and
// reduces in rank order into its output.  No rank ever reads another rank's
// data buffer, so in place needs no barrier at all.
//
// Epochs: one 32-bit counter per (rank, CTA slot) in device memory, advanced
// by one per call (graph replays included).  The launch shape is fixed
// (kLLBlocks CTAs x kLLThreads threads per rank), so a packet position is
// always written and read by the same slot, whose counters advance in step on
// every rank: a stale packet always carries an older epoch.  The buffer starts
// zeroed and epochs start at 1.
#pragma once
#include "collectives.cuh"

namespace dcc {

constexpr int kLLThreads = 128;
constexpr int kLLBlocks = 16;                       // CTAs per rank, fixed
constexpr size_t kLLMaxBytes = 256 * 1024;          // largest message per rank
constexpr size_t kLLBufBytes = 2 * kLLMaxBytes + 64;  // packets of one rank (+ the tail vector)

// A packet half is one naturally aligned 8-byte element {payload, flag}: the
// PTX memory model makes each such element's store and load indivisible, so a
// reader that sees the current flag in a half also sees that half's payload.
__device__ __forceinline__ void st_ll(uint4* p, uint32_t d0, uint32_t d1, uint32_t flag) {
  const unsigned long long a = ((unsigned long long)flag << 32) | d0, b = ((unsigned long long)flag << 32) | d1;
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

// One packet as {payload0, flag0, payload1, flag1}.
__device__ __forceinline__ uint4 ld_pk(const uint4* p) {
  unsigned long long a, b;
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
  return make_uint4((uint32_t)a, (uint32_t)(a >> 32), (uint32_t)b, (uint32_t)(b >> 32));
}

__device__ __forceinline__ bool ld_ll(const uint4* p, uint32_t flag, uint32_t& d0, uint32_t& d1) {
  const uint4 v = ld_pk(p);
  d0 = v.x;
  d1 = v.z;
  return v.y == flag && v.w == flag;
}

// Bounded poll of one 16-byte payload (two packets) of peer `peer`.
__device__ __forceinline__ bool ll_get(const uint4* pk, uint32_t flag, uint4& x, const DevComm& dc, int rank,
                                       int peer, int blk) {
  uint32_t a, b, c, d;
  bool lo = ld_ll(pk, flag, a, b), hi = ld_ll(pk + 1, flag, c, d);
  if (lo && hi) {
    x = make_uint4(a, b, c, d);
    return true;
  }
  const unsigned long long t0 = global_timer_ns();
  for (unsigned it = 1;; ++it) {
    if (!lo) lo = ld_ll(pk, flag, a, b);
    if (!hi) hi = ld_ll(pk + 1, flag, c, d);
    if (lo && hi) {
      x = make_uint4(a, b, c, d);
      return true;
    }
    if ((it & 31u) == 0) {
      if (ld_relaxed_gpu(dc.status) != 0ull) return false;
      if (global_timer_ns() - t0 > dc.timeout_ns) {
        atomicCAS(dc.status, 0ull, pack_status(kStatusTimeout, rank, peer, blk));
        return false;
      }
    }
  }
}

// Reduce vector v in rank order: every peer's payload from its LL buffer, mine
// from `own`.  With a compile-time N all 2(N-1) packet loads are issued before
// any flag is examined, then only the packets still carrying an old epoch are
// polled again (bounded).
template <typename T, int NT>
__device__ __forceinline__ bool ll_reduce(const DevComm& dc, int n, int rank, int blk, size_t v,
                                          uint32_t flag, uint4 own, uint4& out) {
  using L = Lanes<T>;
  typename L::Acc acc;
  if constexpr (NT > 0) {
    uint4 lo[NT], hi[NT];
    unsigned missing = 0;
#pragma unroll
    for (int p = 0; p < NT; ++p) {
      if (p == rank) continue;
      const uint4* pk = reinterpret_cast<const uint4*>(dc.ll_buf + (size_t)p * kLLBufBytes) + 2 * v;
      lo[p] = ld_pk(pk);
      hi[p] = ld_pk(pk + 1);
    }
#pragma unroll
    for (int p = 0; p < NT; ++p)
      if (p != rank && !(lo[p].y == flag && lo[p].w == flag && hi[p].y == flag && hi[p].w == flag))
        missing |= 1u << p;
    if (missing) {
      // re-poll: issue the loads of every packet still missing, then examine
      // them, so one round costs one L2 round trip however many are missing
      const unsigned long long t0 = global_timer_ns();
      for (unsigned it = 1; missing; ++it) {
#pragma unroll
        for (int p = 0; p < NT; ++p) {
          if (!(missing & (1u << p))) continue;
          const uint4* pk = reinterpret_cast<const uint4*>(dc.ll_buf + (size_t)p * kLLBufBytes) + 2 * v;
          lo[p] = ld_pk(pk);
          hi[p] = ld_pk(pk + 1);
        }
#pragma unroll
        for (int p = 0; p < NT; ++p)
          if ((missing & (1u << p)) && lo[p].y == flag && lo[p].w == flag && hi[p].y == flag && hi[p].w == flag)
            missing &= ~(1u << p);
        if (missing && (it & 31u) == 0) {
          if (ld_relaxed_gpu(dc.status) != 0ull) return false;
          if (global_timer_ns() - t0 > dc.timeout_ns) {
            atomicCAS(dc.status, 0ull, pack_status(kStatusTimeout, rank, __ffs(missing) - 1, blk));
            return false;
          }
        }
      }
    }
#pragma unroll
    for (int p = 0; p < NT; ++p) {
      const uint4 xp = p == rank ? own : make_uint4(lo[p].x, lo[p].z, hi[p].x, hi[p].z);
      if (p == 0) L::init(acc, xp); else L::add(acc, xp);
    }
  } else {
    for (int p = 0; p < n; ++p) {
      uint4 x = own;
      if (p != rank) {
        const uint4* pk = reinterpret_cast<const uint4*>(dc.ll_buf + (size_t)p * kLLBufBytes) + 2 * v;
        if (!ll_get(pk, flag, x, dc, rank, p, blk)) return false;
      }
      if (p == 0) L::init(acc, x); else L::add(acc, x);
    }
  }
  out = L::pack(acc);
  return true;
}

// The element tail (< one vector) travels as one zero-padded vector at index nvec.
template <typename T>
__device__ __forceinline__ uint4 load_padded(const DevComm& dc, const CollArgs& a, int rank, size_t nvec) {
  using S = typename Lanes<T>::S;
  S e[16 / sizeof(S)] = {};
  for (size_t i = nvec * Lanes<T>::VW, k = 0; i < a.count; ++i, ++k) e[k] = get_elem<S>(dc, a, rank, i);
  uint4 x;
  memcpy(&x, e, 16);
  return x;
}

template <typename T, int NT>
__global__ void __launch_bounds__(kLLThreads) k_allreduce_oneshot_ll(DevComm dc, CollArgs a) {
  using L = Lanes<T>;
  using S = typename L::S;
  const int n = NT > 0 ? NT : dc.n;
  const int rank = blockIdx.x / kLLBlocks, blk = blockIdx.x % kLLBlocks;
  // every thread reads the slot's epoch itself (one broadcast load, issued
  // alongside its first data load) so publishing waits for no barrier
  unsigned long long* epoch = dc.ll_epoch + (size_t)rank * DCC_MAX_BLOCKS_PER_RANK + blk;
  const uint32_t flag = (uint32_t)(*epoch + 1ull);
  const size_t nvec = a.count / L::VW;
  const size_t nv = nvec + (a.count % L::VW ? 1 : 0);
  const size_t first = (size_t)blk * kLLThreads + threadIdx.x, stride = (size_t)kLLBlocks * kLLThreads;
  uint4* mine = reinterpret_cast<uint4*>(dc.ll_buf + (size_t)rank * kLLBufBytes);

  // publish: my input as packets (the owner of index nvec also publishes the padded tail)
  for (size_t v = first; v < nvec; v += stride) {
    const uint4 x = get_vec(dc, a, rank, v);
    st_ll(mine + 2 * v, x.x, x.y, flag);
    st_ll(mine + 2 * v + 1, x.z, x.w, flag);
  }
  const bool tail_owner = nv > nvec && (nvec % stride) == first;
  if (tail_owner) {
    const uint4 x = load_padded<T>(dc, a, rank, nvec);
    st_ll(mine + 2 * nvec, x.x, x.y, flag);
    st_ll(mine + 2 * nvec + 1, x.z, x.w, flag);
  }
  // gather and reduce in rank order; my own vector comes from my input
  bool ok = true;
  for (size_t v = first; v < nvec && ok; v += stride) {
    uint4 r;
    ok = ll_reduce<T, NT>(dc, n, rank, blk, v, flag, get_vec(dc, a, rank, v), r);
    if (ok) put_vec<kBufRecv>(dc, a, rank, v, r);
  }
  if (ok && tail_owner) {
    uint4 r;
    ok = ll_reduce<T, NT>(dc, n, rank, blk, nvec, flag, load_padded<T>(dc, a, rank, nvec), r);
    if (ok) {
      S e[16 / sizeof(S)];
      memcpy(e, &r, 16);
      for (size_t i = nvec * L::VW, k = 0; i < a.count; ++i, ++k) put_elem<S>(dc, a, rank, i, e[k]);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *epoch = flag;
}

}  // namespace dcc
