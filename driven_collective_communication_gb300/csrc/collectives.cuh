// collectives.cuh -- sum AllReduce (one-shot, two-shot push, two-shot via
// scratch) and ReduceScatter kernels for N virtual ranks; the one-shot,
// two-shot push and ReduceScatter kernels also take MAX / MIN (template
// parameter OP, combiners in reduce_ops.cuh).
//
// The collectives are the standard ones of the MSCCL++ abstract, point (3);
// the AllReduce is the tensor-parallel serving case of the project summary's
// "Highlighted Details".  Every data access goes through a MemoryChannel
// (get = read of a peer's 16-byte vector, put = write into a peer's buffer);
// signal/wait order the phases that need it.
//
// Arithmetic (identical in every kernel, so every algorithm and launch shape
// returns the same bits): per element, acc = x_0; acc += x_p for p = 1..N-1 in
// rank order; fp16/bf16 are widened exactly to fp32, adds are fp32
// round-to-nearest-even (__fadd_rn, no contraction, subnormals kept: the build
// uses no fast-math and no flush-to-zero); one RNE rounding to the output type
// at the end (cvt.rn); int32 adds wrap.
//
// Layout: rank r's buffers are separate allocations; a rank is the group of
// `blocks` consecutive CTAs starting at r * blocks.  Each thread works on
// whole 16-byte vectors; the < 16-byte remainder of a buffer (the "tail") is
// done element by element by one CTA.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "memory_channel.cuh"
#include "reduce_ops.cuh"

namespace dcc {

constexpr int kThreads = 512;       // threads per CTA of the data kernels
constexpr int kInplaceUnroll = 4;   // most vectors per thread per chunk, in-place one-shot
constexpr int kInplaceLargeThreads = 256;  // threads per CTA, large in-place messages
#ifndef DCC_INPLACE_PREFETCH
#define DCC_INPLACE_PREFETCH 1
#endif
constexpr int kInplacePrefetch = DCC_INPLACE_PREFETCH;  // chunks of its slot the in-place one-shot asks L2 for ahead

// ------------------------------------------------------------- element lanes
template <typename T>
struct Lanes;

template <>
struct Lanes<int32_t> {
  static constexpr int VW = 4;  // elements per 16-byte vector
  struct Acc { uint32_t v[4]; };
  using S = int32_t;            // scalar storage
  using SAcc = uint32_t;
  __device__ static void init(Acc& a, uint4 x) { a.v[0] = x.x; a.v[1] = x.y; a.v[2] = x.z; a.v[3] = x.w; }
  __device__ static void add(Acc& a, uint4 x) { a.v[0] += x.x; a.v[1] += x.y; a.v[2] += x.z; a.v[3] += x.w; }
  __device__ static uint4 pack(const Acc& a) { return make_uint4(a.v[0], a.v[1], a.v[2], a.v[3]); }
  __device__ static SAcc sinit(S x) { return (uint32_t)x; }
  __device__ static SAcc sadd(SAcc a, S x) { return a + (uint32_t)x; }
  __device__ static S spack(SAcc a) { return (int32_t)a; }
};

template <>
struct Lanes<float> {
  static constexpr int VW = 4;
  struct Acc { float v[4]; };
  using S = float;
  using SAcc = float;
  __device__ static void init(Acc& a, uint4 x) {
    a.v[0] = __uint_as_float(x.x); a.v[1] = __uint_as_float(x.y);
    a.v[2] = __uint_as_float(x.z); a.v[3] = __uint_as_float(x.w);
  }
  __device__ static void add(Acc& a, uint4 x) {
    a.v[0] = __fadd_rn(a.v[0], __uint_as_float(x.x)); a.v[1] = __fadd_rn(a.v[1], __uint_as_float(x.y));
    a.v[2] = __fadd_rn(a.v[2], __uint_as_float(x.z)); a.v[3] = __fadd_rn(a.v[3], __uint_as_float(x.w));
  }
  __device__ static uint4 pack(const Acc& a) {
    return make_uint4(__float_as_uint(a.v[0]), __float_as_uint(a.v[1]), __float_as_uint(a.v[2]),
                      __float_as_uint(a.v[3]));
  }
  __device__ static SAcc sinit(S x) { return x; }
  __device__ static SAcc sadd(SAcc a, S x) { return __fadd_rn(a, x); }
  __device__ static S spack(SAcc a) { return a; }
};

// 16-bit floats: 8 per vector, widened pairwise (exact), narrowed pairwise RNE.
template <typename H2, typename Ops>
struct HalfLanes {
  static constexpr int VW = 8;
  struct Acc { float v[8]; };
  using S = uint16_t;  // raw storage bits
  using SAcc = float;
  __device__ static float2 widen2(uint32_t w) { return Ops::widen2(w); }
  __device__ static uint32_t narrow2(float lo, float hi) {
    H2 h = Ops::from_floats(lo, hi);
    uint32_t w;
    memcpy(&w, &h, 4);
    return w;
  }
  __device__ static void init(Acc& a, uint4 x) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 f = widen2(w[k]);
      a.v[2 * k] = f.x;
      a.v[2 * k + 1] = f.y;
    }
  }
  __device__ static void add(Acc& a, uint4 x) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 f = widen2(w[k]);
      a.v[2 * k] = __fadd_rn(a.v[2 * k], f.x);
      a.v[2 * k + 1] = __fadd_rn(a.v[2 * k + 1], f.y);
    }
  }
  __device__ static uint4 pack(const Acc& a) {
    return make_uint4(narrow2(a.v[0], a.v[1]), narrow2(a.v[2], a.v[3]), narrow2(a.v[4], a.v[5]),
                      narrow2(a.v[6], a.v[7]));
  }
  __device__ static SAcc sinit(S x) { return widen2((uint32_t)x).x; }
  __device__ static SAcc sadd(SAcc a, S x) { return __fadd_rn(a, widen2((uint32_t)x).x); }
  __device__ static S spack(SAcc a) { return (uint16_t)(narrow2(a, 0.0f) & 0xFFFFu); }
};

// bf16 is the upper half of binary32, so widening places the 16 bits there
// (two integer operations, exact for every pattern); fp16 converts.
struct Bf16Ops {
  __device__ static float2 widen2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  __device__ static __nv_bfloat162 from_floats(float lo, float hi) { return __floats2bfloat162_rn(lo, hi); }
};
struct F16Ops {
  __device__ static float2 widen2(uint32_t w) {
    __half2 h;
    memcpy(&h, &w, 4);
    return __half22float2(h);
  }
  __device__ static __half2 from_floats(float lo, float hi) { return __floats2half2_rn(lo, hi); }
};

template <>
struct Lanes<__nv_bfloat16> : HalfLanes<__nv_bfloat162, Bf16Ops> {};
template <>
struct Lanes<__half> : HalfLanes<__half2, F16Ops> {};

// ------------------------------------------------------------- reductions
// get of vector v from rank p's input (a zero vector where the bounds-checked
// build finds it outside the rank's window)
__device__ __forceinline__ uint4 get_vec(const DevComm& dc, const CollArgs& a, int p, size_t v) {
  return in_bounds(dc, a, kBufSend, p, v * 16, 16) ? ld_vec(static_cast<const uint4*>(a.send[p]) + v)
                                                   : make_uint4(0, 0, 0, 0);
}

// put of vector v into buffer KIND (kBufRecv, kBufScratch) of rank p
template <int KIND>
__device__ __forceinline__ void put_vec(const DevComm& dc, const CollArgs& a, int p, size_t v, uint4 x) {
  void* dst = KIND == kBufScratch ? a.scratch[p] : a.recv[p];
  if (in_bounds(dc, a, KIND, p, v * 16, 16)) st_vec(static_cast<uint4*>(dst) + v, x);
}

// get / put of element i (the sub-vector tail and the element paths)
template <typename S>
__device__ __forceinline__ S get_elem(const DevComm& dc, const CollArgs& a, int p, size_t i) {
  return in_bounds(dc, a, kBufSend, p, i * sizeof(S), sizeof(S)) ? static_cast<const S*>(a.send[p])[i] : S{};
}
template <typename S>
__device__ __forceinline__ void put_elem(const DevComm& dc, const CollArgs& a, int p, size_t i, S x) {
  if (in_bounds(dc, a, kBufRecv, p, i * sizeof(S), sizeof(S))) static_cast<S*>(a.recv[p])[i] = x;
}

// Sum (or, with OP, MAX / MIN: reduce_ops.cuh) of vector v over the N ranks'
// inputs a.send[0..N-1], rank order.  With a compile-time N all N gets are
// issued before the first add.
template <typename T, int NT, int OP = kOpSum>
__device__ __forceinline__ uint4 reduce_vec(const DevComm& dc, const CollArgs& a, int n, size_t v) {
  if constexpr (OP != kOpSum) return pick_ranks_vec<T, NT, OP>(dc, a, n, v);
  using L = Lanes<T>;
  typename L::Acc acc;
  if constexpr (NT > 0) {
    uint4 x[NT];
#pragma unroll
    for (int p = 0; p < NT; ++p) x[p] = get_vec(dc, a, p, v);
    L::init(acc, x[0]);
#pragma unroll
    for (int p = 1; p < NT; ++p) L::add(acc, x[p]);
  } else {
    L::init(acc, get_vec(dc, a, 0, v));
    for (int p = 1; p < n; ++p) L::add(acc, get_vec(dc, a, p, v));
  }
  return L::pack(acc);
}

template <typename T, int OP = kOpSum>
__device__ __forceinline__ typename Lanes<T>::S reduce_scalar(const DevComm& dc, const CollArgs& a, int n,
                                                             size_t i) {
  using L = Lanes<T>;
  using S = typename L::S;
  if constexpr (OP != kOpSum) return pick_ranks_scalar<T, OP, S>(dc, a, n, i);
  typename L::SAcc acc = L::sinit(get_elem<S>(dc, a, 0, i));
  for (int p = 1; p < n; ++p) acc = L::sadd(acc, get_elem<S>(dc, a, p, i));
  return L::spack(acc);
}

// Two-shot shard of rank r, in vectors: whole vectors, the last rank also
// takes the remainder (and the element tail).
__device__ __forceinline__ void shard_vecs(size_t nvec, int n, int r, size_t& s0, size_t& s1) {
  const size_t per = nvec / (size_t)n;
  s0 = per * (size_t)r;
  s1 = (r == n - 1) ? nvec : s0 + per;
}

// Optional entry barrier: before touching peer memory, every CTA tells the
// CTAs of its block slot in the other ranks that its input is ready (signal)
// and waits until all of them have said the same.  Between GPUs this is what
// makes a peer's input safe to read; on one GPU stream order already does, so
// it is off unless the caller asks for it.  The kernels take it as a template
// flag EB, so the default instances carry no trace of it; EB instances are
// launched cooperatively with at most one wave, so every CTA they wait for is
// running.
__device__ __forceinline__ bool entry_barrier(const DevComm& dc, int rank, int n, int blk) {
  if (n == 1) return true;
  unsigned long long expected = 0;
  const bool waiter = (int)threadIdx.x < n && (int)threadIdx.x != rank;
  if (waiter) expected = dc.expect[sem_slot(rank, threadIdx.x, blk)];
  const bool ok = group_barrier(dc, rank, n, blk, expected);
  if (waiter) dc.expect[sem_slot(rank, threadIdx.x, blk)] = expected;
  return ok;
}

// L2 prefetch of chunk c of rank `rank`'s input (chunk = vectors per chunk):
// a hint that returns nothing to the thread, issued for whole 16-byte vectors
// inside the buffer.
__device__ __forceinline__ void prefetch_chunk_l2(const DevComm& dc, const CollArgs& a, int rank, size_t c,
                                                  size_t chunk, size_t nvec) {
  const size_t v0 = c * chunk, nv = nvec - v0 < chunk ? nvec - v0 : chunk;
  if (!in_bounds(dc, a, kBufSend, rank, v0 * 16, nv * 16)) return;
  const char* p = static_cast<const char*>(a.send[rank]) + v0 * 16;
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"((uint32_t)(nv * 16)) : "memory");
}

// ------------------------------------------------------------- one-shot
// Every rank gets all N inputs and reduces its whole output.  Out of place no
// rank writes what another reads, so there is no synchronisation.  In place,
// rank r's output is an input of every peer: the N CTAs of a block slot
// process the same chunk together -- get and reduce into registers, signal
// "this CTA has read the chunk", and store once every peer has signalled the
// same.  The wait is split from the signal: the reduced chunk waits in shared
// memory (thread-private slots) while the next chunk's gets are in flight
// (measured on GB300 for 8 x 64 MiB int32: 0.289 ms against 0.308 with signal
// and wait back to back; holding the two chunks in registers instead took
// 0.49 ms, the extra registers costing occupancy).  The barrier keeps the N
// CTAs of a slot in step, so all N read a chunk at the same moment and the
// first reader's L2 miss holds up the other N-1; each CTA therefore asks L2
// for its own rank's part of a chunk one chunk before it gets it.
template <typename T, int NT, bool EB = false, int OP = kOpSum>
__global__ void __launch_bounds__(kThreads) k_allreduce_oneshot(DevComm dc, CollArgs a) {
  pdl_prologue();
  using L = Lanes<T>;
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  const size_t nvec = a.count / L::VW;
  const size_t tail0 = nvec * L::VW;
  using S = typename L::S;
  if constexpr (EB) {
    if (!entry_barrier(dc, rank, n, blk)) return;
  }

  if (!a.inplace) {
    const size_t stride = (size_t)B * blockDim.x;
    for (size_t v = (size_t)blk * blockDim.x + threadIdx.x; v < nvec; v += stride)
      put_vec<kBufRecv>(dc, a, rank, v, reduce_vec<T, NT, OP>(dc, a, n, v));
    if (blk == 0 && tail0 + threadIdx.x < a.count)
      put_elem<S>(dc, a, rank, tail0 + threadIdx.x, reduce_scalar<T, OP>(dc, a, n, tail0 + threadIdx.x));
    return;
  }

  unsigned long long expected = 0;
  const bool waiter = (int)threadIdx.x < n && (int)threadIdx.x != rank;
  if (waiter) expected = dc.expect[sem_slot(rank, threadIdx.x, blk)];
  // U vectors per thread per chunk: 1 for small messages (one chunk per CTA,
  // all loads of a thread in flight at once), kInplaceUnroll for large ones
  // (fewer chunks, so fewer barrier rounds).  The loop over the U vectors is
  // unrolled so all of a thread's loads of a chunk are in flight together
  // (a loop over a run-time U measured slower on GB300: 0.350 vs 0.310 ms at
  // U = 4, slower still at 8 and 16; so did a compile-time 8 in the pipelined
  // form below, 0.42-0.49 ms: its registers cost occupancy).
  const int U = a.unroll > 0 && a.unroll < kInplaceUnroll ? a.unroll : kInplaceUnroll;
  const size_t chunk = (size_t)U * blockDim.x;
  const size_t nchunks = (nvec + chunk - 1) / chunk;
  bool ok = true;
  // prefetch distance: kInplacePrefetch chunks of this slot ahead
  if (threadIdx.x == 0)
    for (int d = 0; d <= kInplacePrefetch; ++d)
      if ((size_t)blk + (size_t)d * B < nchunks) prefetch_chunk_l2(dc, a, rank, blk + (size_t)d * B, chunk, nvec);
  // Pipelined: the reduced chunk c waits in shared memory (thread-private
  // slots) for the peers' signals while the next chunk's loads are in flight.
  extern __shared__ uint4 held[];
  auto reduce_chunk = [&](size_t c, uint4* res) {
#pragma unroll
    for (int u = 0; u < kInplaceUnroll; ++u) {
      const size_t v = c * chunk + (size_t)u * blockDim.x + threadIdx.x;
      if (u < U && v < nvec) res[u] = reduce_vec<T, NT, OP>(dc, a, n, v);
    }
  };
  if ((size_t)blk < nchunks) {
    uint4 res[kInplaceUnroll];
    reduce_chunk(blk, res);
#pragma unroll
    for (int u = 0; u < kInplaceUnroll; ++u)
      if (u < U) held[u * blockDim.x + threadIdx.x] = res[u];
    group_signal(dc, rank, n, blk);
  }
  for (size_t c = blk; c < nchunks; c += B) {
    const size_t cn = c + B;
    const size_t cp = cn + (size_t)kInplacePrefetch * B;
    if (threadIdx.x == 0 && kInplacePrefetch > 0 && cp < nchunks) prefetch_chunk_l2(dc, a, rank, cp, chunk, nvec);
    uint4 res[kInplaceUnroll];
    if (cn < nchunks) reduce_chunk(cn, res);
    ok = group_wait(dc, rank, n, blk, expected);  // every peer has read chunk c
    if (!ok) break;
#pragma unroll
    for (int u = 0; u < kInplaceUnroll; ++u) {
      const size_t v = c * chunk + (size_t)u * blockDim.x + threadIdx.x;
      if (u < U && v < nvec) put_vec<kBufRecv>(dc, a, rank, v, held[u * blockDim.x + threadIdx.x]);
    }
    if (cn < nchunks) {
#pragma unroll
      for (int u = 0; u < kInplaceUnroll; ++u)
        if (u < U) held[u * blockDim.x + threadIdx.x] = res[u];
      group_signal(dc, rank, n, blk);  // this CTA has read chunk cn
    }
  }
  if (ok && blk == 0 && tail0 < a.count) {  // same on every rank: all slot-0 CTAs take part
    const size_t i = tail0 + threadIdx.x;
    S r{};
    if (i < a.count) r = reduce_scalar<T, OP>(dc, a, n, i);
    ok = group_barrier(dc, rank, n, blk, expected);
    if (ok && i < a.count) put_elem<S>(dc, a, rank, i, r);
  }
  if (waiter) dc.expect[sem_slot(rank, threadIdx.x, blk)] = expected;
}

// ------------------------------------------------------------- two-shot, push
// Rank r gets shard r of all N inputs, reduces it, and puts the result into
// shard r of all N outputs (ReduceScatter fused with a push AllGather).  Only
// rank r's CTAs touch shard r of any buffer and every thread reads all N
// values of a vector before writing it anywhere, so in place is safe without
// synchronisation.  Traffic: N*S read + N*S written in total, the minimum.
template <typename T, int NT, bool EB = false, int OP = kOpSum>
__global__ void __launch_bounds__(kThreads) k_allreduce_twoshot(DevComm dc, CollArgs a) {
  pdl_prologue();
  using L = Lanes<T>;
  using S = typename L::S;
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  const size_t nvec = a.count / L::VW;
  size_t s0, s1;
  shard_vecs(nvec, n, rank, s0, s1);
  if constexpr (EB) {
    if (!entry_barrier(dc, rank, n, blk)) return;
  }
  const size_t stride = (size_t)B * blockDim.x;
  for (size_t v = s0 + (size_t)blk * blockDim.x + threadIdx.x; v < s1; v += stride) {
    const uint4 r = reduce_vec<T, NT, OP>(dc, a, n, v);
    if constexpr (NT > 0) {
#pragma unroll
      for (int p = 0; p < NT; ++p) put_vec<kBufRecv>(dc, a, p, v, r);
    } else {
      for (int p = 0; p < n; ++p) put_vec<kBufRecv>(dc, a, p, v, r);
    }
  }
  const size_t i = nvec * L::VW + threadIdx.x;
  if (rank == n - 1 && blk == 0 && i < a.count) {
    const S r = reduce_scalar<T, OP>(dc, a, n, i);
    for (int p = 0; p < n; ++p) put_elem<S>(dc, a, p, i, r);
  }
}

// ------------------------------------------------------------- two-shot, scratch
// Phase 1: rank r reduces shard r into its own scratch.  Barrier: each CTA
// signals its N-1 peers of the same block slot and waits for theirs.  Phase 2:
// rank r gets every shard q from rank q's scratch into its output.  CTA
// (r, blk) reads exactly the scratch vectors CTA (q, blk) wrote, so the
// per-slot barrier is enough.  In place is safe: rank r overwrites shard q of
// its buffer only after CTA (q, blk) has read it.
template <typename T, int NT, bool EB = false>
__global__ void __launch_bounds__(kThreads) k_allreduce_twoshot_scratch(DevComm dc, CollArgs a) {
  using L = Lanes<T>;
  using S = typename L::S;
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  const size_t nvec = a.count / L::VW;
  const size_t stride = (size_t)B * blockDim.x;
  const size_t first = (size_t)blk * blockDim.x + threadIdx.x;
  const size_t tail_i = nvec * L::VW + threadIdx.x;
  const bool tail_thread = blk == 0 && tail_i < a.count;

  size_t s0, s1;
  shard_vecs(nvec, n, rank, s0, s1);
  if constexpr (EB) {
    if (!entry_barrier(dc, rank, n, blk)) return;
  }
  uint4* mine = static_cast<uint4*>(a.scratch[rank]);
  for (size_t v = s0 + first; v < s1; v += stride) put_vec<kBufScratch>(dc, a, rank, v - s0, reduce_vec<T, NT>(dc, a, n, v));
  if (rank == n - 1 && tail_thread) {
    const S r = reduce_scalar<T>(dc, a, n, tail_i);
    if (in_bounds(dc, a, kBufScratch, rank, (s1 - s0) * 16 + threadIdx.x * sizeof(S), sizeof(S)))
      reinterpret_cast<S*>(mine + (s1 - s0))[threadIdx.x] = r;
  }

  unsigned long long expected = 0;
  const bool waiter = (int)threadIdx.x < n && (int)threadIdx.x != rank;
  if (waiter) expected = dc.expect[sem_slot(rank, threadIdx.x, blk)];
  const bool ok = group_barrier(dc, rank, n, blk, expected);
  if (waiter) dc.expect[sem_slot(rank, threadIdx.x, blk)] = expected;
  if (!ok) return;

  for (int q = 0; q < n; ++q) {
    size_t q0, q1;
    shard_vecs(nvec, n, q, q0, q1);
    MemoryChannel ch = MemoryChannel::make(dc, rank, q, blk, a.scratch[q], nullptr);
    for (size_t v = q0 + first; v < q1; v += stride) {
      const uint4 x = in_bounds(dc, a, kBufScratch, q, (v - q0) * 16, 16)
                          ? ld_vec_l2(reinterpret_cast<const uint4*>(ch.remote_src) + (v - q0))
                          : make_uint4(0, 0, 0, 0);
      put_vec<kBufRecv>(dc, a, rank, v, x);
    }
    if (q == n - 1 && tail_thread) {
      const size_t off = (q1 - q0) * 16 + threadIdx.x * sizeof(S);
      const S x = in_bounds(dc, a, kBufScratch, q, off, sizeof(S))
                      ? __ldcg(reinterpret_cast<const S*>(ch.remote_src + off))
                      : S{};
      put_elem<S>(dc, a, rank, tail_i, x);
    }
  }
}

// ------------------------------------------------------------- ReduceScatter
// recv[r][j] = sum_p send[p][r*m + j].  Rank r's CTAs get shard r of every
// input.  Vector path when a shard starts on a 16-byte boundary, else scalar.
template <typename T, int NT, bool EB = false, int OP = kOpSum>
__global__ void __launch_bounds__(kThreads) k_reduce_scatter(DevComm dc, CollArgs a) {
  pdl_prologue();
  using L = Lanes<T>;
  using S = typename L::S;
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  if constexpr (EB) {
    if (!entry_barrier(dc, rank, n, blk)) return;
  }
  const size_t m = a.count;
  const size_t stride = (size_t)B * blockDim.x;
  const size_t first = (size_t)blk * blockDim.x + threadIdx.x;
  if ((m * sizeof(S)) % 16 == 0) {
    const size_t nv = m / L::VW, base = (size_t)rank * nv;
    for (size_t v = first; v < nv; v += stride) put_vec<kBufRecv>(dc, a, rank, v, reduce_vec<T, NT, OP>(dc, a, n, base + v));
  } else {
    const size_t base = (size_t)rank * m;
    for (size_t j = first; j < m; j += stride) put_elem<S>(dc, a, rank, j, reduce_scalar<T, OP>(dc, a, n, base + j));
  }
}

// ------------------------------------------------------------- kernel tables
enum KernelKind {
  kOneShot = 0, kTwoShot = 1, kTwoShotScratch = 2, kReduceScatter = 3, kTwoShotBulk = 4, kOneShotLL = 5,
  // the same kernels with the entry barrier
  kOneShotEB = 6, kTwoShotEB = 7, kTwoShotScratchEB = 8, kReduceScatterEB = 9,
  kNumKernelKinds = 10
};

// Kernel of `kind` for element type T and n ranks (compile-time N for
// 1..8 and 16, a runtime-N instance otherwise).
template <typename T>
const void* reduce_kernel(int kind, int n);

// MAX / MIN kernels (OP = kOpMax or kOpMin) of kind kOneShot, kTwoShot or
// kReduceScatter (compile-time N for 2, 4, 8 and 16 ranks, a runtime-N
// instance otherwise) and of the matching entry-barrier kinds (runtime-N
// instances only); nullptr for other kinds.
template <typename T, int OP>
const void* reduce_op_kernel(int kind, int n);


}  // namespace dcc
