// bulk.cuh -- shared-memory pipelines fed by the bulk asynchronous copy
// engine (TMA, non-tensor cp.async.bulk) for the large-message kernels.
//
// The MemoryChannel of the MSCCL++ README ("PortChannel and MemoryChannel")
// moves data with GPU threads, and the README notes that bandwidth then takes
// a large number of them.  On sm_103a one thread can hand whole tiles to the
// copy engine instead: a get becomes a cp.async.bulk global->shared load that
// completes on an mbarrier, a put becomes a cp.async.bulk shared->global store.
// Threads only reduce shared-memory tiles; the tile a rank reduced is stored
// from the same shared-memory buffer into all N outputs.
//
// Every mbarrier wait is bounded like a channel wait: on the limit it records
// the failure in the status word, the CTA stops issuing, waits (bounded) for
// the copies it has in flight, and returns.
#pragma once
#include "collectives.cuh"

namespace dcc {

constexpr int kBulkThreads = 256;          // reducing threads per CTA
constexpr int kBulkTile = 4096;            // bytes of one rank's buffer per pipeline stage
constexpr int kBulkTileVecs = kBulkTile / 16;
constexpr int kBulkSmemBudget = 200 * 1024;
constexpr int kAgTile = 16384;             // AllGather: bytes per stage
constexpr int kAgStages = 6;

__host__ __device__ constexpr int bulk_stages(int n) {
  return kBulkSmemBudget / ((n + 1) * kBulkTile) < 2   ? 2
         : kBulkSmemBudget / ((n + 1) * kBulkTile) > 8 ? 8
                                                        : kBulkSmemBudget / ((n + 1) * kBulkTile);
}
// dynamic shared memory of k_allreduce_twoshot_bulk for n ranks (compile-time N = nt, 0 = runtime)
__host__ __device__ constexpr size_t bulk_smem_bytes(int nt, int n) {
  return 128 + (size_t)bulk_stages(nt > 0 ? nt : DCC_MAX_RANKS) * (size_t)(n + 1) * kBulkTile;
}
__host__ __device__ constexpr size_t ag_smem_bytes() { return 128 + (size_t)kAgStages * kAgTile; }

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}
// global -> shared, completes `bytes` of transaction count on `bar`
__device__ __forceinline__ void bulk_load(void* sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(sdst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}
// shared -> global, tracked by bulk groups
__device__ __forceinline__ void bulk_store(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_addr(ssrc)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kPending) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy writes to shared memory become visible to the bulk-copy (async) proxy
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bounded wait on an mbarrier phase; records a timeout in the status word.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const DevComm& dc, int rank,
                                          int blk) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (unsigned it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0 && global_timer_ns() - t0 > dc.timeout_ns) {
      atomicCAS(dc.status, 0ull, pack_status(kStatusTimeout, rank, rank, blk));
      return false;
    }
  }
}

// Sum over ranks of vector v of a stage: in[p * kBulkTileVecs + v], rank order.
template <typename T, int NT>
__device__ __forceinline__ uint4 reduce_stage(const uint4* in, int n, uint32_t v) {
  using L = Lanes<T>;
  typename L::Acc acc;
  if constexpr (NT > 0) {
    uint4 x[NT];
#pragma unroll
    for (int p = 0; p < NT; ++p) x[p] = in[p * kBulkTileVecs + v];
    L::init(acc, x[0]);
#pragma unroll
    for (int p = 1; p < NT; ++p) L::add(acc, x[p]);
  } else {
    L::init(acc, in[v]);
    for (int p = 1; p < n; ++p) L::add(acc, in[p * kBulkTileVecs + v]);
  }
  return L::pack(acc);
}

// ---------------------------------------------------------------- two-shot, bulk
// Same schedule and bits as k_allreduce_twoshot: rank r reduces shard r and
// puts it into all N outputs.  Per CTA: a ring of `ST` stages, each holding the
// N inputs' 4 KiB tiles and one 4 KiB result tile.  Thread 0 issues the N bulk
// loads of a tile onto the stage's mbarrier, all threads reduce it into the
// result tile, and thread 0 bulk-stores the result into the N outputs and
// refills the stage.  The CTA's tiles are t = blk, blk + B, ... of the shard.
template <typename T, int NT>
__global__ void __launch_bounds__(kBulkThreads, 1) k_allreduce_twoshot_bulk(DevComm dc, CollArgs a) {
  pdl_prologue();
  using L = Lanes<T>;
  using S = typename L::S;
  constexpr int ST = bulk_stages(NT > 0 ? NT : DCC_MAX_RANKS);
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  unsigned char* in_base = smem + 128;
  unsigned char* out_base = in_base + (size_t)ST * n * kBulkTile;

  const size_t nvec = a.count / L::VW;
  size_t s0, s1;
  shard_vecs(nvec, n, rank, s0, s1);
  const size_t shard_bytes = (s1 - s0) * 16, base = s0 * 16;
  const size_t ntiles = (shard_bytes + kBulkTile - 1) / kBulkTile;
  const size_t mine = ntiles > (size_t)blk ? (ntiles - (size_t)blk + B - 1) / B : 0;
  auto tile_off = [&](size_t k) { return ((size_t)blk + k * (size_t)B) * kBulkTile; };
  auto tile_bytes = [&](size_t k) {
    const size_t rest = shard_bytes - tile_off(k);
    return (uint32_t)(rest < (size_t)kBulkTile ? rest : (size_t)kBulkTile);
  };
  auto issue = [&](size_t k) {  // thread 0
    const int s = (int)(k % ST);
    const uint32_t bytes = tile_bytes(k);
    bool ok = true;  // bounds-checked build: a tile with a load outside its window loads nothing
    for (int p = 0; p < n; ++p) ok = in_bounds(dc, a, kBufSend, p, base + tile_off(k), bytes) && ok;
    mbar_arrive_expect_tx(&full[s], ok ? bytes * (uint32_t)n : 0u);
    if (ok)
      for (int p = 0; p < n; ++p)
        bulk_load(in_base + ((size_t)s * n + p) * kBulkTile,
                  static_cast<const char*>(a.send[p]) + base + tile_off(k), bytes, &full[s]);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < ST; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0)
    for (size_t k = 0; k < mine && k < (size_t)ST; ++k) issue(k);

  size_t k = 0;
  bool failed = false;
  for (; k < mine; ++k) {
    const int s = (int)(k % ST);
    const uint32_t bytes = tile_bytes(k);
    failed = !mbar_wait(&full[s], (uint32_t)((k / ST) & 1), dc, rank, blk);
    if (!failed) {
      const uint4* in = reinterpret_cast<const uint4*>(in_base + (size_t)s * n * kBulkTile);
      uint4* out = reinterpret_cast<uint4*>(out_base + (size_t)s * kBulkTile);
      for (uint32_t v = threadIdx.x; v < bytes / 16; v += kBulkThreads) out[v] = reduce_stage<T, NT>(in, n, v);
      fence_proxy_async_smem();
    }
    // the result tile written two iterations from now was stored ST tiles ago
    if (threadIdx.x == 0) bulk_wait_read<(ST >= 2 ? ST - 2 : 0)>();
    if (__syncthreads_or(failed)) break;
    if (threadIdx.x == 0) {
      const void* out = out_base + (size_t)s * kBulkTile;
      for (int p = 0; p < n; ++p)
        if (in_bounds(dc, a, kBufRecv, p, base + tile_off(k), bytes))
          bulk_store(static_cast<char*>(a.recv[p]) + base + tile_off(k), out, bytes);
      bulk_commit();
      if (k + ST < mine) issue(k + ST);
    }
  }
  if (threadIdx.x == 0) {
    if (failed)  // let the loads still in flight land before the shared memory goes away
      for (size_t j = k; j < mine && j < k + ST; ++j)
        mbar_wait(&full[j % ST], (uint32_t)((j / ST) & 1), dc, rank, blk);
    bulk_wait_all();
  }
  const size_t i = nvec * L::VW + threadIdx.x;
  if (!failed && rank == n - 1 && blk == 0 && i < a.count) {
    const S r = reduce_scalar<T>(dc, a, n, i);
    for (int p = 0; p < n; ++p) put_elem<S>(dc, a, p, i, r);
  }
}

// ---------------------------------------------------------------- AllGather, bulk
// recv[p][q*m + j] = send[q][j]: rank q's CTA loads a 16 KiB tile of its input
// into shared memory with one bulk copy and stores that same buffer into slot q
// of all N outputs with N bulk copies.  One thread drives the copy engine.
// Requires m * elem_bytes to be a multiple of 16 (host checks).
template <int NT>
__global__ void __launch_bounds__(32, 1) k_allgather_bulk(DevComm dc, CollArgs a, int elem_bytes) {
  pdl_prologue();
  if (threadIdx.x != 0) return;
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  unsigned char* stage = smem + 128;
  const size_t bytes = a.count * (size_t)elem_bytes;
  const size_t ntiles = (bytes + kAgTile - 1) / kAgTile;
  const size_t mine = ntiles > (size_t)blk ? (ntiles - (size_t)blk + B - 1) / B : 0;
  auto off = [&](size_t k) { return ((size_t)blk + k * (size_t)B) * kAgTile; };
  auto len = [&](size_t k) {
    const size_t rest = bytes - off(k);
    return (uint32_t)(rest < (size_t)kAgTile ? rest : (size_t)kAgTile);
  };
  auto issue = [&](size_t k) {
    const int s = (int)(k % kAgStages);
    const bool ok = in_bounds(dc, a, kBufSend, rank, off(k), len(k));  // bounds-checked build
    mbar_arrive_expect_tx(&full[s], ok ? len(k) : 0u);
    if (ok) bulk_load(stage + (size_t)s * kAgTile, static_cast<const char*>(a.send[rank]) + off(k), len(k), &full[s]);
  };
  for (int s = 0; s < kAgStages; ++s) mbar_init(&full[s], 1);
  fence_mbar_init();
  for (size_t k = 0; k < mine && k < (size_t)kAgStages; ++k) issue(k);
  size_t k = 0;
  bool failed = false;
  for (; k < mine; ++k) {
    const int s = (int)(k % kAgStages);
    if (!mbar_wait(&full[s], (uint32_t)((k / kAgStages) & 1), dc, rank, blk)) {
      failed = true;
      break;
    }
    for (int p = 0; p < n; ++p)
      if (in_bounds(dc, a, kBufRecv, p, (size_t)rank * bytes + off(k), len(k)))
        bulk_store(static_cast<char*>(a.recv[p]) + (size_t)rank * bytes + off(k), stage + (size_t)s * kAgTile, len(k));
    bulk_commit();
    // refill the stage of the previous tile once its stores have read it
    if (k >= 1 && k - 1 + kAgStages < mine) {
      bulk_wait_read<1>();
      issue(k - 1 + kAgStages);
    }
  }
  if (failed)
    for (size_t j = k; j < mine && j < k + kAgStages; ++j)
      mbar_wait(&full[j % kAgStages], (uint32_t)((j / kAgStages) & 1), dc, rank, blk);
  bulk_wait_all();
}

}  // namespace dcc
