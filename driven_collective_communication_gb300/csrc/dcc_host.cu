// dcc_host.cu -- host side of libdcc: communicator, buffer registration,
// channel table, argument checks, algorithm choice and kernel launches.
//
// The MSCCL++ README ("Host-Side Communication Proxy") sets up a bootstrap, a
// Communicator and the connections on the host, then launches kernels; the
// "Channels" section builds channels on the host and copies them to the GPU.
// Here one process owns all N virtual ranks of one GPU, so the bootstrap
// collapses into dcc_comm_create and a "connection" is a channel-table entry.
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "allgather.cuh"
#include "bulk.cuh"
#include "ll.cuh"
#include "collectives.cuh"
#include "comm.h"
#include "fused.cuh"
#include "fused_bulk.cuh"
#include "fused_mma.cuh"
#include "sync_kernels.cuh"

namespace {

using namespace dcc_host;

int check_channels_all_pairs(const dcc_comm* c) {
  for (int r = 0; r < c->n; ++r)
    for (int p = 0; p < c->n; ++p)
      if (r != p && !c->chan[r][p]) return DCC_ERR_NO_CHANNEL;
  return DCC_OK;
}

void shard_of(size_t count, int n, int rank, size_t eb, size_t* b, size_t* e) {
  const size_t vw = 16 / eb;
  const size_t nvec = count / vw;
  const size_t per = nvec / (size_t)n;
  *b = per * (size_t)rank * vw;
  *e = (rank == n - 1) ? count : per * (size_t)(rank + 1) * vw;
}

int upload_table(dcc_comm* c, cudaStream_t s) {
  if (!c->table_dirty) return DCC_OK;
  for (int a = 0; a < c->n; ++a) {
    for (int b = 0; b < c->n; ++b) {
      dcc::DevChannel& d = c->h_table[a * DCC_MAX_RANKS + b];
      std::memset(&d, 0, sizeof d);
      if (!c->chan[a][b]) continue;
      d.connected = 1;
      auto first = [&](int rank, int kind, char** p, size_t* bytes) {
        if (!c->win[rank][kind].empty()) {
          *p = c->win[rank][kind][0].ptr;
          *bytes = c->win[rank][kind][0].bytes;
        }
      };
      first(a, DCC_BUF_INPUT, &d.local_in, &d.local_in_bytes);
      first(a, DCC_BUF_OUTPUT, &d.local_out, &d.local_out_bytes);
      first(b, DCC_BUF_INPUT, &d.remote_in, &d.remote_in_bytes);
      first(b, DCC_BUF_OUTPUT, &d.remote_out, &d.remote_out_bytes);
    }
  }
  if (cudaMemcpyAsync(c->d_table, c->h_table, sizeof(c->h_table), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return DCC_ERR_CUDA;
  // the host copy must not change before the transfer has read it
  if (cudaStreamSynchronize(s) != cudaSuccess) return DCC_ERR_CUDA;
  c->table_dirty = false;
  return DCC_OK;
}

const void* reduce_kernel_for(dcc_dtype_t t, int kind, int n) {
  switch (t) {
    case DCC_INT32: return dcc::reduce_kernel<int32_t>(kind, n);
    case DCC_FP32: return dcc::reduce_kernel<float>(kind, n);
    case DCC_FP16: return dcc::reduce_kernel<__half>(kind, n);
    case DCC_BF16: return dcc::reduce_kernel<__nv_bfloat16>(kind, n);
    default: return nullptr;
  }
}

template <typename T>
const void* op_kernel_of(bool mx, int kind, int n) {
  return mx ? dcc::reduce_op_kernel<T, dcc::kOpMax>(kind, n) : dcc::reduce_op_kernel<T, dcc::kOpMin>(kind, n);
}

// Kernel of `kind` for reduction op (DCC_OP_SUM / MAX / MIN); MAX and MIN
// exist for the one-shot, two-shot push and ReduceScatter kinds only.
const void* op_kernel_for(dcc_dtype_t t, int op, int kind, int n) {
  if (op == DCC_OP_SUM) return reduce_kernel_for(t, kind, n);
  const bool mx = op == DCC_OP_MAX;
  if (!mx && op != DCC_OP_MIN) return nullptr;
  switch (t) {
    case DCC_INT32: return op_kernel_of<int32_t>(mx, kind, n);
    case DCC_FP32: return op_kernel_of<float>(mx, kind, n);
    case DCC_FP16: return op_kernel_of<__half>(mx, kind, n);
    case DCC_BF16: return op_kernel_of<__nv_bfloat16>(mx, kind, n);
    default: return nullptr;
  }
}

// CTAs per rank.  A kernel whose CTAs wait on one another, or rely on running
// together (one_wave), gets at most one co-resident wave and at most
// DCC_MAX_BLOCKS_PER_RANK (its semaphore slots).  A streaming kernel that
// never waits covers its work with as many CTAs as it takes and lets the block
// scheduler refill the SMs: on GB300 the 8 x 256 MiB bf16 two-shot moves
// 6.36 TB/s with one wave of 304 CTAs and 7.0 TB/s with one 16-byte vector
// per thread (neighbouring CTAs then stream neighbouring DRAM pages).
int pick_blocks(const dcc_comm* c, const void* fn, int threads, size_t work_vecs_per_rank,
                int* blocks, size_t smem = 0, size_t work_per_block = 0, bool one_wave = true) {
  const int per_sm = max_active_per_sm(fn, threads, smem);
  if (per_sm < 1) return DCC_ERR_LAUNCH;
  size_t bmax;
  if (one_wave) {
    bmax = (size_t)per_sm * c->num_sms / c->n;
    if (bmax < 1) return DCC_ERR_LAUNCH;
    if (bmax > DCC_MAX_BLOCKS_PER_RANK) bmax = DCC_MAX_BLOCKS_PER_RANK;
  } else {
    bmax = ((size_t)1 << 24) / (size_t)c->n;  // grid well inside the 2^31 - 1 limit
  }
  const size_t unit = work_per_block ? work_per_block : (size_t)threads;
  size_t want = c->blocks_override > 0 ? (size_t)c->blocks_override
                                       : (work_vecs_per_rank + unit - 1) / unit;
  if (want < 1) want = 1;
  *blocks = (int)(want > bmax ? bmax : want);
  return DCC_OK;
}

// AUTO: in place, the two-shot push needs no synchronisation while one-shot
// must wait for every peer to read a chunk before overwriting it (measured on
// GB300 at 16 KiB x 8 ranks: 1.5 us vs 4.8 us), so in-place requests always go
// two-shot; out of place, one-shot up to the per-dtype threshold.
dcc_algo_t resolve_algo(const dcc_comm* c, size_t count, dcc_dtype_t t, dcc_algo_t a,
                        bool inplace = false) {
  if (a != DCC_ALGO_AUTO) return a;
  if (c->forced_algo > 0) return (dcc_algo_t)c->forced_algo;
  if (count * elem_bytes(t) >= c->bulk_min_bytes) return c->large_algo;
  if (inplace) return DCC_ALGO_TWO_SHOT;
  return count * elem_bytes(t) <= c->one_shot_max[t] ? DCC_ALGO_ONE_SHOT : DCC_ALGO_TWO_SHOT;
}

dcc::DevComm dev_view(const dcc_comm* c) { return c->dev; }

// Device address of host memory the GPU can reach directly (pinned and mapped
// into the device's address space); false for anything else.
bool device_address(const void* p, size_t bytes, void** dptr) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer || !at.hostPointer) return false;
  // the whole range must lie in the same allocation; the runtime maps pinned
  // allocations contiguously, so checking the last byte is enough
  cudaPointerAttributes end;
  if (bytes && (cudaPointerGetAttributes(&end, static_cast<const char*>(p) + bytes - 1) != cudaSuccess ||
                end.type != cudaMemoryTypeHost)) {
    cudaGetLastError();
    return false;
  }
  *dptr = at.devicePointer;
  return true;
}

struct Shape {
  const void* fn;
  int blocks;
  int threads;
  bool cooperative;
  size_t smem;
  int unroll = 0;  // in-place one-shot: vectors per thread per chunk
};

// The compile-time rank count a kernel table holds for n (0 = runtime-N instance).
int compiled_n(int n) { return (n >= 1 && n <= 8) || n == 16 ? n : 0; }

int allreduce_shape(const dcc_comm* c, size_t count, dcc_dtype_t t, dcc_algo_t algo, bool inplace,
                    Shape* sh, int op = DCC_OP_SUM) {
  if (op != DCC_OP_SUM && algo != DCC_ALGO_ONE_SHOT && algo != DCC_ALGO_TWO_SHOT) return DCC_ERR_UNSUPPORTED;
  const size_t vw = 16 / elem_bytes(t);
  const size_t nvec = count / vw;
  int kind;
  size_t work;
  const bool eb = c->entry_barrier;  // instances with the entry barrier
  switch (algo) {
    case DCC_ALGO_ONE_SHOT: kind = eb ? dcc::kOneShotEB : dcc::kOneShot; work = nvec; break;
    case DCC_ALGO_TWO_SHOT: kind = eb ? dcc::kTwoShotEB : dcc::kTwoShot; work = nvec / c->n + 1; break;
    case DCC_ALGO_TWO_SHOT_SCRATCH:
      kind = eb ? dcc::kTwoShotScratchEB : dcc::kTwoShotScratch;
      work = nvec / c->n + 1;
      break;
    case DCC_ALGO_TWO_SHOT_BULK: kind = dcc::kTwoShotBulk; work = nvec / c->n + 1; break;
    case DCC_ALGO_ONE_SHOT_LL: kind = dcc::kOneShotLL; work = nvec; break;
    default: return DCC_ERR_INVALID_ARG;
  }
  sh->fn = op_kernel_for(t, op, kind, c->n);
  if (!sh->fn) return DCC_ERR_INVALID_ARG;
  sh->smem = 0;
  // the entry barrier is built into the thread-copy kernels only
  if (c->entry_barrier && (algo == DCC_ALGO_ONE_SHOT_LL || algo == DCC_ALGO_TWO_SHOT_BULK))
    return DCC_ERR_UNSUPPORTED;
  if (algo == DCC_ALGO_ONE_SHOT_LL) {  // fixed launch shape (see ll.cuh)
    if (count * elem_bytes(t) > dcc::kLLMaxBytes) return DCC_ERR_UNSUPPORTED;
    sh->threads = dcc::kLLThreads;
    sh->blocks = dcc::kLLBlocks;
    sh->cooperative = c->n > 1;
    const int per_sm = max_active_per_sm(sh->fn, sh->threads);
    if (per_sm < 1 || per_sm * c->num_sms < dcc::kLLBlocks * c->n) return DCC_ERR_LAUNCH;
    return DCC_OK;
  }
  if (algo == DCC_ALGO_TWO_SHOT_BULK) {
    sh->threads = dcc::kBulkThreads;
    sh->cooperative = false;
    sh->smem = dcc::bulk_smem_bytes(compiled_n(c->n), c->n);
    return pick_blocks(c, sh->fn, sh->threads, work, &sh->blocks, sh->smem, dcc::kBulkTileVecs);
  }
  sh->threads = c->threads_override > 0 ? c->threads_override : threads_for(algo, work);
  sh->cooperative = (algo == DCC_ALGO_ONE_SHOT && inplace && c->n > 1) ||
                    (algo == DCC_ALGO_TWO_SHOT_SCRATCH && c->n > 1) || (c->entry_barrier && c->n > 1);
  if (algo == DCC_ALGO_ONE_SHOT && inplace) {
    // one vector per thread while one chunk per CTA of the co-resident grid
    // covers the message (a single barrier round, every load in flight at
    // once), else kInplaceUnroll vectors per thread in 256-thread CTAs (fewer
    // barrier rounds: measured on GB300 at 8 x 64 MiB int32, 0.289 ms against
    // 0.306 with 512-thread CTAs, 0.320 with 128 and 0.342 with two vectors)
    if (c->threads_override <= 0 && work > 65536) sh->threads = dcc::kInplaceLargeThreads;
    sh->unroll = c->inplace_unroll;
    if (sh->unroll <= 0) {
      int b1 = 0;
      const int rc = pick_blocks(c, sh->fn, sh->threads, nvec, &b1, 0, 0, true);
      if (rc != DCC_OK) return rc;
      sh->unroll = (size_t)b1 * sh->threads >= nvec ? 1 : dcc::kInplaceUnroll;
    }
    work = (nvec + sh->unroll - 1) / sh->unroll;
    sh->smem = (size_t)dcc::kInplaceUnroll * sh->threads * 16;  // the chunk held while the signals travel
  }
  // one-shot keeps one wave even out of place: every rank reads every input,
  // and the ranks' CTAs reading a region together is what lets L2 serve it
  const bool one_wave = sh->cooperative || algo == DCC_ALGO_ONE_SHOT;
  return pick_blocks(c, sh->fn, sh->threads, work, &sh->blocks, sh->smem, 0, one_wave);
}

int run_allreduce(dcc_comm* c, void* const* send, void* const* recv, size_t count, dcc_dtype_t t,
                  dcc_algo_t algo, bool inplace, cudaStream_t s, int op = DCC_OP_SUM);

// MAX / MIN run on the one-shot and two-shot push kernels: AUTO keeps the
// size-based choice between those two and takes two-shot where it would pick
// another schedule; an explicit other schedule is unsupported.
dcc_algo_t resolve_op_algo(const dcc_comm* c, size_t count, dcc_dtype_t t, dcc_algo_t a, bool inplace,
                           int op) {
  const dcc_algo_t r = resolve_algo(c, count, t, a, inplace);
  if (op == DCC_OP_SUM || a != DCC_ALGO_AUTO || r == DCC_ALGO_ONE_SHOT) return r;
  return DCC_ALGO_TWO_SHOT;
}

int allreduce_launch(dcc_comm* c, void* const* send, void* const* recv, size_t count,
                     dcc_dtype_t t, dcc_algo_t a, cudaStream_t s, int op = DCC_OP_SUM) {
  if (c->sticky != DCC_OK) return c->sticky;
  if (elem_bytes(t) == 0) return DCC_ERR_INVALID_ARG;
  if (op != DCC_OP_SUM && op != DCC_OP_MAX && op != DCC_OP_MIN) return DCC_ERR_INVALID_ARG;
  if (a < DCC_ALGO_AUTO || a > DCC_ALGO_ONE_SHOT_LL) return DCC_ERR_INVALID_ARG;
  if (count == 0) return DCC_OK;
  const size_t bytes = count * elem_bytes(t);
  if (bytes / elem_bytes(t) != count) return DCC_ERR_INVALID_ARG;
  bool inplace = false;
  int rc = check_buffers(c, send, bytes, recv, bytes, true, &inplace);
  if (rc != DCC_OK) return rc;
  rc = check_channels_all_pairs(c);
  if (rc != DCC_OK) return rc;
  return run_allreduce(c, send, recv, count, t, resolve_op_algo(c, count, t, a, inplace, op), inplace, s, op);
}

// Builds the arguments and launches an AllReduce whose buffers are already
// checked (pointers, alignment, overlaps, channels).
int run_allreduce(dcc_comm* c, void* const* send, void* const* recv, size_t count, dcc_dtype_t t,
                  dcc_algo_t algo, bool inplace, cudaStream_t s, int op) {
  const size_t bytes = count * elem_bytes(t);
  int rc;
  dcc::CollArgs args{};
  for (int r = 0; r < c->n; ++r) {
    args.send[r] = send[r];
    args.recv[r] = recv[r];
  }
  args.count = count;
  args.inplace = inplace ? 1 : 0;
  for (int r = 0; r < c->n; ++r) {
    set_extent(args, dcc::kBufSend, r, bytes);
    set_extent(args, dcc::kBufRecv, r, bytes);
  }
  if (algo == DCC_ALGO_TWO_SHOT_SCRATCH) {
    for (int r = 0; r < c->n; ++r) {
      size_t b, e;
      shard_of(count, c->n, r, elem_bytes(t), &b, &e);
      const size_t need = (e - b) * elem_bytes(t);
      if (c->win[r][DCC_BUF_SCRATCH].empty()) return DCC_ERR_NOT_REGISTERED;
      const Window& w = c->win[r][DCC_BUF_SCRATCH][0];
      if (w.bytes < need) return DCC_ERR_NOT_REGISTERED;
      for (int p = 0; p < c->n; ++p)
        if (overlaps(w.ptr, need, send[p], bytes) || overlaps(w.ptr, need, recv[p], bytes))
          return DCC_ERR_INVALID_ARG;
      args.scratch[r] = w.ptr;
      set_extent(args, dcc::kBufScratch, r, need);
    }
  }
  Shape sh;
  rc = allreduce_shape(c, count, t, algo, inplace, &sh, op);
  if (rc != DCC_OK) return rc;
  args.blocks = sh.blocks;
  args.unroll = sh.unroll;
  if (c->log)
    std::fprintf(stderr, "dcc_allreduce: n=%d count=%zu dtype=%d op=%d algo=%d inplace=%d blocks/rank=%d\n",
                 c->n, count, (int)t, op, (int)algo, (int)inplace, sh.blocks);
  dcc::DevComm dc = dev_view(c);
  void* kargs[] = {&dc, &args};
  // programmatic dependent launch for the schedules whose CTAs never wait on
  // one another (out-of-place one-shot, two-shot push, bulk two-shot)
  const bool pdl = c->pdl && !sh.cooperative &&
                   (algo == DCC_ALGO_ONE_SHOT || algo == DCC_ALGO_TWO_SHOT || algo == DCC_ALGO_TWO_SHOT_BULK);
  return launch(sh.fn, sh.blocks * c->n, sh.threads, sh.cooperative, kargs, s, sh.smem, pdl);
}

}  // namespace

namespace {

// Calls visit(fn) for every kernel of the library's collectives, fused layer
// and MemoryChannel primitives; stops at the first false.
template <typename F>
bool visit_kernels(F&& visit) {
  const dcc_dtype_t types[] = {DCC_INT32, DCC_FP32, DCC_FP16, DCC_BF16};
  const int ns[] = {1, 2, 3, 4, 5, 6, 7, 8, 16, 9};  // 9: the runtime-N instances
  auto v = [&](const void* fn) { return !fn || visit(fn); };
  for (dcc_dtype_t t : types)
    for (int n : ns)
      for (int kind = 0; kind < dcc::kNumKernelKinds; ++kind)
        if (!v(reduce_kernel_for(t, kind, n)) || !v(op_kernel_for(t, DCC_OP_MAX, kind, n)) ||
            !v(op_kernel_for(t, DCC_OP_MIN, kind, n)))
          return false;
  for (int n : ns)
    if (!v(dcc::allgather_kernel(n, false)) || !v(dcc::allgather_kernel(n, true)) ||
        !v(dcc::allgather_bulk_kernel(n)) || !v(dcc::linear_allreduce_kernel<__nv_bfloat16>(n)) ||
        !v(dcc::linear_allreduce_kernel<__half>(n)) || !v(dcc::linear_allreduce_bulk_kernel<__nv_bfloat16>(n)) ||
        !v(dcc::linear_allreduce_bulk_kernel<__half>(n)) ||
        !v(dcc::linear_allreduce_mma_kernel(n, 1, dcc::kMmaPairThreads, false)) ||
        !v(dcc::linear_allreduce_mma_kernel(n, 1, dcc::kMmaThreads, false)) ||
        !v(dcc::linear_allreduce_mma_kernel(n, 2, dcc::kMmaThreads, false)) ||
        !v(dcc::linear_allreduce_mma_kernel(n, 1, dcc::kMmaPairThreads, true)) ||
        !v(dcc::linear_allreduce_mma_kernel(n, 1, dcc::kMmaThreads, true)) ||
        !v(dcc::linear_allreduce_mma_kernel(n, 2, dcc::kMmaThreads, true)))
      return false;
  return v(dcc::ring_barrier_kernel()) && v(dcc::ring_barrier_cluster_kernel()) && v(dcc::channel_put_kernel()) &&
         v(dcc::channel_get_kernel());
}

}  // namespace

// Loads every collective kernel of the library into the current context now
// rather than at its first launch.  With lazy module loading, loading a kernel
// waits for the kernels already running; if one of those waits on the host
// proxy, the proxy's CUDA calls stall behind the load until that kernel's wait
// limit runs out.  Preloading before the proxy starts removes the hazard for
// this library's own kernels.
int dcc_preload_kernels() {
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  cudaFuncAttributes attr;
  const bool ok = visit_kernels([&](const void* fn) {
    if (cudaFuncGetAttributes(&attr, fn) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    return true;
  });
  return ok ? DCC_OK : DCC_ERR_CUDA;
}

namespace {

// The fused layer with (residual != nullptr) or without a residual per output
// rank.  Residual q is rows elements like y; it may be y[q] itself (in place)
// but must not partially overlap y[q] nor overlap any other output.
int tokens_launch(dcc_comm_t c, void* const* weight, void* const* x, void* const* residual, void* const* y,
                  size_t tokens, size_t rows, size_t kp, dcc_dtype_t t, dcc_stream_t s);

int linear_launch(dcc_comm_t c, void* const* weight, void* const* x, void* const* residual, void* const* y,
                  size_t rows, size_t kp, dcc_dtype_t t, dcc_stream_t s) {
  if (!c || !weight || !x || !y) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  if (t != DCC_BF16 && t != DCC_FP16) return DCC_ERR_UNSUPPORTED;
  if (rows % 8 || kp % 8) return DCC_ERR_UNSUPPORTED;  // the documented shape rule
  if (rows == 0 || kp == 0) return DCC_OK;
  const size_t eb = 2;
  if (rows > ((size_t)1 << 40) / kp) return DCC_ERR_INVALID_ARG;
  const size_t wb = rows * kp * eb, xb = kp * eb, yb = rows * eb;
  for (int r = 0; r < c->n; ++r) {
    if (!weight[r] || !x[r] || !y[r]) return DCC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(weight[r]) | reinterpret_cast<uintptr_t>(x[r]) |
         reinterpret_cast<uintptr_t>(y[r])) & 15u)
      return DCC_ERR_MISALIGNED;
    const void* ptrs[3] = {weight[r], x[r], y[r]};
    const size_t lens[3] = {wb, xb, yb};
    for (int j = 0; j < 3; ++j)
      if (!in_window(c, r, DCC_BUF_INPUT, ptrs[j], lens[j]) && !in_window(c, r, DCC_BUF_OUTPUT, ptrs[j], lens[j]))
        return DCC_ERR_NOT_REGISTERED;
  }
  for (int r = 0; r < c->n; ++r)
    for (int p = 0; p < c->n; ++p) {
      if (overlaps(y[r], yb, weight[p], wb) || overlaps(y[r], yb, x[p], xb)) return DCC_ERR_INVALID_ARG;
      if (p != r && overlaps(y[r], yb, y[p], yb)) return DCC_ERR_INVALID_ARG;
    }
  if (residual) {
    for (int r = 0; r < c->n; ++r) {
      if (!residual[r]) return DCC_ERR_INVALID_ARG;
      if (reinterpret_cast<uintptr_t>(residual[r]) & 15u) return DCC_ERR_MISALIGNED;
      if (!in_window(c, r, DCC_BUF_INPUT, residual[r], yb) && !in_window(c, r, DCC_BUF_OUTPUT, residual[r], yb))
        return DCC_ERR_NOT_REGISTERED;
      for (int p = 0; p < c->n; ++p)
        if (overlaps(residual[r], yb, y[p], yb) && !(p == r && residual[r] == y[r])) return DCC_ERR_INVALID_ARG;
    }
  }
  // kp up to kFusedTensorMaxKp: the tensor-core kernel, as the batched layer
  // with one token (same layouts: x is 1 x kp, y 1 x rows)
  if (kp <= ((size_t)1 << 31) / (size_t)c->n && rows <= ((size_t)1 << 31) &&
      (c->fused_kernel == 2 || (c->fused_kernel < 0 && kp <= kFusedTensorMaxKp)))
    return tokens_launch(c, weight, x, residual, y, 1, rows, kp, t, s);
  int rc = check_channels_all_pairs(c);
  if (rc != DCC_OK) return rc;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  dcc::LinearArgs a{};
  for (int r = 0; r < c->n; ++r) {
    a.weight[r] = weight[r];
    a.x[r] = x[r];
    a.residual[r] = residual ? residual[r] : nullptr;
    a.y[r] = y[r];
  }
  a.rows = rows;
  a.kp = kp;
  for (int r = 0; r < c->n; ++r) {
    set_extent(a, dcc::kBufSend, r, wb);
    set_extent(a, dcc::kBufX, r, xb);
    set_extent(a, dcc::kBufRecv, r, yb);
    set_extent(a, dcc::kBufResidual, r, residual ? yb : 0);
  }
  dcc::DevComm dc = dev_view(c);
  void* kargs[] = {&dc, &a};
  if (c->fused_kernel == 1 || (c->fused_kernel < 0 && kp >= kFusedBulkMinKp)) {
    const void* fn = t == DCC_BF16 ? dcc::linear_allreduce_bulk_kernel<__nv_bfloat16>(c->n)
                                   : dcc::linear_allreduce_bulk_kernel<__half>(c->n);
    const size_t smem = dcc::fused_bulk_smem_bytes();
    const size_t items = rows / dcc::kFusedBulkRows / (size_t)c->n + 1;  // 2-row items per rank
    rc = pick_blocks(c, fn, dcc::kFusedThreads, items, &a.blocks, smem, 1, false);  // one item per CTA
    if (rc != DCC_OK) return rc;
    return launch(fn, a.blocks * c->n, dcc::kFusedThreads, false, kargs, static_cast<cudaStream_t>(s), smem, c->pdl);
  }
  const void* fn = t == DCC_BF16 ? dcc::linear_allreduce_kernel<__nv_bfloat16>(c->n)
                                 : dcc::linear_allreduce_kernel<__half>(c->n);
  const size_t items = rows / dcc::kFusedRows / (size_t)c->n + 1;  // items per rank
  rc = pick_blocks(c, fn, dcc::kFusedThreads, items, &a.blocks, 0, 1, false);  // one item per CTA
  if (rc != DCC_OK) return rc;
  return launch(fn, a.blocks * c->n, dcc::kFusedThreads, false, kargs, static_cast<cudaStream_t>(s), 0, c->pdl);
}

// cuTensorMapEncodeTiled from the driver (through the runtime, so the library
// needs no link against the driver library)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// A 2-D tensor map over a row-major outer x inner matrix of 16-bit elements,
// box 64 (inner, one 128-byte swizzle row) x box_rows, 128-byte swizzle,
// elements outside the matrix read as zero.  Cached on the communicator.
int tensor_map(dcc_comm* c, const void* ptr, size_t inner, size_t outer, unsigned box_rows, dcc_dtype_t t,
               CUtensorMap* out) {
  const dcc_comm::MapKey key{ptr, inner, outer, box_rows, (unsigned)t};
  auto it = c->tmaps.find(key);
  if (it != c->tmaps.end()) {
    *out = it->second;
    return DCC_OK;
  }
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return DCC_ERR_UNSUPPORTED;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  const cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  const cuuint32_t box[2] = {(cuuint32_t)dcc::kMmaBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap m;
  if (enc(&m, t == DCC_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
          const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return DCC_ERR_INVALID_ARG;
  if (c->tmaps.size() >= 4096) c->tmaps.clear();
  c->tmaps.emplace(key, m);
  *out = m;
  return DCC_OK;
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

const char* dcc_error_string(int code) {
  switch (code) {
    case DCC_OK: return "DCC_OK";
    case DCC_ERR_INVALID_ARG: return "DCC_ERR_INVALID_ARG";
    case DCC_ERR_NOT_REGISTERED: return "DCC_ERR_NOT_REGISTERED";
    case DCC_ERR_MISALIGNED: return "DCC_ERR_MISALIGNED";
    case DCC_ERR_NO_CHANNEL: return "DCC_ERR_NO_CHANNEL";
    case DCC_ERR_CUDA: return "DCC_ERR_CUDA";
    case DCC_ERR_LAUNCH: return "DCC_ERR_LAUNCH";
    case DCC_ERR_TIMEOUT: return "DCC_ERR_TIMEOUT";
    case DCC_ERR_UNSUPPORTED: return "DCC_ERR_UNSUPPORTED";
    case DCC_ERR_BOUNDS: return "DCC_ERR_BOUNDS";
    default: return "DCC_ERR_UNKNOWN";
  }
}

const char* dcc_version(void) { return "dcc 0.2 (sm_103a)"; }

int dcc_kernel_binary_version(int* version) {
  if (!version) return DCC_ERR_INVALID_ARG;
  int seen = 0;
  bool mixed = false;
  const bool ok = visit_kernels([&](const void* fn) {
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, fn) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    if (seen && attr.binaryVersion != seen) mixed = true;
    seen = attr.binaryVersion;
    return true;
  });
  if (!ok) return DCC_ERR_CUDA;
  if (mixed) return DCC_ERR_UNSUPPORTED;
  *version = seen;
  return DCC_OK;
}

int dcc_shard_range(size_t count, int n_ranks, int rank, size_t eb, size_t* begin, size_t* end) {
  if (n_ranks < 1 || n_ranks > DCC_MAX_RANKS || rank < 0 || rank >= n_ranks || !begin || !end)
    return DCC_ERR_INVALID_ARG;
  if (eb != 2 && eb != 4) return DCC_ERR_INVALID_ARG;
  shard_of(count, n_ranks, rank, eb, begin, end);
  return DCC_OK;
}

int dcc_comm_create(int n_ranks, dcc_comm_t* out) {
  if (!out || n_ranks < 1 || n_ranks > DCC_MAX_RANKS) return DCC_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  dcc_comm* c = new dcc_comm();
  c->n = n_ranks;
  c->device = dev;
  for (int t = 0; t < 4; ++t) c->one_shot_max[t] = dcc_host::default_one_shot_max(n_ranks, (dcc_dtype_t)t);
  if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->smem_reserved_cta, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return DCC_ERR_CUDA;
  }
  const size_t sem_words = dcc::kSemSlots * dcc::kSemWords;
  const size_t ll_epochs = (size_t)DCC_MAX_RANKS * DCC_MAX_BLOCKS_PER_RANK;
  // sem | expect | status (own 256-byte line) | LL epochs
  const size_t words = sem_words + dcc::kSemSlots + 32 + ll_epochs;
  const size_t ll_bytes = (size_t)n_ranks * dcc::kLLBufBytes;
  if (cudaMalloc(&c->d_block, words * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMalloc(&c->d_table, sizeof(c->h_table)) != cudaSuccess ||
      cudaMalloc(&c->d_ll, ll_bytes) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(c->d_block);
    cudaFree(c->d_table);
    cudaFree(c->d_ll);
    delete c;
    return DCC_ERR_CUDA;
  }
  if (cudaMemset(c->d_block, 0, words * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMemset(c->d_table, 0, sizeof(c->h_table)) != cudaSuccess ||
      cudaMemset(c->d_ll, 0, ll_bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    cudaFree(c->d_block);
    cudaFree(c->d_table);
    cudaFree(c->d_ll);
    delete c;
    return DCC_ERR_CUDA;
  }
  c->dev.n = n_ranks;
  c->dev.skip_signal_rank = -1;
  c->dev.timeout_ns = 2000000ull * 1000ull;
  if (const char* v = std::getenv("DCC_WAIT_TIMEOUT_US")) {
    const unsigned long long us = std::strtoull(v, nullptr, 10);
    if (us > 0) c->dev.timeout_ns = us * 1000ull;
  }
  if (const char* v = std::getenv("DCC_BLOCKS_PER_RANK")) c->blocks_override = std::atoi(v);
  if (const char* v = std::getenv("DCC_THREADS")) {
    const int t = std::atoi(v);
    if (t >= 32 && t <= dcc::kThreads && t % 32 == 0) c->threads_override = t;
  }
  if (const char* v = std::getenv("DCC_ALGO")) {
    if (!std::strcmp(v, "one_shot")) c->forced_algo = DCC_ALGO_ONE_SHOT;
    else if (!std::strcmp(v, "two_shot")) c->forced_algo = DCC_ALGO_TWO_SHOT;
    else if (!std::strcmp(v, "two_shot_scratch")) c->forced_algo = DCC_ALGO_TWO_SHOT_SCRATCH;
    else if (!std::strcmp(v, "two_shot_bulk")) c->forced_algo = DCC_ALGO_TWO_SHOT_BULK;
  }
  c->log = env_flag("DCC_LOG");
  if (const char* v = std::getenv("DCC_AG_BULK")) c->ag_bulk = std::strcmp(v, "0") != 0;
  if (const char* v = std::getenv("DCC_ZERO_COPY")) c->zero_copy = std::strcmp(v, "0") != 0;
  if (const char* v = std::getenv("DCC_FUSED_BULK")) c->fused_kernel = std::strcmp(v, "0") != 0 ? 1 : 0;
  if (const char* v = std::getenv("DCC_FUSED_KERNEL")) {
    if (!std::strcmp(v, "thread")) c->fused_kernel = 0;
    else if (!std::strcmp(v, "bulk")) c->fused_kernel = 1;
    else if (!std::strcmp(v, "tensor")) c->fused_kernel = 2;
  }
  if (const char* v = std::getenv("DCC_MMA_FORM")) {
    if (!std::strcmp(v, "pair")) c->mma_form = kMmaFormPair;
    else if (!std::strcmp(v, "one")) c->mma_form = kMmaFormOne;
    else if (!std::strcmp(v, "two")) c->mma_form = kMmaFormTwo;
  }
  if (const char* v = std::getenv("DCC_INPLACE_UNROLL")) {
    const int u = std::atoi(v);
    if (u >= 1 && u <= dcc::kInplaceUnroll) c->inplace_unroll = u;
  }
  c->entry_barrier = env_flag("DCC_ENTRY_BARRIER");
  if (const char* v = std::getenv("DCC_PDL")) c->pdl = std::strcmp(v, "0") != 0;
  if (const char* v = std::getenv("DCC_RING_CLUSTER")) c->ring_cluster = std::strcmp(v, "0") != 0;
  c->dev.sem = c->d_block;
  c->dev.expect = c->d_block + sem_words;
  c->dev.status = c->d_block + sem_words + dcc::kSemSlots + 8;  // own 64-byte line
  c->dev.ll_epoch = c->d_block + sem_words + dcc::kSemSlots + 32;
  c->dev.ll_buf = c->d_ll;
  *out = c;
  return DCC_OK;
}

int dcc_comm_destroy(dcc_comm_t c) {
  if (!c) return DCC_OK;
  int rc = DCC_OK;
  {
    DeviceScope ds(c->device);
    dcc_proxy_release(c);
    if (cudaDeviceSynchronize() != cudaSuccess) rc = DCC_ERR_CUDA;
    if (c->pipe_ready) {
      cudaStreamDestroy(c->pipe_in);
      cudaStreamDestroy(c->pipe_out);
      cudaEventDestroy(c->ev_start);
      cudaEventDestroy(c->ev_in);
      cudaEventDestroy(c->ev_kernel);
      cudaEventDestroy(c->ev_done);
    }
    if (cudaFree(c->d_block) != cudaSuccess) rc = DCC_ERR_CUDA;
    if (cudaFree(c->d_table) != cudaSuccess) rc = DCC_ERR_CUDA;
    if (cudaFree(c->d_ll) != cudaSuccess) rc = DCC_ERR_CUDA;
    cudaGetLastError();
  }
  delete c;
  return rc;
}

int dcc_register_buffer(dcc_comm_t c, int rank, dcc_buf_kind_t kind, void* dev_ptr, size_t bytes) {
  if (!c || rank < 0 || rank >= c->n || kind < DCC_BUF_INPUT || kind > DCC_BUF_SCRATCH ||
      !dev_ptr || bytes == 0)
    return DCC_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(dev_ptr) & 15u) return DCC_ERR_MISALIGNED;
  auto& v = c->win[rank][kind];
  for (const Window& w : v)
    if (w.ptr == dev_ptr && w.bytes == bytes) return DCC_OK;
  if (v.size() >= DCC_MAX_WINDOWS) return DCC_ERR_INVALID_ARG;
  v.push_back(Window{static_cast<char*>(dev_ptr), bytes});
  c->table_dirty = true;
  return DCC_OK;
}

int dcc_memory_channel_make(dcc_comm_t c, int src, int dst) {
  if (!c || src < 0 || dst < 0 || src >= c->n || dst >= c->n || src == dst)
    return DCC_ERR_INVALID_ARG;
  c->chan[src][dst] = true;
  c->table_dirty = true;
  return DCC_OK;
}

int dcc_allreduce(dcc_comm_t c, void* const* send, void* const* recv, size_t count, dcc_dtype_t t,
                  dcc_algo_t a, dcc_stream_t s) {
  if (!c) return DCC_ERR_INVALID_ARG;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  return allreduce_launch(c, send, recv, count, t, a, static_cast<cudaStream_t>(s));
}

int dcc_allreduce_op(dcc_comm_t c, void* const* send, void* const* recv, size_t count, dcc_dtype_t t,
                     dcc_red_op_t op, dcc_algo_t a, dcc_stream_t s) {
  if (!c) return DCC_ERR_INVALID_ARG;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  return allreduce_launch(c, send, recv, count, t, a, static_cast<cudaStream_t>(s), (int)op);
}

// The message is cut into chunks of whole vectors.  Chunk i's inputs are
// copied in on the copy-in stream, reduced on the caller's stream once they
// have landed, and copied out on the copy-out stream once reduced, so the two
// copy directions and the kernels of different chunks overlap.  The caller's
// stream first hands its prior work to both copy streams and finally waits
// for the last copy out, so the call is one stream-ordered operation on s.
int dcc_allreduce_from_host(dcc_comm_t c, const void* const* host_send, void* const* host_recv,
                            void* const* dev_send, void* const* dev_recv, size_t count,
                            dcc_dtype_t t, dcc_algo_t a, dcc_stream_t s) {
  if (!c || !host_send || !host_recv) return DCC_ERR_INVALID_ARG;
  if (elem_bytes(t) == 0) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  if (count == 0) return DCC_OK;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  const size_t eb = elem_bytes(t);
  const size_t bytes = count * eb;
  bool inplace = false;
  int rc = check_buffers(c, dev_send, bytes, dev_recv, bytes, true, &inplace);
  if (rc != DCC_OK) return rc;
  rc = check_channels_all_pairs(c);
  if (rc != DCC_OK) return rc;
  for (int r = 0; r < c->n; ++r)
    if (!host_send[r] || !host_recv[r]) return DCC_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(s);
  // Zero copy: when every host buffer is pinned memory the GPU can address,
  // the two-shot kernel reads the inputs and writes the outputs over the
  // host link directly (each input byte crosses once, each output byte
  // once), which keeps both link directions busy with no staging in HBM.
  // Measured on GB300 for 8 x 256 MiB bf16: 13.5 ms vs 14.8-15.4 ms staged.
  if (c->zero_copy && (a == DCC_ALGO_AUTO || a == DCC_ALGO_TWO_SHOT)) {
    void* zs[DCC_MAX_RANKS];
    void* zr[DCC_MAX_RANKS];
    bool ok = true;
    for (int r = 0; r < c->n && ok; ++r)
      ok = device_address(host_send[r], bytes, &zs[r]) && device_address(host_recv[r], bytes, &zr[r]) &&
           !((reinterpret_cast<uintptr_t>(zs[r]) | reinterpret_cast<uintptr_t>(zr[r])) & 15u);
    bool zinplace = false;
    for (int r = 0; r < c->n && ok; ++r)
      for (int p = 0; p < c->n && ok; ++p) {
        if (overlaps(zr[r], bytes, zs[p], bytes)) {
          ok = r == p && zr[r] == zs[r];
          zinplace = zinplace || ok;
        }
        if (ok && p != r && overlaps(zr[r], bytes, zr[p], bytes)) ok = false;
      }
    if (ok) return run_allreduce(c, zs, zr, count, t, DCC_ALGO_TWO_SHOT, zinplace, st);
  }
  if (!c->pipe_ready) {
    if (cudaStreamCreateWithFlags(&c->pipe_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&c->pipe_out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->ev_start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->ev_in, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->ev_kernel, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->ev_done, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return DCC_ERR_CUDA;
    }
    c->pipe_ready = true;
  }
  const size_t vw = 16 / eb;
  size_t chunk = kPipeChunkBytes / eb / vw * vw;
  if (chunk < vw) chunk = vw;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ok(cudaEventRecord(c->ev_start, st)) || !ok(cudaStreamWaitEvent(c->pipe_in, c->ev_start, 0)) ||
      !ok(cudaStreamWaitEvent(c->pipe_out, c->ev_start, 0)))
    return DCC_ERR_CUDA;
  void* send_i[DCC_MAX_RANKS];
  void* recv_i[DCC_MAX_RANKS];
  for (size_t c0 = 0; c0 < count; c0 += chunk) {
    const size_t n_el = count - c0 < chunk ? count - c0 : chunk;
    const size_t off = c0 * eb, nb = n_el * eb;
    for (int r = 0; r < c->n; ++r) {
      send_i[r] = static_cast<char*>(dev_send[r]) + off;
      recv_i[r] = static_cast<char*>(dev_recv[r]) + off;
      if (!ok(cudaMemcpyAsync(send_i[r], static_cast<const char*>(host_send[r]) + off, nb,
                              cudaMemcpyHostToDevice, c->pipe_in)))
        return DCC_ERR_CUDA;
    }
    if (!ok(cudaEventRecord(c->ev_in, c->pipe_in)) || !ok(cudaStreamWaitEvent(st, c->ev_in, 0)))
      return DCC_ERR_CUDA;
    rc = allreduce_launch(c, send_i, recv_i, n_el, t, a, st);
    if (rc != DCC_OK) return rc;
    if (!ok(cudaEventRecord(c->ev_kernel, st)) || !ok(cudaStreamWaitEvent(c->pipe_out, c->ev_kernel, 0)))
      return DCC_ERR_CUDA;
    for (int r = 0; r < c->n; ++r)
      if (!ok(cudaMemcpyAsync(static_cast<char*>(host_recv[r]) + off, recv_i[r], nb,
                              cudaMemcpyDeviceToHost, c->pipe_out)))
        return DCC_ERR_CUDA;
  }
  if (!ok(cudaEventRecord(c->ev_done, c->pipe_out)) || !ok(cudaStreamWaitEvent(st, c->ev_done, 0)))
    return DCC_ERR_CUDA;
  return DCC_OK;
}

int dcc_reduce_scatter(dcc_comm_t c, void* const* send, void* const* recv, size_t recv_count,
                       dcc_dtype_t t, dcc_stream_t s) {
  return dcc_reduce_scatter_op(c, send, recv, recv_count, t, DCC_OP_SUM, s);
}

int dcc_reduce_scatter_op(dcc_comm_t c, void* const* send, void* const* recv, size_t recv_count,
                          dcc_dtype_t t, dcc_red_op_t op, dcc_stream_t s) {
  if (!c || elem_bytes(t) == 0) return DCC_ERR_INVALID_ARG;
  if (op != DCC_OP_SUM && op != DCC_OP_MAX && op != DCC_OP_MIN) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  if (recv_count == 0) return DCC_OK;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  const size_t rb = recv_count * elem_bytes(t);
  const size_t sb = rb * (size_t)c->n;
  if (rb / elem_bytes(t) != recv_count || sb / (size_t)c->n != rb) return DCC_ERR_INVALID_ARG;
  bool inplace = false;
  int rc = check_buffers(c, send, sb, recv, rb, false, &inplace);
  if (rc != DCC_OK) return rc;
  rc = check_channels_all_pairs(c);
  if (rc != DCC_OK) return rc;
  dcc::CollArgs args{};
  for (int r = 0; r < c->n; ++r) {
    args.send[r] = send[r];
    args.recv[r] = recv[r];
  }
  args.count = recv_count;
  for (int r = 0; r < c->n; ++r) {
    set_extent(args, dcc::kBufSend, r, sb);
    set_extent(args, dcc::kBufRecv, r, rb);
  }
  // with the entry barrier the CTAs wait on one another: one cooperative wave
  const bool coop = c->entry_barrier && c->n > 1;
  const void* fn = op_kernel_for(t, (int)op, coop ? dcc::kReduceScatterEB : dcc::kReduceScatter, c->n);
  if (!fn) return DCC_ERR_INVALID_ARG;
  const size_t vw = 16 / elem_bytes(t);
  const size_t work = (recv_count + vw - 1) / vw;
  const int threads = c->threads_override > 0 ? c->threads_override : threads_for(DCC_ALGO_TWO_SHOT, work);
  rc = pick_blocks(c, fn, threads, work, &args.blocks, 0, 0, coop);
  if (rc != DCC_OK) return rc;
  dcc::DevComm dc = dev_view(c);
  void* kargs[] = {&dc, &args};
  return launch(fn, args.blocks * c->n, threads, coop, kargs, static_cast<cudaStream_t>(s), 0,
                c->pdl && !coop);
}

int dcc_allgather(dcc_comm_t c, void* const* send, void* const* recv, size_t send_count,
                  dcc_dtype_t t, dcc_stream_t s) {
  if (!c || elem_bytes(t) == 0) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  if (send_count == 0) return DCC_OK;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  const size_t sb = send_count * elem_bytes(t);
  const size_t rb = sb * (size_t)c->n;
  if (sb / elem_bytes(t) != send_count || rb / (size_t)c->n != sb) return DCC_ERR_INVALID_ARG;
  bool inplace = false;
  int rc = check_buffers(c, send, sb, recv, rb, false, &inplace);
  if (rc != DCC_OK) return rc;
  rc = check_channels_all_pairs(c);
  if (rc != DCC_OK) return rc;
  dcc::CollArgs args{};
  for (int r = 0; r < c->n; ++r) {
    args.send[r] = send[r];
    args.recv[r] = recv[r];
  }
  args.count = send_count;
  for (int r = 0; r < c->n; ++r) {
    set_extent(args, dcc::kBufSend, r, sb);
    set_extent(args, dcc::kBufRecv, r, rb);
  }
  int eb = (int)elem_bytes(t);
  dcc::DevComm dc = dev_view(c);
  void* kargs[] = {&dc, &args, &eb};
  // with the entry barrier the CTAs wait on one another: one cooperative wave
  // of the thread-copy kernel (the bulk-copy kernel has no entry barrier)
  const bool coop = c->entry_barrier && c->n > 1;
  if (!coop && c->ag_bulk && sb % 16 == 0 && sb >= kAgBulkMinBytes) {
    const void* fn = dcc::allgather_bulk_kernel(c->n);
    const size_t smem = dcc::ag_smem_bytes();
    rc = pick_blocks(c, fn, 32, (sb + dcc::kAgTile - 1) / dcc::kAgTile, &args.blocks, smem, 1);
    if (rc != DCC_OK) return rc;
    return launch(fn, args.blocks * c->n, 32, false, kargs, static_cast<cudaStream_t>(s), smem, c->pdl);
  }
  const void* fn = dcc::allgather_kernel(c->n, coop);
  const size_t work = (sb + 15) / 16;
  const int threads = c->threads_override > 0 ? c->threads_override : threads_for(DCC_ALGO_TWO_SHOT, work);
  // vector path: kAgUnroll vectors per thread; element path: one element per thread
  const size_t per_block = sb % 16 == 0 ? (size_t)dcc::kAgUnroll * threads : (size_t)threads;
  rc = pick_blocks(c, fn, threads, sb % 16 == 0 ? work : send_count, &args.blocks, 0, per_block, coop);
  if (rc != DCC_OK) return rc;
  return launch(fn, args.blocks * c->n, threads, coop, kargs, static_cast<cudaStream_t>(s), 0,
                c->pdl && !coop);
}


int dcc_linear_allreduce(dcc_comm_t c, void* const* weight, void* const* x, void* const* y, size_t rows,
                         size_t kp, dcc_dtype_t t, dcc_stream_t s) {
  return linear_launch(c, weight, x, nullptr, y, rows, kp, t, s);
}

int dcc_linear_allreduce_residual(dcc_comm_t c, void* const* weight, void* const* x, void* const* residual,
                                  void* const* y, size_t rows, size_t kp, dcc_dtype_t t, dcc_stream_t s) {
  if (!residual) return DCC_ERR_INVALID_ARG;
  return linear_launch(c, weight, x, residual, y, rows, kp, t, s);
}

}  // extern "C"

namespace {
// Raises fn's dynamic shared-memory limit on the current device to at least
// smem, with all of the SM's unified memory as shared memory.  It never
// lowers the limit (a function attribute holds for every communicator, and a
// plan one of them cached must stay launchable).  Called when a plan is made.
int raise_smem_limit(const void* fn, size_t smem) {
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, fn) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_LAUNCH;
  }
  if ((size_t)fa.maxDynamicSharedSizeBytes >= smem) return DCC_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess ||
      cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_LAUNCH;
  }
  return DCC_OK;
}

// The form: "pair", 128-thread CTAs two to an SM with half the shared memory
// each and one accumulator (the K split can then be twice as deep at the same
// bytes in flight per SM); "one", 256-thread CTAs one to an SM with one
// accumulator; "two", the same with two accumulators sharing each token tile.
// Then tiles of bm weight rows (a multiple of 8; 64..128 with one
// accumulator, 136..256 with two) and ks K splits (a cluster of ks CTAs per
// tile, ks <= kMmaMaxSplit and at most one 64-element block each): for each
// ks the tile count that fills the most of one wave (at most as many
// clusters as fit on the device at once, which the GPCs' SM counts make
// fewer than SMs / ks), and of those the deepest split that keeps at least
// 3/4 of the best CTA count (measured on GB300: the weight stream runs faster
// the deeper the split, 23.5 us for 134 MB with a 4-way split against 27.3
// with a 2-way one).
MmaPlan plan_mma(dcc_comm_t c, int form, int ntile, size_t rows, size_t kp, bool res) {
  const auto pkey = std::make_tuple(form, ntile, rows, kp, res);
  const auto hit = c->mma_plans.find(pkey);
  if (hit != c->mma_plans.end()) return hit->second;
  MmaPlan p;
  int macc = form == kMmaFormTwo ? 2 : 1;
  // one accumulator where the rows, the tensor memory (512 columns) or the
  // epilogue's room in the stage buffers do not allow two
  const int acc_cols = ntile <= 32 ? 32 : ntile <= 64 ? 64 : ntile <= 128 ? 128 : 256;
  if (macc == 2 && (rows <= (size_t)dcc::kMmaBM || acc_cols * 2 > 512 ||
                    !dcc::mma_epilogue_fits(ntile, dcc::mma_stages(ntile, 2), 2, 1)))
    macc = 1;
  const int threads = form == kMmaFormPair ? dcc::kMmaPairThreads : dcc::kMmaThreads;
  const unsigned budget = form == kMmaFormPair ? dcc::kMmaPairStageBudget : dcc::kMmaStageBudget;
  const void* fn = dcc::linear_allreduce_mma_kernel(c->n, macc, threads, res);
  const int stages = dcc::mma_stages(ntile, macc, budget);
  const size_t smem = dcc::mma_smem_bytes(ntile, stages, macc);
  p.rc = raise_smem_limit(fn, smem);
  if (p.rc != DCC_OK) return p;
  // two CTAs' shared memory fit one SM (the pair form with a small token tile)
  const bool two_per_sm = threads == dcc::kMmaPairThreads &&
                          2 * (smem + (size_t)c->smem_reserved_cta) <= (size_t)c->smem_per_sm;
  auto fit = [&](int ks) -> long long {  // clusters of ks CTAs resident at once
    const auto key = std::make_tuple(fn, ks, smem);
    const auto it = c->mma_clusters.find(key);
    if (it != c->mma_clusters.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ks);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)ks;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int num = 0;
    if (cudaOccupancyMaxActiveClusters(&num, fn, &cfg) != cudaSuccess) {
      cudaGetLastError();
      num = c->num_sms / ks;
    }
    // The query counts one CTA per SM for a kernel that allocates tensor
    // memory; two pair-form CTAs whose shared memory fits run side by side
    // (measured on GB300: a grid of twice the SMs takes the time of one).
    // Were they not to, the extra clusters would only form a second wave: no
    // cluster waits on another.
    if (two_per_sm) num *= 2;
    c->mma_clusters[key] = num;
    return num;
  };
  const int bm_lo = macc == 1 ? 64 : dcc::kMmaBM + 8, bm_hi = macc * dcc::kMmaBM;
  const int kblocks = c->n * (int)((kp + dcc::kMmaBK - 1) / dcc::kMmaBK);
  auto tiles = [&](int bm) { return (long long)((rows + bm - 1) / bm); };
  int ks_bm[dcc::kMmaMaxSplit + 1] = {};  // per split: the tile height, 0 = none fits one wave
  long long ks_ctas[dcc::kMmaMaxSplit + 1] = {}, most = 0;
  for (int ks = 1; ks <= dcc::kMmaMaxSplit && ks <= kblocks; ks *= 2) {
    if (!dcc::mma_epilogue_fits(ntile, stages, macc, ks)) break;  // no room for the epilogue's inbox
    const long long cap = fit(ks);
    for (int bm = bm_lo; bm <= bm_hi; bm += 8) {  // shorter tiles: more CTAs
      if (tiles(bm) > cap) continue;
      int tall = bm;  // the tallest tile with the same tile count
      while (tall + 8 <= bm_hi && tiles(tall + 8) == tiles(bm)) tall += 8;
      ks_bm[ks] = tall;
      ks_ctas[ks] = tiles(bm) * ks;
      if (ks_ctas[ks] > most) most = ks_ctas[ks];
      break;
    }
  }
  p.bm = bm_hi;  // more tiles than fit even at the tallest tile: several waves, no split
  p.ks = 1;
  for (int ks = dcc::kMmaMaxSplit; ks >= 1; ks /= 2)
    if (ks_bm[ks] && 4 * ks_ctas[ks] >= 3 * most) {
      p.bm = ks_bm[ks];
      p.ks = ks;
      p.one_wave = true;
      break;
    }
  p.fn = fn;
  p.threads = threads;
  p.macc = macc;
  p.stages = stages;
  p.smem = smem;
  p.rounds = dcc::mma_epilogue_rounds(ntile, stages, macc, p.ks);
  if (c->mma_plans.size() >= 4096) c->mma_plans.clear();
  c->mma_plans.emplace(pkey, p);
  return p;
}

// Whether plan a should run rather than plan b: a grid in one wave first,
// then an epilogue in one round, then the deeper K split; on a tie b stays.
// Measured on GB300 (8 ranks, bf16): with the two-accumulator form's rule
// beside it, this picks the faster form, or one within 4 % (about the
// run-to-run spread), over rows 4096 / 8192 / 16384 / 28672, kp 512 / 1024 /
// 2048 and 1 to 256 tokens.
bool better_plan(const MmaPlan& a, const MmaPlan& b) {
  if (a.one_wave != b.one_wave) return a.one_wave;
  if ((a.rounds == 1) != (b.rounds == 1)) return a.rounds == 1;
  return a.ks > b.ks;
}

int tokens_launch(dcc_comm_t c, void* const* weight, void* const* x, void* const* residual, void* const* y,
                  size_t tokens, size_t rows, size_t kp, dcc_dtype_t t, dcc_stream_t s) {
  if (!c || !weight || !x || !y) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  if (t != DCC_BF16 && t != DCC_FP16) return DCC_ERR_UNSUPPORTED;
  // kp: rows of the tensor maps are 16-byte multiples
  if (tokens > (size_t)dcc::kMmaMaxTokens || rows % 8 || kp % 8) return DCC_ERR_UNSUPPORTED;
  if (tokens == 0 || rows == 0 || kp == 0) return DCC_OK;
  if (rows > ((size_t)1 << 31) || kp > ((size_t)1 << 31) / (size_t)c->n) return DCC_ERR_UNSUPPORTED;
  const size_t wb = rows * kp * 2, xb = tokens * kp * 2, yb = tokens * rows * 2;
  for (int r = 0; r < c->n; ++r) {
    if (!weight[r] || !x[r] || !y[r]) return DCC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(weight[r]) | reinterpret_cast<uintptr_t>(x[r]) |
         reinterpret_cast<uintptr_t>(y[r])) & 15u)
      return DCC_ERR_MISALIGNED;
    const void* ptrs[3] = {weight[r], x[r], y[r]};
    const size_t lens[3] = {wb, xb, yb};
    for (int j = 0; j < 3; ++j)
      if (!in_window(c, r, DCC_BUF_INPUT, ptrs[j], lens[j]) && !in_window(c, r, DCC_BUF_OUTPUT, ptrs[j], lens[j]))
        return DCC_ERR_NOT_REGISTERED;
  }
  for (int r = 0; r < c->n; ++r)
    for (int p = 0; p < c->n; ++p) {
      if (overlaps(y[r], yb, weight[p], wb) || overlaps(y[r], yb, x[p], xb)) return DCC_ERR_INVALID_ARG;
      if (p != r && overlaps(y[r], yb, y[p], yb)) return DCC_ERR_INVALID_ARG;
    }
  if (residual) {
    for (int r = 0; r < c->n; ++r) {
      if (!residual[r]) return DCC_ERR_INVALID_ARG;
      if (reinterpret_cast<uintptr_t>(residual[r]) & 15u) return DCC_ERR_MISALIGNED;
      if (!in_window(c, r, DCC_BUF_INPUT, residual[r], yb) && !in_window(c, r, DCC_BUF_OUTPUT, residual[r], yb))
        return DCC_ERR_NOT_REGISTERED;
      for (int p = 0; p < c->n; ++p)
        if (overlaps(residual[r], yb, y[p], yb) && !(p == r && residual[r] == y[r])) return DCC_ERR_INVALID_ARG;
    }
  }
  int rc = check_channels_all_pairs(c);
  if (rc != DCC_OK) return rc;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  const int ntile = tokens <= 16 ? 16 : (int)((tokens + 15) / 16 * 16);
  dcc::MmaMaps maps;
  std::memset(&maps, 0, sizeof maps);
  // Launch shape (plan_mma): with no form requested, the pair form and the
  // one-accumulator form are both planned and the better plan runs
  // (better_plan); the two-accumulator form only where neither fits one wave
  // and it does (its taller tiles halve the tile count; measured on GB300,
  // 28672 rows x 256 tokens: 106 us against 126, while with both in one wave
  // its deeper split loses to the one-accumulator form's, 33.3 against 30.6
  // us at 8192 rows x 128 tokens).  DCC_MMA_FORM forces one.
  const bool res = residual != nullptr;  // the residual form is its own kernel
  MmaPlan plan;
  if (c->mma_form >= 0) {
    plan = plan_mma(c, c->mma_form, ntile, rows, kp, res);
  } else {
    plan = plan_mma(c, kMmaFormOne, ntile, rows, kp, res);
    if (plan.rc != DCC_OK) return plan.rc;
    const MmaPlan pair = plan_mma(c, kMmaFormPair, ntile, rows, kp, res);
    if (pair.rc != DCC_OK) return pair.rc;
    if (better_plan(pair, plan)) plan = pair;
    if (!plan.one_wave) {
      const MmaPlan two = plan_mma(c, kMmaFormTwo, ntile, rows, kp, res);
      if (two.rc != DCC_OK) return two.rc;
      if (two.macc == 2 && two.one_wave) plan = two;
    }
  }
  if (plan.rc != DCC_OK) return plan.rc;
  const void* fn = plan.fn;
  const int threads = plan.threads, macc = plan.macc, stages = plan.stages, best_bm = plan.bm, best_ks = plan.ks;
  const size_t smem = plan.smem;
  const int bm0 = macc == 1 ? best_bm : dcc::kMmaBM, bm_last = best_bm - dcc::kMmaBM * (macc - 1);
  for (int r = 0; r < c->n; ++r) {
    rc = tensor_map(c, weight[r], kp, rows, (unsigned)bm0, t, &maps.w[r]);
    if (rc == DCC_OK && macc > 1) rc = tensor_map(c, weight[r], kp, rows, (unsigned)bm_last, t, &maps.w2[r]);
    if (rc == DCC_OK) rc = tensor_map(c, x[r], kp, tokens, (unsigned)ntile, t, &maps.x[r]);
    if (rc != DCC_OK) return rc;
  }
  dcc::MmaArgs a{};
  for (int r = 0; r < c->n; ++r) {
    a.y[r] = y[r];
    a.res[r] = residual ? residual[r] : nullptr;
    set_extent(a, dcc::kBufRecv, r, yb);
    set_extent(a, dcc::kBufResidual, r, residual ? yb : 0);
  }
  a.tokens = (int)tokens;
  a.rows = (int)rows;
  a.kp = (int)kp;
  a.ntile = ntile;
  a.fp16 = t == DCC_FP16 ? 1 : 0;
  a.macc = macc;
  a.rounds = plan.rounds;
  a.stages = stages;
  a.bm = best_bm;
  a.ks = best_ks;
  const int mtiles = (int)((rows + best_bm - 1) / best_bm);
  if (c->log)
    std::fprintf(stderr,
                 "dcc_linear_allreduce_tokens: tokens=%zu rows=%zu kp=%zu threads=%d macc=%d bm=%d ks=%d ctas=%d "
                 "stages=%d rounds=%d smem=%zu one_wave=%d\n",
                 tokens, rows, kp, threads, macc, best_bm, best_ks, mtiles * best_ks, stages, a.rounds, smem,
                 plan.one_wave ? 1 : 0);
  dcc::DevComm dc = dev_view(c);
  void* kargs[] = {&maps, &dc, &a};
  return launch(fn, mtiles * best_ks, threads, false, kargs, static_cast<cudaStream_t>(s), smem, c->pdl, best_ks);
}
}  // namespace

extern "C" {

int dcc_linear_allreduce_tokens(dcc_comm_t c, void* const* weight, void* const* x, void* const* y, size_t tokens,
                                size_t rows, size_t kp, dcc_dtype_t t, dcc_stream_t s) {
  return tokens_launch(c, weight, x, nullptr, y, tokens, rows, kp, t, s);
}

int dcc_linear_allreduce_tokens_residual(dcc_comm_t c, void* const* weight, void* const* x, void* const* residual,
                                         void* const* y, size_t tokens, size_t rows, size_t kp, dcc_dtype_t t,
                                         dcc_stream_t s) {
  if (!residual) return DCC_ERR_INVALID_ARG;
  return tokens_launch(c, weight, x, residual, y, tokens, rows, kp, t, s);
}

int dcc_ring_barrier(dcc_comm_t c, int iters, dcc_stream_t s) {
  if (!c || iters < 0) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  for (int r = 0; r < c->n && c->n > 1; ++r)
    if (!c->chan[r][(r + 1) % c->n]) return DCC_ERR_NO_CHANNEL;
  if (iters == 0) return DCC_OK;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  dcc::DevComm dc = dev_view(c);
  void* kargs[] = {&dc, &iters};
  // up to 8 ranks (the portable cluster size) the token goes through
  // distributed shared memory, one CTA per rank in one cluster
  if (c->ring_cluster && c->n <= 8) {
    const int rc = launch(dcc::ring_barrier_cluster_kernel(), c->n, 32, false, kargs, static_cast<cudaStream_t>(s), 0,
                          false, c->n);
    if (rc != DCC_ERR_CUDA) return rc;  // a cluster shape the device refuses: the global-memory ring instead
  }
  return launch(dcc::ring_barrier_kernel(), c->n, 32, true, kargs, static_cast<cudaStream_t>(s));
}

int dcc_comm_check(dcc_comm_t c, dcc_stream_t s) {
  if (!c) return DCC_ERR_INVALID_ARG;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(s)) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  unsigned long long st = 0;
  if (cudaMemcpy(&st, c->dev.status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  if (st != 0 && c->sticky == DCC_OK) {
    c->err_rank = (int)((st >> 8) & 0xFF);
    c->err_peer = (int)((st >> 16) & 0xFF);
    if ((st & 0xFF) == dcc::kStatusBounds) {  // bounds-checked build: buffer kind, 16-byte offset
      const unsigned long long off = st >> 24;
      c->sticky = DCC_ERR_BOUNDS;
      c->err_block = off > 0x7fffffffull ? 0x7fffffff : (int)off;
    } else {
      c->sticky = DCC_ERR_TIMEOUT;
      c->err_block = (int)((st >> 24) & 0xFFFF);
    }
  }
  return c->sticky;
}

int dcc_comm_error_detail(dcc_comm_t c, int* rank, int* peer, int* block) {
  if (!c || c->sticky == DCC_OK) return DCC_ERR_INVALID_ARG;
  if (rank) *rank = c->err_rank;
  if (peer) *peer = c->err_peer;
  if (block) *block = c->err_block;
  return DCC_OK;
}

int dcc_channel_put(dcc_comm_t c, int src, int dst, size_t remote_off, size_t local_off,
                    size_t bytes, int signal, dcc_stream_t s) {
  if (!c || src < 0 || dst < 0 || src >= c->n || dst >= c->n || src == dst)
    return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  if (!c->chan[src][dst] || (signal && !c->chan[dst][src])) return DCC_ERR_NO_CHANNEL;
  if ((remote_off | local_off | bytes) & 15u) return DCC_ERR_MISALIGNED;
  if (c->win[src][DCC_BUF_INPUT].empty() || c->win[dst][DCC_BUF_OUTPUT].empty())
    return DCC_ERR_NOT_REGISTERED;
  const Window& li = c->win[src][DCC_BUF_INPUT][0];
  const Window& ro = c->win[dst][DCC_BUF_OUTPUT][0];
  if (local_off > li.bytes || bytes > li.bytes - local_off || remote_off > ro.bytes ||
      bytes > ro.bytes - remote_off)
    return DCC_ERR_NOT_REGISTERED;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(s);
  int rc = upload_table(c, st);
  if (rc != DCC_OK) return rc;
  dcc::PrimArgs pa{src, dst, remote_off, local_off, bytes, signal ? 1 : 0, c->d_table};
  dcc::DevComm dc = dev_view(c);
  void* kargs[] = {&dc, &pa};
  return launch(dcc::channel_put_kernel(), 2, 256, true, kargs, st);
}

int dcc_channel_get(dcc_comm_t c, int src, int dst, size_t remote_off, size_t local_off,
                    size_t bytes, dcc_stream_t s) {
  if (!c || src < 0 || dst < 0 || src >= c->n || dst >= c->n || src == dst)
    return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  if (!c->chan[src][dst]) return DCC_ERR_NO_CHANNEL;
  if ((remote_off | local_off | bytes) & 15u) return DCC_ERR_MISALIGNED;
  if (c->win[src][DCC_BUF_OUTPUT].empty() || c->win[dst][DCC_BUF_INPUT].empty())
    return DCC_ERR_NOT_REGISTERED;
  const Window& lo = c->win[src][DCC_BUF_OUTPUT][0];
  const Window& ri = c->win[dst][DCC_BUF_INPUT][0];
  if (local_off > lo.bytes || bytes > lo.bytes - local_off || remote_off > ri.bytes ||
      bytes > ri.bytes - remote_off)
    return DCC_ERR_NOT_REGISTERED;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(s);
  int rc = upload_table(c, st);
  if (rc != DCC_OK) return rc;
  dcc::PrimArgs pa{src, dst, remote_off, local_off, bytes, 0, c->d_table};
  dcc::DevComm dc = dev_view(c);
  void* kargs[] = {&dc, &pa};
  return launch(dcc::channel_get_kernel(), 1, 256, false, kargs, st);
}

int dcc_comm_read_semaphores(dcc_comm_t c, int block, uint64_t* inbound, uint64_t* expected,
                             dcc_stream_t s) {
  if (!c || block < 0 || block >= DCC_MAX_BLOCKS_PER_RANK) return DCC_ERR_INVALID_ARG;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(s)) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  for (int d = 0; d < c->n; ++d) {
    for (int q = 0; q < c->n; ++q) {
      const size_t slot = dcc::sem_slot(d, q, block);
      if (inbound && cudaMemcpy(&inbound[d * c->n + q], c->dev.sem + slot * dcc::kSemWords,
                                sizeof(uint64_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DCC_ERR_CUDA;
      if (expected && cudaMemcpy(&expected[d * c->n + q], c->dev.expect + slot, sizeof(uint64_t),
                                 cudaMemcpyDeviceToHost) != cudaSuccess)
        return DCC_ERR_CUDA;
    }
  }
  return DCC_OK;
}

int dcc_set_wait_timeout_us(dcc_comm_t c, uint64_t us) {
  if (!c || us == 0 || us > 3600ull * 1000000ull) return DCC_ERR_INVALID_ARG;
  c->dev.timeout_ns = us * 1000ull;
  return DCC_OK;
}

int dcc_set_blocks_per_rank(dcc_comm_t c, int blocks) {
  if (!c || blocks < 0 || blocks > DCC_MAX_BLOCKS_PER_RANK) return DCC_ERR_INVALID_ARG;
  c->blocks_override = blocks;
  return DCC_OK;
}

int dcc_set_pdl(dcc_comm_t c, int on) {
  if (!c) return DCC_ERR_INVALID_ARG;
  c->pdl = on != 0;
  return DCC_OK;
}

int dcc_set_entry_barrier(dcc_comm_t c, int on) {
  if (!c) return DCC_ERR_INVALID_ARG;
  c->entry_barrier = on != 0;
  return DCC_OK;
}

int dcc_set_algo_threshold(dcc_comm_t c, dcc_dtype_t t, size_t bytes) {
  if (!c || elem_bytes(t) == 0) return DCC_ERR_INVALID_ARG;
  c->one_shot_max[t] = bytes;
  return DCC_OK;
}

int dcc_auto_threshold(int n_ranks, dcc_dtype_t t, size_t* bytes) {
  if (!bytes || n_ranks < 1 || n_ranks > DCC_MAX_RANKS || elem_bytes(t) == 0) return DCC_ERR_INVALID_ARG;
  *bytes = dcc_host::default_one_shot_max(n_ranks, t);
  return DCC_OK;
}

int dcc_select_algo(dcc_comm_t c, size_t count, dcc_dtype_t t, dcc_algo_t* out) {
  if (!c || !out || elem_bytes(t) == 0) return DCC_ERR_INVALID_ARG;
  *out = resolve_algo(c, count, t, DCC_ALGO_AUTO);
  return DCC_OK;
}

int dcc_debug_skip_signal(dcc_comm_t c, int rank) {
  if (!c || rank < -1 || rank >= c->n) return DCC_ERR_INVALID_ARG;
  c->dev.skip_signal_rank = rank;
  return DCC_OK;
}

int dcc_launch_shape(dcc_comm_t c, size_t count, dcc_dtype_t t, dcc_algo_t a, int* blocks,
                     int* threads) {
  if (!c || !blocks || !threads || elem_bytes(t) == 0) return DCC_ERR_INVALID_ARG;
  *blocks = 0;
  *threads = 0;
  if (count == 0) return DCC_OK;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  Shape sh;
  const int rc = allreduce_shape(c, count, t, resolve_algo(c, count, t, a), false, &sh);
  if (rc != DCC_OK) return rc;
  *blocks = sh.blocks;
  *threads = sh.threads;
  return DCC_OK;
}

}  // extern "C"
