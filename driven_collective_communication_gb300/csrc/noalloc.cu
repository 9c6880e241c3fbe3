// noalloc.cu -- an AllReduce entry point that allocates no device memory.
//
// Some callers cannot call cudaMalloc at the point where they need an
// AllReduce: a framework whose caching allocator has reserved the GPU's
// memory up front and forbids side allocations, a latency-critical serving
// loop where cudaMalloc's implicit device synchronisation is not acceptable,
// or a deployment that must fit a fixed, audited memory budget.  Such callers
// cannot create a communicator (dcc_comm_create allocates its semaphore block
// and channel table).  dcc_allreduce_noalloc gives them the two-shot
// AllReduce through scratch with every piece of working memory -- the
// reduced shards, the semaphores, the waiters' counters and the status word
// -- in one file-scope device array of fixed size, which the CUDA runtime
// places on each GPU when the library's module is loaded there and keeps
// until the process exits.
//
// The kernel is the communicator path's k_allreduce_twoshot_scratch,
// unchanged: only where its memory comes from differs.
//
// No per-call clearing: in a call that completes, every semaphore slot the
// kernel uses receives exactly one signal and is waited on exactly once, so
// each slot's signal count equals its waiter count again afterwards, whatever
// the rank count or launch shape of the next call.  Only a wait that ran out
// breaks that balance; it also records itself in the status word, and
// dcc_noalloc_check, which reports it, zeroes the whole synchronisation part
// of the array so that the next call starts balanced.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "collectives.cuh"
#include "dcc.h"
#include "dcc_internal.h"

namespace {

constexpr size_t kSemBytes = dcc::kSemSlots * dcc::kSemWords * sizeof(unsigned long long);
constexpr size_t kExpectBytes = dcc::kSemSlots * sizeof(unsigned long long);
constexpr size_t kStatusBytes = 256;
constexpr size_t kSyncBytes = kSemBytes + kExpectBytes + kStatusBytes;
constexpr size_t kArrayBytes = kSyncBytes + (size_t)DCC_NOALLOC_MAX_BYTES;
constexpr int kMaxDevices = 64;

// The working memory.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_array[kArrayBytes];

std::mutex g_mu;
struct DeviceState {
  unsigned char* base = nullptr;  // device address of g_noalloc_array on this device
  int sms = 0;
  unsigned long long timeout_ns = 0;
  int skip_signal_rank = -1;
  int per_sm[4][DCC_MAX_RANKS + 1] = {};  // resident CTAs per SM by (dtype, n); 0 = not yet queried
};
DeviceState g_dev[kMaxDevices];

// Once per device, with that device current: resolve the array's device
// address (no allocation happens here; the array already exists), zero its
// synchronisation part, and read the wait limit and the test knob from the
// environment.
int setup_device(int dev, DeviceState** out) {
  if (dev < 0 || dev >= kMaxDevices) return DCC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.base) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_array) != cudaSuccess || !p) {
      cudaGetLastError();
      return DCC_ERR_CUDA;
    }
    int n_sms = 0;
    if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaMemset(p, 0, kSyncBytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaGetLastError();
      return DCC_ERR_CUDA;
    }
    d.timeout_ns = 2000000ull * 1000ull;
    if (const char* v = std::getenv("DCC_WAIT_TIMEOUT_US")) {
      const unsigned long long us = std::strtoull(v, nullptr, 10);
      if (us > 0) d.timeout_ns = us * 1000ull;
    }
    // test knob: this rank sends no signals, so its peers' waits run out
    if (const char* v = std::getenv("DCC_NOALLOC_SKIP_SIGNAL")) d.skip_signal_rank = std::atoi(v);
    d.sms = n_sms;
    d.base = static_cast<unsigned char*>(p);
  }
  *out = &d;
  return DCC_OK;
}

const void* scratch_kernel(dcc_dtype_t t, int n) {
  switch (t) {
    case DCC_INT32: return dcc::reduce_kernel<int32_t>(dcc::kTwoShotScratch, n);
    case DCC_FP32: return dcc::reduce_kernel<float>(dcc::kTwoShotScratch, n);
    case DCC_FP16: return dcc::reduce_kernel<__half>(dcc::kTwoShotScratch, n);
    case DCC_BF16: return dcc::reduce_kernel<__nv_bfloat16>(dcc::kTwoShotScratch, n);
    default: return nullptr;
  }
}

// the bounds-checked build's extent of pointer `rank` of buffer `kind`
void dcc_set_extent_(dcc::CollArgs& a, int kind, int rank, size_t bytes) {
#if DCC_CHECK_BOUNDS
  a.ext[kind][rank] = bytes;
#else
  (void)a; (void)kind; (void)rank; (void)bytes;
#endif
}

size_t elem_size(dcc_dtype_t t) {
  return (t == DCC_INT32 || t == DCC_FP32) ? 4 : (t == DCC_FP16 || t == DCC_BF16) ? 2 : 0;
}

bool ranges_overlap(const void* a, const void* b, size_t n) {
  const char* x = static_cast<const char*>(a);
  const char* y = static_cast<const char*>(b);
  return n && x < y + n && y < x + n;
}

}  // namespace

extern "C" int dcc_allreduce_noalloc(int n_ranks, void* const* send, void* const* recv,
                                     size_t count, dcc_dtype_t t, dcc_stream_t s) {
  const size_t eb = elem_size(t);
  if (n_ranks < 1 || n_ranks > DCC_MAX_RANKS || !send || !recv || eb == 0)
    return DCC_ERR_INVALID_ARG;
  if (count == 0) return DCC_OK;
  if (count > (size_t)DCC_NOALLOC_MAX_BYTES / eb) return DCC_ERR_UNSUPPORTED;  // beyond the array
  const size_t bytes = count * eb;
  for (int r = 0; r < n_ranks; ++r) {
    if (!send[r] || !recv[r]) return DCC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(send[r]) | reinterpret_cast<uintptr_t>(recv[r])) & 15u)
      return DCC_ERR_MISALIGNED;
  }
  bool inplace = false;
  for (int r = 0; r < n_ranks; ++r)
    for (int p = 0; p < n_ranks; ++p) {
      if (ranges_overlap(recv[r], send[p], bytes)) {
        if (r != p || recv[r] != send[r]) return DCC_ERR_INVALID_ARG;
        inplace = true;
      }
      if (p != r && ranges_overlap(recv[r], recv[p], bytes)) return DCC_ERR_INVALID_ARG;
    }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  DeviceState* d = nullptr;
  int rc = setup_device(dev, &d);
  if (rc != DCC_OK) return rc;
  unsigned char* base = d->base;

  const void* fn = scratch_kernel(t, n_ranks);
  if (!fn) return DCC_ERR_INVALID_ARG;
  int per_sm;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    per_sm = d->per_sm[t][n_ranks];
  }
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, dcc::kThreads, 0) != cudaSuccess) {
      cudaGetLastError();
      return DCC_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    d->per_sm[t][n_ranks] = per_sm;
  }
  int bmax = per_sm * d->sms / n_ranks;
  if (bmax > DCC_MAX_BLOCKS_PER_RANK) bmax = DCC_MAX_BLOCKS_PER_RANK;
  if (bmax < 1) return DCC_ERR_LAUNCH;
  const size_t vw = 16 / eb;
  const size_t work = count / vw / (size_t)n_ranks + 1;
  const size_t want = (work + dcc::kThreads - 1) / dcc::kThreads;
  const int blocks = want > (size_t)bmax ? bmax : (int)(want < 1 ? 1 : want);

  dcc::DevComm dc{};
  dc.n = n_ranks;
  dc.skip_signal_rank = d->skip_signal_rank;
  dc.timeout_ns = d->timeout_ns;
  dc.sem = reinterpret_cast<unsigned long long*>(base);
  dc.expect = reinterpret_cast<unsigned long long*>(base + kSemBytes);
  dc.status = reinterpret_cast<unsigned long long*>(base + kSemBytes + kExpectBytes);

  dcc::CollArgs a{};
  unsigned char* scratch = base + kSyncBytes;
  const size_t nvec = count / vw, per = nvec / (size_t)n_ranks;
  for (int r = 0; r < n_ranks; ++r) {
    a.send[r] = send[r];
    a.recv[r] = recv[r];
    a.scratch[r] = scratch + per * (size_t)r * 16;  // rank r's shard, 16-byte aligned
  }
  a.count = count;
  a.blocks = blocks;
  a.inplace = inplace ? 1 : 0;
  for (int r = 0; r < n_ranks; ++r) {
    dcc_set_extent_(a, dcc::kBufSend, r, bytes);
    dcc_set_extent_(a, dcc::kBufRecv, r, bytes);
    // rank r's shard: `per` vectors, the last rank also the remaining vectors and the element tail
    dcc_set_extent_(a, dcc::kBufScratch, r, r == n_ranks - 1 ? bytes - per * (size_t)r * 16 : per * 16);
  }

  cudaStream_t st = static_cast<cudaStream_t>(s);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks * n_ranks));
  cfg.blockDim = dim3((unsigned)dcc::kThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = n_ranks > 1 ? 1 : 0;
  void* kargs[] = {&dc, &a};
  const cudaError_t e = cudaLaunchKernelExC(&cfg, fn, kargs);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    cudaGetLastError();
    return DCC_ERR_LAUNCH;
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  return DCC_OK;
}

extern "C" int dcc_noalloc_check(dcc_stream_t s, int* rank, int* peer, int* block) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  DeviceState* d = nullptr;
  const int rc = setup_device(dev, &d);
  if (rc != DCC_OK) return rc;
  unsigned long long st = 0;
  unsigned char* status = d->base + kSemBytes + kExpectBytes;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(s)) != cudaSuccess ||
      cudaMemcpy(&st, status, sizeof st, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  if (st == 0) return DCC_OK;
  if (rank) *rank = (int)((st >> 8) & 0xFF);
  if (peer) *peer = (int)((st >> 16) & 0xFF);
  if (block) *block = (int)((st >> 24) & 0xFFFF);
  // the semaphores are unbalanced after a wait gave up: start again from zero
  if (cudaMemset(d->base, 0, kSyncBytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  return DCC_ERR_TIMEOUT;
}
