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
constexpr size_t kSyncBytes = kSemBytes + kExpectBytes + kStatusBytes;  // cleared every call
constexpr size_t kArrayBytes = kSyncBytes + (size_t)DCC_NOALLOC_MAX_BYTES;
constexpr int kMaxDevices = 64;

// The working memory.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_array[kArrayBytes];

std::mutex g_mu;
unsigned char* g_base[kMaxDevices] = {};  // device address of g_noalloc_array per device
int g_sms[kMaxDevices] = {};

// Once per device, with that device current: resolve the array's device
// address (no allocation happens here; the array already exists).
int setup_device(int dev, unsigned char** base, int* sms) {
  if (dev < 0 || dev >= kMaxDevices) return DCC_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_base[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_array) != cudaSuccess || !p) {
      cudaGetLastError();
      return DCC_ERR_CUDA;
    }
    int n_sms = 0;
    if (cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return DCC_ERR_CUDA;
    }
    g_base[dev] = static_cast<unsigned char*>(p);
    g_sms[dev] = n_sms;
  }
  *base = g_base[dev];
  *sms = g_sms[dev];
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
  unsigned char* base = nullptr;
  int sms = 0;
  int rc = setup_device(dev, &base, &sms);
  if (rc != DCC_OK) return rc;

  const void* fn = scratch_kernel(t, n_ranks);
  int per_sm = 0;
  if (!fn || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, dcc::kThreads, 0) !=
                 cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  int bmax = per_sm * sms / n_ranks;
  if (bmax > DCC_MAX_BLOCKS_PER_RANK) bmax = DCC_MAX_BLOCKS_PER_RANK;
  if (bmax < 1) return DCC_ERR_LAUNCH;
  const size_t vw = 16 / eb;
  const size_t work = count / vw / (size_t)n_ranks + 1;
  const size_t want = (work + dcc::kThreads - 1) / dcc::kThreads;
  const int blocks = want > (size_t)bmax ? bmax : (int)(want < 1 ? 1 : want);

  dcc::DevComm dc{};
  dc.n = n_ranks;
  dc.skip_signal_rank = -1;
  dc.timeout_ns = 2000000ull * 1000ull;
  if (const char* v = std::getenv("DCC_WAIT_TIMEOUT_US")) {
    const unsigned long long us = std::strtoull(v, nullptr, 10);
    if (us > 0) dc.timeout_ns = us * 1000ull;
  }
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

  cudaStream_t st = static_cast<cudaStream_t>(s);
  // Counters, waiter counts and status start at zero for every call: the
  // array keeps whatever the previous call (on any stream) left there.
  if (cudaMemsetAsync(base, 0, kSyncBytes, st) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
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
