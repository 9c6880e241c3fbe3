// comm.h -- the communicator object and host helpers shared by the host
// translation units of libdcc (dcc_host.cu, proxy.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <map>
#include <tuple>
#include <unordered_map>
#include <vector>

#include "dcc.h"
#include "dcc_internal.h"
#include "dcc_tuning.h"

struct ProxyState;  // proxy.cu
struct dcc_comm;
void dcc_proxy_release(dcc_comm* c);  // proxy.cu: stops the proxy thread and frees its state
int dcc_preload_kernels();            // dcc_host.cu: loads every collective kernel now

namespace dcc_host {
struct Window {
  char* ptr;
  size_t bytes;
};

inline size_t elem_bytes(dcc_dtype_t t) {
  switch (t) {
    case DCC_INT32: case DCC_FP32: return 4;
    case DCC_FP16: case DCC_BF16: return 2;
    default: return 0;
  }
}

inline bool env_flag(const char* name) {
  const char* v = std::getenv(name);
  return v && *v && std::strcmp(v, "0") != 0;
}

// Messages at or below this many bytes per rank run one-shot under AUTO, by
// rank count and dtype: the measured crossover table (the JSON file under
// tuning/, turned into dcc_tuning.h by the build).
inline size_t default_one_shot_max(int n_ranks, dcc_dtype_t t) {
  if (n_ranks < 1 || n_ranks > DCC_MAX_RANKS || (int)t < 0 || (int)t > 3) return 0;
  return (size_t)kOneShotMaxTable[n_ranks][(int)t];
}

// Threads per CTA of the thread-copy kernels, by work (16-byte vectors per
// rank): small messages want many small CTAs spread over many SMs (latency),
// large ones one full wave of 512-thread CTAs (bandwidth).  Measured on GB300
// over 16 KiB .. 4 MiB per rank.
inline int threads_for(dcc_algo_t algo, size_t work_vecs_per_rank) {
  if (algo == DCC_ALGO_ONE_SHOT) return work_vecs_per_rank <= 65536 ? 128 : 512;
  if (work_vecs_per_rank <= 8192) return 64;
  if (work_vecs_per_rank <= 65536) return 128;
  return 512;
}

// Host-buffer AllReduce: elements per rank per pipeline chunk (8 MiB of bf16).
constexpr size_t kPipeChunkBytes = 8u << 20;

// Fused linear + AllReduce: rows of at least this many elements per rank
// stream through the bulk-copy kernel (fused_bulk.cuh), shorter ones through
// thread loads (fused.cuh).  Measured on GB300, 8 ranks x 8192 rows bf16,
// thread / bulk (us): kp 2048 46.7 / 62.7, 2560 58.9 / 67.2, 3072 68.0 / 70.6,
// 3584 79.1 / 75.1, 4096 87.3 / 80.5, 8192 169 / 152.
constexpr size_t kFusedBulkMinKp = 3584;

// One-token fused linear + AllReduce: kp up to this runs on the tensor-core
// kernel (the batched layer with one token, pair form).
// Measured on GB300, 8 ranks x 8192 rows bf16, tensor-core / thread-load /
// bulk-copy kernel (us; one weight set reused by every call, which at kp 1024
// stays partly in L2: 22.5 us for the tensor-core kernel with two sets
// alternating): kp 1024 20.9 / 25.1 / 53.4, 2048 40.5 / 44.1 / 60.3,
// 3584 69.4 / 74.4 / 71.6, 4096 80.2 / 82.5 / 78.1, 6144 118.3 / 121.3 /
// 119.5, 8192 155.9 / 159.9 / 149.1; kp not a multiple of 64 (two weight
// sets alternating), tensor-core / thread-load: 1000 22.8 / 25.1, 1016
// 23.0 / 25.1, 1960 41.7 / 43.6, 3576 73.2 / 74.5.
constexpr size_t kFusedTensorMaxKp = 3584;

// Tensor-core layer over a batch of tokens, its forms: "pair" (128-thread
// CTAs, two per SM, one accumulator), "one" (256-thread CTAs, one per SM,
// one accumulator), "two" (the same with two accumulators sharing each token
// tile).  With no form requested the library plans the forms and runs the
// better plan (plan_mma, better_plan).  Measured on GB300, 8 ranks x 8192
// rows x kp 1024 bf16, pair / one / two (us): 1 token 21.0 / 28.0 / 24.4,
// 32 tokens 22.8 / 28.4 / 25.8, 96 tokens 27.9 / 29.8 / 31.0, 128 tokens
// 31.3 (4-way split, epilogue in two rounds) / 30.6 / 33.3, 160 tokens 33.6
// / 31.8 / 35.6, 256 tokens 42.0 (one CTA per SM: the token tile leaves no
// room for two) / 36.5 / 48.8.
enum { kMmaFormPair = 0, kMmaFormOne = 1, kMmaFormTwo = 2 };

// A launch plan of the tensor-core layer for one form (kMmaForm*): the kernel,
// its threads, accumulators, stages and shared memory, the tile height bm and
// K split ks, the epilogue's rounds, and whether the grid fits one wave.
struct MmaPlan {
  int rc = DCC_OK;
  const void* fn = nullptr;
  int threads = 0, macc = 1, stages = 0, bm = 0, ks = 1, rounds = 1;
  size_t smem = 0;
  bool one_wave = false;
};

// AllGather inputs of at least this many bytes per rank use the bulk-copy kernel.
constexpr size_t kAgBulkMinBytes = 64 * 1024;

}  // namespace dcc_host

struct dcc_comm {
  int n = 0;
  int device = 0;
  int num_sms = 0;
  int smem_per_sm = 0;       // shared memory per SM and reserved per CTA, bytes
  int smem_reserved_cta = 0;
  std::vector<dcc_host::Window> win[DCC_MAX_RANKS][3];
  bool chan[DCC_MAX_RANKS][DCC_MAX_RANKS] = {};
  bool table_dirty = true;
  dcc::DevChannel h_table[DCC_MAX_RANKS * DCC_MAX_RANKS] = {};
  dcc::DevChannel* d_table = nullptr;
  unsigned long long* d_block = nullptr;  // sem | expect | status | LL epochs
  char* d_ll = nullptr;                   // LL packet buffers
  dcc::DevComm dev{};
  int blocks_override = 0;
  int threads_override = 0;  // threads per CTA of the thread-copy kernels (0 = by size)
  size_t one_shot_max[4] = {};  // set from the rank count at creation
  int forced_algo = -1;  // DCC_ALGO environment override of AUTO
  // AUTO: messages of at least bulk_min_bytes per rank run large_algo
  size_t bulk_min_bytes = (size_t)1 << 62;
  dcc_algo_t large_algo = DCC_ALGO_TWO_SHOT;
  // kernel of the one-token fused linear + AllReduce: -1 by kp (measured
  // crossovers), 0 thread loads, 1 bulk copies (DCC_FUSED_BULK=0 / 1), 2 the
  // tensor-core kernel where kp allows (DCC_FUSED_KERNEL=thread|bulk|tensor)
  int fused_kernel = -1;
  // tensor-core layer: its form (kMmaForm*), -1 by token count (DCC_MMA_FORM)
  int mma_form = -1;
  bool entry_barrier = false;  // DCC_ENTRY_BARRIER / dcc_set_entry_barrier
  bool pdl = true;             // DCC_PDL / dcc_set_pdl: programmatic dependent launch of the wait-free kernels
  bool ring_cluster = true;    // DCC_RING_CLUSTER=0: the ring barrier through L2 even when the ranks fit one cluster
  int inplace_unroll = 0;      // DCC_INPLACE_UNROLL: force the in-place one-shot's vectors per thread
  bool ag_bulk = false;  // DCC_AG_BULK=1: AllGather through the bulk-copy pipeline when aligned and large
  bool zero_copy = true;  // host-buffer AllReduce reads/writes mapped pinned host memory directly
  int sticky = DCC_OK;
  int err_rank = -1, err_peer = -1, err_block = -1;
  bool log = false;
  // host-buffer pipeline (created on first use): copy-in and copy-out streams
  // and the events that chain them to the caller's stream
  bool pipe_ready = false;
  cudaStream_t pipe_in = nullptr, pipe_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in = nullptr, ev_kernel = nullptr, ev_done = nullptr;
  ProxyState* proxy = nullptr;  // PortChannel proxy (created by dcc_proxy_start)
  // tensor maps of the tensor-core linear layer, by (pointer, inner extent,
  // outer extent, box rows, element type); encoded on the host once
  struct MapKey {
    const void* ptr;
    unsigned long long inner, outer;
    unsigned box_rows, dtype;
    bool operator==(const MapKey& o) const {
      return ptr == o.ptr && inner == o.inner && outer == o.outer && box_rows == o.box_rows && dtype == o.dtype;
    }
  };
  struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
      return std::hash<const void*>()(k.ptr) ^ (std::hash<unsigned long long>()(k.inner * 1315423911ull + k.outer) << 1) ^
             ((size_t)k.box_rows << 20) ^ k.dtype;
    }
  };
  std::unordered_map<MapKey, CUtensorMap, MapKeyHash> tmaps;
  // clusters of the tensor-core layer that fit on the device at once, by
  // (kernel, cluster size, dynamic shared memory); 0 = not measured yet
  std::map<std::tuple<const void*, int, size_t>, int> mma_clusters;
  // launch plans of the tensor-core layer by (form, token tile, rows, kp, residual)
  std::map<std::tuple<int, int, size_t, size_t, bool>, dcc_host::MmaPlan> mma_plans;
};

namespace dcc_host {

// Makes the communicator's device current for the scope of a call (and puts
// the caller's device back only if it had to change it).
class DeviceScope {
 public:
  explicit DeviceScope(int dev) {
    if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
    if (prev_ != dev) {
      ok_ = cudaSetDevice(dev) == cudaSuccess;
      changed_ = ok_ && prev_ >= 0;
    }
  }
  ~DeviceScope() {
    if (changed_) cudaSetDevice(prev_);
  }
  bool ok() const { return ok_; }

 private:
  int prev_ = -1;
  bool ok_ = true;
  bool changed_ = false;
};

// Resident CTAs per SM of `fn` with `threads` threads and `smem` bytes of
// dynamic shared memory (raising the kernel's dynamic shared-memory limit the
// first time).  Cached per (kernel, smem, threads).
inline int max_active_per_sm(const void* fn, int threads, size_t smem = 0) {
  static std::mutex mu;
  static std::unordered_map<const void*, std::unordered_map<size_t, int>> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto& per_fn = cache[fn];
  const size_t key = smem * 2048 + (size_t)threads;
  auto it = per_fn.find(key);
  if (it != per_fn.end()) return it->second;
  int nb = 0;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fn, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  per_fn[key] = nb;
  return nb;
}

inline bool in_window(const dcc_comm* c, int rank, int kind, const void* p, size_t bytes) {
  const char* q = static_cast<const char*>(p);
  for (const Window& w : c->win[rank][kind])
    if (q >= w.ptr && bytes <= w.bytes && (size_t)(q - w.ptr) <= w.bytes - bytes) return true;
  return false;
}

inline bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
  const char* x = static_cast<const char*>(a);
  const char* y = static_cast<const char*>(b);
  return an && bn && x < y + bn && y < x + an;
}

// Checks the send/recv arrays of a collective.  inplace_ok: send[r] == recv[r]
// (same byte count) is allowed.  Reports whether any rank is in place.
inline int check_buffers(const dcc_comm* c, void* const* send, size_t send_bytes, void* const* recv,
                  size_t recv_bytes, bool inplace_ok, bool* any_inplace) {
  if (!send || !recv) return DCC_ERR_INVALID_ARG;
  *any_inplace = false;
  for (int r = 0; r < c->n; ++r) {
    if (!send[r] || !recv[r]) return DCC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(send[r]) | reinterpret_cast<uintptr_t>(recv[r])) & 15u)
      return DCC_ERR_MISALIGNED;
    if (!in_window(c, r, DCC_BUF_INPUT, send[r], send_bytes) &&
        !in_window(c, r, DCC_BUF_OUTPUT, send[r], send_bytes))
      return DCC_ERR_NOT_REGISTERED;
    if (!in_window(c, r, DCC_BUF_INPUT, recv[r], recv_bytes) &&
        !in_window(c, r, DCC_BUF_OUTPUT, recv[r], recv_bytes))
      return DCC_ERR_NOT_REGISTERED;
  }
  for (int r = 0; r < c->n; ++r) {
    for (int p = 0; p < c->n; ++p) {
      if (overlaps(recv[r], recv_bytes, send[p], send_bytes)) {
        const bool same = r == p && recv[r] == send[r] && send_bytes == recv_bytes;
        if (!(inplace_ok && same)) return DCC_ERR_INVALID_ARG;
        *any_inplace = true;
      }
      if (p != r && overlaps(recv[r], recv_bytes, recv[p], recv_bytes)) return DCC_ERR_INVALID_ARG;
    }
  }
  return DCC_OK;
}

// Bounds-checked build (DCC_CHECK_BOUNDS): the bytes a kernel may touch from
// pointer `rank` of buffer `kind` -- the call's own range, which the host
// checks already lies inside a registered window.  A no-op otherwise.
template <typename A>
inline void set_extent(A& a, int kind, int rank, size_t bytes) {
#if DCC_CHECK_BOUNDS
  a.ext[kind][rank] = bytes;
#else
  (void)a; (void)kind; (void)rank; (void)bytes;
#endif
}

// pdl: launch with programmatic stream serialization (only kernels that open
// with pdl_prologue() and whose CTAs never wait on one another; never together
// with a cooperative launch).
// cluster > 0: thread-block clusters of that many CTAs along x (grid a
// multiple of it; never with cooperative, may go with pdl).
inline int launch(const void* fn, int grid, int threads, bool cooperative, void** args, cudaStream_t s,
           size_t smem = 0, bool pdl = false, int cluster = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  unsigned na = 0;
  if (cluster > 0) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  } else if (pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = na ? attr : nullptr;
  cfg.numAttrs = na;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
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

}  // namespace dcc_host
