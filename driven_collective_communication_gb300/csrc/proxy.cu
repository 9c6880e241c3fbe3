// proxy.cu -- PortChannel host proxy: FIFO, proxy thread, and the kernels and
// C entry points that use PortChannels.
//
// MSCCL++ README, "Host-Side Communication Proxy": a host thread keeps
// checking for triggers that GPU threads have posted and does what each one
// asks (started and stopped around the application's kernels); a custom
// proxy replaces the trigger handling.  "PortChannel and MemoryChannel": the
// proxy performs the transfer with cudaMemcpy* (InfiniBand verbs between
// nodes -- not on one GPU) and the synchronisation.
//
// GB300 reading: the FIFO lives in pinned host memory mapped into the GPU's
// address space (Grace and the GPU share it coherently over NVLink-C2C); the
// proxy issues cudaMemcpyAsync device-to-device on the copy engines and
// reports signals and flushes back with 64-bit value writes
// (cuStreamWriteValue64) into device memory that the GPU polls.  Copies and
// signals to rank d go to proxy stream d % K, so stream order puts every
// signal behind the copies of its channel, and K copy engines work at once; a
// flush is written after every stream's earlier work (events).  K is 4 by
// default (DCC_PROXY_STREAMS, 1..8): measured on GB300 for the 8 x 8 MiB fp16
// AllGather, 0.573 / 0.345 / 0.253 / 0.281 ms with K = 1 / 2 / 4 / 8.  Signal
// writes queue per stream and go out together (one batch of stream memory
// operations) when the FIFO runs empty, after 256 triggers, or before a flush
// or a custom trigger: fewer host calls when one thread issues everything
// (K = 1: 0.573 -> 0.473 ms), the same with K = 4, where the copy engines
// bound it.  Every wait on either side is bounded.
//
// The kernels that push triggers keep running while the proxy's streams work
// for them.  If the GPU multiplexes a proxy stream onto the same hardware
// queue as the pushing kernel's stream (an application with more streams than
// CUDA_DEVICE_MAX_CONNECTIONS), the proxy's work queues behind that kernel and
// its waits run out: run PortChannel code with enough connections.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <thread>
#include <vector>

#include "comm.h"
#include "port_channel.cuh"

using dcc_host::DeviceScope;

typedef void (*dcc_trigger_handler_t)(uint64_t fst, uint64_t snd, void* user);

namespace {

constexpr unsigned long long kFifoCapacity = 1024;
constexpr int kMaxCustom = 32;
constexpr int kMaxProxyStreams = 8;

typedef CUresult (*WriteValue64Fn)(CUstream, CUdeviceptr, cuuint64_t, unsigned int);
typedef CUresult (*BatchMemOpFn)(CUstream, unsigned int, CUstreamBatchMemOpParams*, unsigned int);
constexpr int kMaxTakePerRound = 256;  // triggers the proxy takes from the FIFO in one round

}  // namespace

struct ProxyState {
  std::thread thread;
  std::atomic<bool> stop{false};
  std::atomic<unsigned long long> drain_to{0};  // on stop: take triggers up to this sequence
  bool running = false;
  // FIFO: slots + tail in one pinned, mapped host allocation
  unsigned char* h_fifo = nullptr;
  dcc::ProxyTrigger* h_slots = nullptr;
  unsigned long long* h_tail = nullptr;
  unsigned char* d_fifo = nullptr;  // device address of h_fifo
  // device words: head | done | sem[kSemSlots*kSemWords] | expect[kSemSlots]
  unsigned long long* d_words = nullptr;
  dcc::PortDev dev{};
  // Copies and signals to rank d go to streams[d % nstreams], in FIFO order
  // per stream; a flush is written on streams[0] after the work of every
  // stream that had some since the previous flush (events).
  int nstreams = 4;
  cudaStream_t streams[kMaxProxyStreams] = {};
  cudaEvent_t events[kMaxProxyStreams] = {};
  bool dirty[kMaxProxyStreams] = {};
  unsigned long long sig_count[DCC_MAX_RANKS][DCC_MAX_RANKS] = {};
  WriteValue64Fn write_value = nullptr;
  BatchMemOpFn batch_mem_op = nullptr;
  // signal writes waiting to be issued, per stream: the values go out together
  // (one stream memory-operation batch per stream) after the round's copies
  std::vector<CUstreamBatchMemOpParams> pending[kMaxProxyStreams];
  dcc_trigger_handler_t handler = nullptr;
  void* user = nullptr;
  std::atomic<unsigned long long> processed{0}, custom{0};
  std::atomic<int> error{DCC_OK};
};

namespace {

// ------------------------------------------------------------------ kernels
struct PortPutArgs {
  int src, dst;
  size_t remote_off, local_off, bytes;
  int signal, flush;
};

__global__ void k_port_put(dcc::DevComm dc, dcc::PortDev pd, PortPutArgs pa) {
  if (threadIdx.x != 0) return;
  const dcc::PortChannel ch{pd, pa.src, pa.dst};
  if (blockIdx.x == 0) {
    unsigned long long seq;
    if (!ch.put(pa.remote_off, pa.local_off, pa.bytes, pa.signal ? dcc::kTrigSignal : 0, seq, dc)) return;
    if (pa.flush) ch.flush(dc);
  } else if (pa.signal) {
    ch.wait(dc);
  }
}

struct PortAgArgs {
  size_t send_off[DCC_MAX_RANKS];  // byte offset of send[q] in rank q's first INPUT window
  size_t recv_off[DCC_MAX_RANKS];  // byte offset of recv[p] in rank p's first OUTPUT window
  size_t bytes;                    // per-rank input bytes (multiple of 16)
};

// AllGather through PortChannels: one thread per rank.  Rank q asks the proxy
// to copy its input into slot q of every output (its own included), each copy
// to a peer carrying a signal; then it flushes (its own copy is done) and
// waits for the N-1 peers' signals (their copies into its output are done).
__global__ void k_port_allgather(dcc::DevComm dc, dcc::PortDev pd, PortAgArgs a) {
  if (threadIdx.x != 0) return;
  const int n = dc.n, q = blockIdx.x;
  bool ok = true;
  for (int i = 0; i < n && ok; ++i) {
    const int p = (q + i) % n;  // stagger destinations across ranks
    unsigned long long seq;
    ok = dcc::PortChannel{pd, q, p}.put(a.recv_off[p] + (size_t)q * a.bytes, a.send_off[q], a.bytes,
                                        p == q ? 0 : dcc::kTrigSignal, seq, dc);
  }
  if (ok) ok = dcc::PortChannel{pd, q, q}.flush(dc);
  for (int i = 1; i < n && ok; ++i) ok = dcc::PortChannel{pd, (q + i) % n, q}.wait(dc);
}

struct CustomArgs {
  int count;
  dcc::ProxyTrigger t[kMaxCustom];
};

// The README's custom-proxy example: one thread pushes user-defined triggers.
__global__ void k_fifo_push(dcc::DevComm dc, dcc::PortDev pd, CustomArgs a) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  for (int i = 0; i < a.count; ++i) {
    unsigned long long seq;
    if (!dcc::fifo_push(pd, a.t[i], seq, dc, 0)) return;
  }
}

// ------------------------------------------------------------------ proxy thread
void set_error(ProxyState& P, int code) {
  int expected = DCC_OK;
  P.error.compare_exchange_strong(expected, code);
}

bool window_range(const dcc_comm* c, int rank, int kind, size_t off, size_t bytes, char** p) {
  if (c->win[rank][kind].empty()) return false;
  const dcc_host::Window& w = c->win[rank][kind][0];
  if (off > w.bytes || bytes > w.bytes - off) return false;
  *p = w.ptr + off;
  return true;
}

// Issue the signal writes queued on each stream: a single write as is, several
// as one batch of stream memory operations (in queue order).
void issue_pending_signals(ProxyState& P) {
  for (int k = 0; k < P.nstreams; ++k) {
    std::vector<CUstreamBatchMemOpParams>& q = P.pending[k];
    if (q.empty()) continue;
    CUresult r = CUDA_SUCCESS;
    if (q.size() == 1 || !P.batch_mem_op) {
      for (size_t i = 0; i < q.size() && r == CUDA_SUCCESS; ++i)
        r = P.write_value((CUstream)P.streams[k], q[i].writeValue.address, q[i].writeValue.value64,
                          CU_STREAM_WRITE_VALUE_DEFAULT);
    } else {
      r = P.batch_mem_op((CUstream)P.streams[k], (unsigned)q.size(), q.data(), 0);
    }
    if (r != CUDA_SUCCESS) set_error(P, DCC_ERR_CUDA);
    q.clear();
  }
}

void handle(dcc_comm* c, ProxyState& P, unsigned long long fst, unsigned long long snd,
            unsigned long long seq) {
  P.processed.fetch_add(1, std::memory_order_relaxed);
  const auto t_start = std::chrono::steady_clock::now();
  struct LogOnExit {
    const dcc_comm* c;
    unsigned long long seq, fst, snd;
    std::chrono::steady_clock::time_point t0;
    ~LogOnExit() {  // DCC_LOG: report handler calls that took over 1 ms
      if (!c->log) return;
      const long long us = (long long)std::chrono::duration_cast<std::chrono::microseconds>(
                               std::chrono::steady_clock::now() - t0).count();
      if (us > 1000)
        std::fprintf(stderr, "dcc proxy: seq %llu fst %016llx snd %016llx took %lld us\n", seq, fst, snd, us);
    }
  } log_on_exit{c, seq, fst, snd, t_start};
  if (!(fst & dcc::kTrigBuiltin)) {
    P.custom.fetch_add(1, std::memory_order_relaxed);
    issue_pending_signals(P);  // the handler sees every earlier trigger carried out
    if (P.handler) P.handler(fst, snd, P.user);
    return;
  }
  const int src = (int)((fst >> 40) & 0xFF), dst = (int)((fst >> 48) & 0xFF);
  const size_t bytes = fst & dcc::kTrigSizeMask;
  const size_t dst_off = (size_t)(snd & 0xFFFFFFFFull) * 16, src_off = (size_t)(snd >> 32) * 16;
  if (src >= c->n || dst >= c->n) {
    set_error(P, DCC_ERR_INVALID_ARG);
    return;
  }
  const int k = dst % P.nstreams;
  cudaStream_t st = P.streams[k];
  if (fst & (dcc::kTrigPut | dcc::kTrigSignal)) P.dirty[k] = true;
  if (fst & dcc::kTrigPut) {
    char *d = nullptr, *s = nullptr;
    if (!window_range(c, dst, DCC_BUF_OUTPUT, dst_off, bytes, &d) ||
        !window_range(c, src, DCC_BUF_INPUT, src_off, bytes, &s)) {
      set_error(P, DCC_ERR_NOT_REGISTERED);  // skip the copy; signals/flushes still go out
    } else if (bytes && cudaMemcpyAsync(d, s, bytes, cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
      set_error(P, DCC_ERR_CUDA);
    }
  }
  if (fst & dcc::kTrigSignal) {  // queued behind this stream's copies of the round
    const unsigned long long v = ++P.sig_count[dst][src];
    CUstreamBatchMemOpParams op;
    std::memset(&op, 0, sizeof op);
    op.writeValue.operation = CU_STREAM_MEM_OP_WRITE_VALUE_64;
    op.writeValue.address = (CUdeviceptr)(P.dev.sem + dcc::sem_slot(dst, src, 0) * dcc::kSemWords);
    op.writeValue.value64 = v;
    op.writeValue.flags = CU_STREAM_WRITE_VALUE_DEFAULT;
    P.pending[k].push_back(op);
  }
  if (fst & dcc::kTrigFlush) {  // after everything issued so far, on every stream
    issue_pending_signals(P);
    for (int j = 1; j < P.nstreams; ++j) {
      if (!P.dirty[j]) continue;
      if (cudaEventRecord(P.events[j], P.streams[j]) != cudaSuccess ||
          cudaStreamWaitEvent(P.streams[0], P.events[j], 0) != cudaSuccess)
        set_error(P, DCC_ERR_CUDA);
      P.dirty[j] = false;
    }
    if (P.write_value((CUstream)P.streams[0], (CUdeviceptr)P.dev.done, seq + 1, CU_STREAM_WRITE_VALUE_DEFAULT) !=
        CUDA_SUCCESS)
      set_error(P, DCC_ERR_CUDA);
  }
}

void proxy_loop(dcc_comm* c) {
  ProxyState& P = *c->proxy;
  cudaSetDevice(c->device);
  unsigned long long tail = __atomic_load_n(P.h_tail, __ATOMIC_ACQUIRE);
  unsigned idle = 0;
  int taken = 0;  // triggers handled since the queued signal writes last went out
  bool draining = false;
  std::chrono::steady_clock::time_point deadline;
  for (;;) {
    if (P.stop.load(std::memory_order_acquire)) {
      // stopping: take what was pushed before the stop, but never wait forever
      if (!draining) {
        draining = true;
        deadline = std::chrono::steady_clock::now() + std::chrono::seconds(5);
      }
      if (tail >= P.drain_to.load(std::memory_order_relaxed) || std::chrono::steady_clock::now() > deadline)
        break;
    }
    dcc::ProxyTrigger* s = P.h_slots + (tail % kFifoCapacity);
    const unsigned long long fst = __atomic_load_n(&s->fst, __ATOMIC_ACQUIRE);
    if (fst == 0) {
      // the FIFO is empty for now: the round's queued signals go out
      if (taken) {
        issue_pending_signals(P);
        taken = 0;
      }
      if (++idle > 4096) std::this_thread::yield();
      continue;
    }
    idle = 0;
    const unsigned long long snd = __atomic_load_n(&s->snd, __ATOMIC_RELAXED);
    __atomic_store_n(&s->fst, 0ull, __ATOMIC_RELAXED);
    const unsigned long long seq = tail++;
    __atomic_store_n(P.h_tail, tail, __ATOMIC_RELEASE);
    handle(c, P, fst, snd, seq);
    if (++taken >= kMaxTakePerRound) {  // a steady stream of triggers still gets its signals
      issue_pending_signals(P);
      taken = 0;
    }
  }
  issue_pending_signals(P);
}

int ensure_proxy(dcc_comm* c) {
  if (c->proxy) return DCC_OK;
  ProxyState* P = new ProxyState();
  auto fail = [&](int code) {
    cudaGetLastError();
    if (P->h_fifo) cudaFreeHost(P->h_fifo);
    if (P->d_words) cudaFree(P->d_words);
    for (int j = 0; j < kMaxProxyStreams; ++j) {
      if (P->streams[j]) cudaStreamDestroy(P->streams[j]);
      if (P->events[j]) cudaEventDestroy(P->events[j]);
    }
    delete P;
    return code;
  };
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue64", &fn, 12000, cudaEnableDefault, &q) !=
          cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return fail(DCC_ERR_CUDA);
  P->write_value = reinterpret_cast<WriteValue64Fn>(fn);
  void* fb = nullptr;
  if (cudaGetDriverEntryPointByVersion("cuStreamBatchMemOp", &fb, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess && fb)
    P->batch_mem_op = reinterpret_cast<BatchMemOpFn>(fb);
  else
    cudaGetLastError();  // single writes then
  const size_t fifo_bytes = kFifoCapacity * sizeof(dcc::ProxyTrigger) + 64;
  if (cudaHostAlloc(reinterpret_cast<void**>(&P->h_fifo), fifo_bytes, cudaHostAllocMapped) != cudaSuccess)
    return fail(DCC_ERR_CUDA);
  std::memset(P->h_fifo, 0, fifo_bytes);
  if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&P->d_fifo), P->h_fifo, 0) != cudaSuccess)
    return fail(DCC_ERR_CUDA);
  P->h_slots = reinterpret_cast<dcc::ProxyTrigger*>(P->h_fifo);
  P->h_tail = reinterpret_cast<unsigned long long*>(P->h_fifo + kFifoCapacity * sizeof(dcc::ProxyTrigger));
  const size_t words = 2 + dcc::kSemSlots * dcc::kSemWords + dcc::kSemSlots + 14;
  if (cudaMalloc(&P->d_words, words * sizeof(unsigned long long)) != cudaSuccess ||
      cudaMemset(P->d_words, 0, words * sizeof(unsigned long long)) != cudaSuccess)
    return fail(DCC_ERR_CUDA);
  if (const char* v = std::getenv("DCC_PROXY_STREAMS")) {
    const int k = std::atoi(v);
    if (k >= 1 && k <= kMaxProxyStreams) P->nstreams = k;
  }
  for (int j = 0; j < P->nstreams; ++j)
    if (cudaStreamCreateWithFlags(&P->streams[j], cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&P->events[j], cudaEventDisableTiming) != cudaSuccess)
      return fail(DCC_ERR_CUDA);
  if (cudaDeviceSynchronize() != cudaSuccess) return fail(DCC_ERR_CUDA);
  P->dev.slots = reinterpret_cast<dcc::ProxyTrigger*>(P->d_fifo);
  P->dev.tail = reinterpret_cast<unsigned long long*>(P->d_fifo + kFifoCapacity * sizeof(dcc::ProxyTrigger));
  P->dev.head = P->d_words;
  P->dev.done = P->d_words + 1;
  P->dev.sem = P->d_words + 16;  // 128-byte aligned
  P->dev.expect = P->dev.sem + dcc::kSemSlots * dcc::kSemWords;
  P->dev.capacity = kFifoCapacity;
  c->proxy = P;
  return DCC_OK;
}

int require_running(const dcc_comm* c) {
  if (!c->proxy || !c->proxy->running) return DCC_ERR_INVALID_ARG;
  return DCC_OK;
}

int port_launch(dcc_comm* c, const void* fn, int grid, void** args, cudaStream_t s) {
  return dcc_host::launch(fn, grid, 32, true, args, s);
}

}  // namespace

// Frees the proxy (stopping its thread first); called by dcc_comm_destroy.
void dcc_proxy_release(dcc_comm* c) {
  if (!c->proxy) return;
  ProxyState* P = c->proxy;
  if (P->running) {
    P->drain_to.store(0);
    P->stop.store(true, std::memory_order_release);
    P->thread.join();
    P->running = false;
  }
  cudaDeviceSynchronize();
  for (int j = 0; j < kMaxProxyStreams; ++j) {
    if (P->streams[j]) cudaStreamDestroy(P->streams[j]);
    if (P->events[j]) cudaEventDestroy(P->events[j]);
  }
  cudaFree(P->d_words);
  cudaFreeHost(P->h_fifo);
  cudaGetLastError();
  delete P;
  c->proxy = nullptr;
}

extern "C" {

int dcc_proxy_start(dcc_comm_t c) {
  if (!c) return DCC_ERR_INVALID_ARG;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  int rc = ensure_proxy(c);
  if (rc != DCC_OK) return rc;
  // every kernel of the library loaded now, not at a first launch that could
  // stall the proxy behind a running PortChannel kernel
  rc = dcc_preload_kernels();
  if (rc != DCC_OK) return rc;
  cudaFuncAttributes attr;
  if (cudaFuncGetAttributes(&attr, reinterpret_cast<const void*>(&k_port_put)) != cudaSuccess ||
      cudaFuncGetAttributes(&attr, reinterpret_cast<const void*>(&k_port_allgather)) != cudaSuccess ||
      cudaFuncGetAttributes(&attr, reinterpret_cast<const void*>(&k_fifo_push)) != cudaSuccess) {
    cudaGetLastError();
    return DCC_ERR_CUDA;
  }
  ProxyState& P = *c->proxy;
  if (P.running) return DCC_OK;
  P.stop.store(false);
  P.thread = std::thread(proxy_loop, c);
  P.running = true;
  return DCC_OK;
}

int dcc_proxy_stop(dcc_comm_t c) {
  if (!c) return DCC_ERR_INVALID_ARG;
  if (!c->proxy || !c->proxy->running) return DCC_OK;
  ProxyState& P = *c->proxy;
  DeviceScope ds(c->device);
  // every trigger claimed so far (kernels that push must have finished)
  unsigned long long head = 0;
  if (cudaMemcpy(&head, P.dev.head, sizeof head, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    head = 0;
  }
  P.drain_to.store(head);
  P.stop.store(true, std::memory_order_release);
  P.thread.join();
  P.running = false;
  for (int j = 0; j < P.nstreams; ++j) cudaStreamSynchronize(P.streams[j]);
  return P.error.load();
}

int dcc_proxy_set_handler(dcc_comm_t c, dcc_trigger_handler_t fn, void* user) {
  if (!c) return DCC_ERR_INVALID_ARG;
  if (c->proxy && c->proxy->running) return DCC_ERR_INVALID_ARG;  // stop the proxy first
  DeviceScope ds(c->device);
  const int rc = ensure_proxy(c);
  if (rc != DCC_OK) return rc;
  c->proxy->handler = fn;
  c->proxy->user = user;
  return DCC_OK;
}

int dcc_proxy_state(dcc_comm_t c, uint64_t* words, int nwords) {
  if (!c || !c->proxy || !words || nwords < 6 + 2 * c->n * c->n) return DCC_ERR_INVALID_ARG;
  DeviceScope ds(c->device);
  ProxyState& P = *c->proxy;
  unsigned long long hd[2];
  if (cudaMemcpy(hd, P.dev.head, sizeof hd, cudaMemcpyDeviceToHost) != cudaSuccess) return DCC_ERR_CUDA;
  words[0] = hd[0];
  words[1] = __atomic_load_n(P.h_tail, __ATOMIC_ACQUIRE);
  words[2] = hd[1];
  words[3] = P.processed.load();
  words[4] = P.custom.load();
  words[5] = (uint64_t)(int64_t)P.error.load();
  for (int d = 0; d < c->n; ++d)
    for (int s = 0; s < c->n; ++s) {
      const size_t slot = dcc::sem_slot(d, s, 0);
      if (cudaMemcpy(&words[6 + d * c->n + s], P.dev.sem + slot * dcc::kSemWords, 8, cudaMemcpyDeviceToHost) !=
              cudaSuccess ||
          cudaMemcpy(&words[6 + c->n * c->n + d * c->n + s], P.dev.expect + slot, 8, cudaMemcpyDeviceToHost) !=
              cudaSuccess)
        return DCC_ERR_CUDA;
    }
  return DCC_OK;
}

int dcc_proxy_stats(dcc_comm_t c, uint64_t* processed, uint64_t* custom) {
  if (!c || !c->proxy) return DCC_ERR_INVALID_ARG;
  if (processed) *processed = c->proxy->processed.load();
  if (custom) *custom = c->proxy->custom.load();
  return c->proxy->error.load();
}

int dcc_port_put(dcc_comm_t c, int src, int dst, size_t remote_off, size_t local_off, size_t bytes,
                 int signal, int flush, dcc_stream_t s) {
  if (!c || src < 0 || dst < 0 || src >= c->n || dst >= c->n || src == dst) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  int rc = require_running(c);
  if (rc != DCC_OK) return rc;
  if (!c->chan[src][dst] || (signal && !c->chan[dst][src])) return DCC_ERR_NO_CHANNEL;
  if ((remote_off | local_off | bytes) & 15u) return DCC_ERR_MISALIGNED;
  if (bytes > dcc::kTrigSizeMask || remote_off / 16 > 0xFFFFFFFFull || local_off / 16 > 0xFFFFFFFFull)
    return DCC_ERR_INVALID_ARG;
  char* p;
  if (!window_range(c, src, DCC_BUF_INPUT, local_off, bytes, &p) ||
      !window_range(c, dst, DCC_BUF_OUTPUT, remote_off, bytes, &p))
    return DCC_ERR_NOT_REGISTERED;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  dcc::DevComm dc = c->dev;
  dcc::PortDev pd = c->proxy->dev;
  PortPutArgs pa{src, dst, remote_off, local_off, bytes, signal ? 1 : 0, flush ? 1 : 0};
  void* args[] = {&dc, &pd, &pa};
  return port_launch(c, reinterpret_cast<const void*>(&k_port_put), 2, args, static_cast<cudaStream_t>(s));
}

int dcc_port_allgather(dcc_comm_t c, void* const* send, void* const* recv, size_t send_count,
                       dcc_dtype_t t, dcc_stream_t s) {
  const size_t eb = dcc_host::elem_bytes(t);
  if (!c || eb == 0 || !send || !recv) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  int rc = require_running(c);
  if (rc != DCC_OK) return rc;
  if (send_count == 0) return DCC_OK;
  const size_t sb = send_count * eb, rb = sb * (size_t)c->n;
  if (sb % 16) return DCC_ERR_MISALIGNED;
  if (sb > dcc::kTrigSizeMask) return DCC_ERR_INVALID_ARG;
  PortAgArgs a{};
  for (int r = 0; r < c->n; ++r) {
    if (!send[r] || !recv[r]) return DCC_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(send[r]) | reinterpret_cast<uintptr_t>(recv[r])) & 15u)
      return DCC_ERR_MISALIGNED;
    if (c->win[r][DCC_BUF_INPUT].empty() || c->win[r][DCC_BUF_OUTPUT].empty()) return DCC_ERR_NOT_REGISTERED;
    const dcc_host::Window& wi = c->win[r][DCC_BUF_INPUT][0];
    const dcc_host::Window& wo = c->win[r][DCC_BUF_OUTPUT][0];
    const char* sp = static_cast<const char*>(send[r]);
    const char* rp = static_cast<const char*>(recv[r]);
    if (sp < wi.ptr || (size_t)(sp - wi.ptr) > wi.bytes || sb > wi.bytes - (size_t)(sp - wi.ptr) ||
        rp < wo.ptr || (size_t)(rp - wo.ptr) > wo.bytes || rb > wo.bytes - (size_t)(rp - wo.ptr))
      return DCC_ERR_NOT_REGISTERED;  // must lie in the rank's first INPUT / OUTPUT window
    a.send_off[r] = (size_t)(sp - wi.ptr);
    a.recv_off[r] = (size_t)(rp - wo.ptr);
    if ((a.send_off[r] + sb) / 16 > 0xFFFFFFFFull || (a.recv_off[r] + rb) / 16 > 0xFFFFFFFFull)
      return DCC_ERR_INVALID_ARG;
  }
  for (int r = 0; r < c->n; ++r)
    for (int p = 0; p < c->n; ++p) {
      if (dcc_host::overlaps(recv[r], rb, send[p], sb)) return DCC_ERR_INVALID_ARG;
      if (p != r && dcc_host::overlaps(recv[r], rb, recv[p], rb)) return DCC_ERR_INVALID_ARG;
      if (p != r && !c->chan[r][p]) return DCC_ERR_NO_CHANNEL;
    }
  a.bytes = sb;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  dcc::DevComm dc = c->dev;
  dcc::PortDev pd = c->proxy->dev;
  void* args[] = {&dc, &pd, &a};
  return port_launch(c, reinterpret_cast<const void*>(&k_port_allgather), c->n, args,
                     static_cast<cudaStream_t>(s));
}

int dcc_fifo_push(dcc_comm_t c, const uint64_t* fst, const uint64_t* snd, int count, dcc_stream_t s) {
  if (!c || !fst || count < 0 || count > kMaxCustom) return DCC_ERR_INVALID_ARG;
  if (c->sticky != DCC_OK) return c->sticky;
  int rc = require_running(c);
  if (rc != DCC_OK) return rc;
  CustomArgs a{};
  a.count = count;
  for (int i = 0; i < count; ++i) {
    if (fst[i] == 0 || (fst[i] & dcc::kTrigBuiltin)) return DCC_ERR_INVALID_ARG;
    a.t[i].fst = fst[i];
    a.t[i].snd = snd ? snd[i] : 0;
  }
  if (count == 0) return DCC_OK;
  DeviceScope ds(c->device);
  if (!ds.ok()) return DCC_ERR_CUDA;
  dcc::DevComm dc = c->dev;
  dcc::PortDev pd = c->proxy->dev;
  void* args[] = {&dc, &pd, &a};
  return dcc_host::launch(reinterpret_cast<const void*>(&k_fifo_push), 1, 32, false, args,
                          static_cast<cudaStream_t>(s));
}

}  // extern "C"
