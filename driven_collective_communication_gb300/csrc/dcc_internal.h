// dcc_internal.h -- structures passed from the host library to the kernels.
#pragma once
#include <cstddef>
#include <cstdint>

#include "dcc.h"

namespace dcc {

// One inbound semaphore per (dst rank, src rank, block slot), each in its own
// 32-byte sector so that no two counters (and no data) share a sector.
constexpr int kSemWords = 4;

__host__ __device__ inline size_t sem_slot(int dst, int src, int blk) {
  return ((size_t)dst * DCC_MAX_RANKS + (size_t)src) * DCC_MAX_BLOCKS_PER_RANK + (size_t)blk;
}
constexpr size_t kSemSlots = (size_t)DCC_MAX_RANKS * DCC_MAX_RANKS * DCC_MAX_BLOCKS_PER_RANK;

// Packed first-failure record written by a device wait that gave up.
//   bits 0..7 code (1 = timeout), 8..15 rank, 16..23 peer, 24..39 block.
constexpr unsigned long long kStatusTimeout = 1ull;
__host__ __device__ inline unsigned long long pack_status(unsigned long long code, int rank,
                                                          int peer, int blk) {
  return code | ((unsigned long long)(rank & 0xFF) << 8) |
         ((unsigned long long)(peer & 0xFF) << 16) | ((unsigned long long)(blk & 0xFFFF) << 24);
}

// Bounds-checked build (compiled with -DDCC_CHECK_BOUNDS=1, libdcc_checked.so):
// every data access of the collectives and the fused layer is checked against
// the extent of the registered window its pointer lies in; the first access
// outside is skipped and recorded as
//   bits 0..7 code 2, 8..15 the buffer's rank, 16..23 the buffer kind,
//   24..63 the offending byte offset / 16 from the buffer pointer.
#ifndef DCC_CHECK_BOUNDS
#define DCC_CHECK_BOUNDS 0
#endif
constexpr unsigned long long kStatusBounds = 2ull;
enum BufKind { kBufSend = 0, kBufRecv = 1, kBufScratch = 2, kBufX = 3, kBufResidual = 4, kNumBufKinds = 5 };
__host__ __device__ inline unsigned long long pack_bounds(int rank, int kind, size_t byte_off) {
  return kStatusBounds | ((unsigned long long)(rank & 0xFF) << 8) | ((unsigned long long)(kind & 0xFF) << 16) |
         (((unsigned long long)(byte_off / 16) & ((1ull << 40) - 1)) << 24);
}

// Device view of a communicator, passed by value to every kernel.
struct DevComm {
  int n;                        // virtual ranks
  int skip_signal_rank;         // test knob: this rank sends no signals (-1 = none)
  unsigned long long timeout_ns;
  unsigned long long* sem;      // kSemSlots counters, kSemWords apart
  unsigned long long* expect;   // kSemSlots waiter-side completed-wait counts
  unsigned long long* status;   // first failure, 0 = none
  unsigned long long* ll_epoch; // LL protocol epochs, [rank][slot] (DCC_MAX_BLOCKS_PER_RANK slots)
  char* ll_buf;                 // LL packet buffers, one per rank (library-owned, zeroed at create)
};

// A channel as the host builds it (one per ordered pair src -> dst) and copies
// to the device: the local and remote windows it binds.
struct DevChannel {
  char* local_in;
  char* local_out;
  char* remote_in;
  char* remote_out;
  size_t local_in_bytes, local_out_bytes, remote_in_bytes, remote_out_bytes;
  int connected;
  int pad;
};

// Per-call arguments of a collective kernel.
struct CollArgs {
  void* send[DCC_MAX_RANKS];
  void* recv[DCC_MAX_RANKS];
  void* scratch[DCC_MAX_RANKS];
  size_t count;   // elements: per-rank buffer (AllReduce), recv_count (RS), send_count (AG)
  int blocks;     // CTAs per rank
  int inplace;    // some rank has send == recv
  int unroll;     // in-place one-shot: vectors per thread per chunk (1..4; 0 = 4)
#if DCC_CHECK_BOUNDS
  size_t ext[kNumBufKinds][DCC_MAX_RANKS];  // bytes from each pointer to its window's end
#endif
};

// Arguments of the primitive (put/get) kernels.
struct PrimArgs {
  int src, dst;
  size_t remote_off, local_off, bytes;
  int signal;
  const DevChannel* table;  // device channel table, [src * DCC_MAX_RANKS + dst]
};

}  // namespace dcc
