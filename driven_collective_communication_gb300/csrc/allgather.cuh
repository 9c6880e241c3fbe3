// allgather.cuh -- AllGather: every rank's input put into its slot of every
// rank's output (the gathering half of a two-shot AllReduce; the collective
// interface of the MSCCL++ abstract, point 3).
//
//   recv[p][q*m + j] = send[q][j]      for all ranks p, q and j < m
//
// A bit copy: the element type only sets the size.  Rank q's CTAs read their
// input once and put it into the N outputs, so one launch reads S bytes per
// rank and writes N*S.
//
// On GB300 this write-heavy mix is bound by how long a load waits behind the
// write stream, not by the writes themselves (a store-only kernel of the same
// shape writes 7.1 TB/s; one load then N stores per thread moves 4.0 TB/s).
// So each thread first issues kAgUnroll independent 16-byte loads, then puts
// them destination by destination with evict-first (streaming) stores: each
// output region is then written in one contiguous burst per warp and the
// output does not push the inputs out of L2.  Measured on GB300 at 8 x 8 MiB
// fp16 in: 93.7 us (6.45 TB/s of S + N*S bytes) vs 151 us for one load per
// thread and 107 us for the bulk-copy (TMA) pipeline.
#pragma once
#include "collectives.cuh"

namespace dcc {

constexpr int kAgUnroll = 8;  // 16-byte vectors each thread has in flight

__device__ __forceinline__ void st_vec_stream(uint4* p, uint4 v) { __stcs(p, v); }

template <int NT, bool EB = false>
__global__ void __launch_bounds__(kThreads) k_allgather(DevComm dc, CollArgs a, int elem_bytes) {
  pdl_prologue();
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  const size_t bytes = a.count * (size_t)elem_bytes;
  if constexpr (EB) {
    if (!entry_barrier(dc, rank, n, blk)) return;
  }
  if (bytes % 16 == 0) {
    // thread t of CTA c covers vectors c*U*T + j*T + t, j < U: every load and
    // store instruction of a warp touches 512 contiguous bytes
    const size_t nv = bytes / 16;
    const size_t T = blockDim.x;
    const uint4* src = static_cast<const uint4*>(a.send[rank]);
    const size_t dst_off = (size_t)rank * nv;
    for (size_t v0 = (size_t)blk * kAgUnroll * T + threadIdx.x; v0 < nv; v0 += (size_t)B * kAgUnroll * T) {
      uint4 x[kAgUnroll];
#pragma unroll
      for (int j = 0; j < kAgUnroll; ++j)
        if (v0 + j * T < nv)
          x[j] = in_bounds(dc, a, kBufSend, rank, (v0 + j * T) * 16, 16) ? ld_vec(src + v0 + j * T)
                                                                         : make_uint4(0, 0, 0, 0);
      auto put = [&](int p) {
        uint4* d = static_cast<uint4*>(a.recv[p]) + dst_off;
#pragma unroll
        for (int j = 0; j < kAgUnroll; ++j)
          if (v0 + j * T < nv && in_bounds(dc, a, kBufRecv, p, (dst_off + v0 + j * T) * 16, 16))
            st_vec_stream(d + v0 + j * T, x[j]);
      };
      if constexpr (NT > 0) {
#pragma unroll
        for (int p = 0; p < NT; ++p) put(p);
      } else {
        for (int p = 0; p < n; ++p) put(p);
      }
    }
    return;
  }
  // inputs whose size is not a whole number of 16-byte vectors: element copies
  const size_t stride = (size_t)B * blockDim.x;
  const size_t first = (size_t)blk * blockDim.x + threadIdx.x;
  auto copy = [&](auto zero) {
    using E = decltype(zero);
    for (size_t j = first; j < a.count; j += stride) {
      const E x = get_elem<E>(dc, a, rank, j);
      for (int p = 0; p < n; ++p) put_elem<E>(dc, a, p, (size_t)rank * a.count + j, x);
    }
  };
  if (elem_bytes == 4) copy(uint32_t{0});
  else copy(uint16_t{0});
}

// Kernel tables (compile-time N for 1, 2, 4, 8, 16; a runtime-N instance
// otherwise); eb selects the instance with the entry barrier.
const void* allgather_kernel(int n, bool eb = false);
const void* allgather_bulk_kernel(int n);

}  // namespace dcc
