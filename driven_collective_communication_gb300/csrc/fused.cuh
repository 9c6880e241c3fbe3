// fused.cuh -- row-parallel linear layer fused with the sum AllReduce.
//
// The project summary ("How It Works") counts communication-to-computation
// overlap among the channel interfaces' uses, and its "Highlighted Details"
// single out AllReduce for tensor-parallel LLM serving.  In a tensor-parallel
// decode step a row-parallel layer leaves rank p with the partial product
// W_p x_p of its slice of the contraction dimension, and the AllReduce sums
// the partials.  Here the two are one kernel: the reduction over ranks is
// the epilogue of the matrix-vector product, and the result is put straight
// into every rank's output.
//
//   y_r[i] = R( sum_p  sum_k W_p[i][k] x_p[k] )   for every rank r
//
// Schedule (two-shot, like k_allreduce_twoshot): rank r's CTAs own shard r of
// the rows, in items of 8 rows (one 16-byte output vector), one item per CTA
// at a time.  The CTA's warps take the ranks in parallel: warp w gets the 8
// weight rows of W_p and x_p from rank p = w, w + 8, ... in 16-byte vectors
// (lanes stride the row, coalesced), accumulates 8 fp32 dot products with
// fused multiply-adds and reduces them across lanes with a fixed shuffle
// tree.  One thread per row then adds the ranks' partials in rank order and
// lanes 0..N-1 put the packed vector into the N outputs.  Every output
// element is computed once, so every rank receives the same bits.
//
// The per-rank dot products are reordered relative to a sequential sum (lane
// strides and a shuffle tree), so results are exact when every fp32 partial
// sum is exact (small-integer data) and otherwise within the fp32
// dot-product error bound plus one rounding to the output type.
#pragma once
#include "collectives.cuh"

namespace dcc {

constexpr int kFusedThreads = 256;
constexpr int kFusedRows = 8;  // output rows per warp item: one 16-byte vector

struct LinearArgs {
  const void* weight[DCC_MAX_RANKS];  // rows x kp, row-major
  const void* x[DCC_MAX_RANKS];       // kp
  void* y[DCC_MAX_RANKS];             // rows
  size_t rows, kp;
  int blocks;
};

template <typename T>
__device__ __forceinline__ void dot8_acc(float& acc, uint4 w, uint4 x) {
  using L = Lanes<T>;
  const uint32_t ww[4] = {w.x, w.y, w.z, w.w}, xx[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 a = L::widen2(ww[j]), b = L::widen2(xx[j]);
    acc = __fmaf_rn(a.x, b.x, acc);
    acc = __fmaf_rn(a.y, b.y, acc);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <typename T, int NT>
__global__ void __launch_bounds__(kFusedThreads) k_linear_allreduce(DevComm dc, LinearArgs a) {
  using L = Lanes<T>;
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const size_t kv = a.kp / 8;             // 16-byte vectors per weight row
  const size_t items = a.rows / kFusedRows;
  __shared__ float part_s[DCC_MAX_RANKS][kFusedRows];
  size_t s0, s1;
  shard_vecs(items, n, rank, s0, s1);
  for (size_t v = s0 + blk; v < s1; v += B) {
    // warp w computes the partial products of ranks w, w + nwarps, ... for
    // the item's 8 rows; the ranks' partials meet in shared memory
    for (int p = warp; p < n; p += nwarps) {
      const uint4* w = static_cast<const uint4*>(a.weight[p]) + v * kFusedRows * kv;
      const uint4* x = static_cast<const uint4*>(a.x[p]);
      float part[kFusedRows];
#pragma unroll
      for (int r = 0; r < kFusedRows; ++r) part[r] = 0.0f;
      size_t k = lane;
      for (; k + 32 < kv; k += 64) {  // two vectors per lane in flight per row
        const uint4 x0 = ld_vec(x + k), x1 = ld_vec(x + k + 32);
        uint4 w0[kFusedRows], w1[kFusedRows];
#pragma unroll
        for (int r = 0; r < kFusedRows; ++r) {
          w0[r] = ld_vec(w + r * kv + k);
          w1[r] = ld_vec(w + r * kv + k + 32);
        }
#pragma unroll
        for (int r = 0; r < kFusedRows; ++r) {
          dot8_acc<T>(part[r], w0[r], x0);
          dot8_acc<T>(part[r], w1[r], x1);
        }
      }
      if (k < kv) {
        const uint4 x0 = ld_vec(x + k);
#pragma unroll
        for (int r = 0; r < kFusedRows; ++r) dot8_acc<T>(part[r], ld_vec(w + r * kv + k), x0);
      }
#pragma unroll
      for (int r = 0; r < kFusedRows; ++r) {
        const float sum = warp_sum(part[r]);
        if (lane == 0) part_s[p][r] = sum;
      }
    }
    __syncthreads();
    // one thread per row adds the ranks' partials in rank order; the packed
    // result goes to all N outputs
    if (warp == 0) {
      float acc = 0.0f;
      if (lane < kFusedRows) {
        acc = part_s[0][lane];
        for (int p = 1; p < n; ++p) acc = __fadd_rn(acc, part_s[p][lane]);
      }
      typename L::Acc out;
#pragma unroll
      for (int r = 0; r < kFusedRows; ++r) out.v[r] = __shfl_sync(0xffffffffu, acc, r);
      const uint4 packed = L::pack(out);
      for (int q = lane; q < n; q += 32) st_vec(static_cast<uint4*>(a.y[q]) + v, packed);
    }
    __syncthreads();
  }
}

template <typename T>
const void* linear_allreduce_kernel(int n);

}  // namespace dcc
