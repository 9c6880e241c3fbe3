// fused.cuh -- row-parallel linear layer fused with the sum AllReduce.
//
// The project summary ("How It Works") counts overlapping communication with
// computation among the channel interfaces' uses, and its "Highlighted Details"
// single out AllReduce for tensor-parallel LLM serving.  In a tensor-parallel
// decode step a row-parallel layer leaves rank p with the partial product
// W_p x_p of its slice of the contraction dimension, and the AllReduce sums
// the partials.  Here the two are one kernel: the reduction over ranks is
// the epilogue of the matrix-vector product, and the result is put straight
// into every rank's output.
//
//   y_r[i] = R( sum_p  sum_k W_p[i][k] x_p[k] )   for every rank r
//
// optionally with a residual per output rank joining the sum before the
// rounding, y_r[i] = R( ... + res_r[i] ) (the tensor-parallel residual
// stream update h <- h + layer(h), in place when res_r is y_r).
//
// Schedule (two-shot, like k_allreduce_twoshot): rank r's CTAs own shard r of
// the rows, in items of kFusedRows rows, one item per CTA at a time.  The
// CTA's warps take the ranks in parallel: warp w gets the item's rows of W_p
// and x_p from rank p = w, w + 8, ... in 16-byte vectors, kFusedVecs per lane
// and row per round so that a row's loads of one round are all in flight
// (lanes stride the row, coalesced), accumulates fp32 dot products with fused
// multiply-adds and reduces them across lanes with a fixed shuffle tree.  One
// thread per row then adds the ranks' partials in rank order and lanes
// 0..N-1 put the packed rows into the N outputs.  Every output element is
// computed once, so every rank receives the same bits.  Measured on GB300 (8
// ranks x 8192 rows): two-row items with four vectors per lane per round
// beat eight-row items with two by 7-9 % at kp 2048-2560 and match them at
// kp 1024; more rows per item or fewer vectors per round were slower.
//
// The per-rank dot products are reordered relative to a sequential sum (lane
// strides and a shuffle tree), so results are exact when every fp32 partial
// sum is exact (small-integer data) and otherwise within the fp32
// dot-product error bound plus one rounding to the output type.
#pragma once
#include "collectives.cuh"

namespace dcc {

constexpr int kFusedThreads = 256;
constexpr int kFusedRows = 2;  // output rows per item: one 4-byte packed store per rank
constexpr int kFusedVecs = 4;  // 16-byte vectors per lane and row per round

struct LinearArgs {
  const void* weight[DCC_MAX_RANKS];    // rows x kp, row-major
  const void* x[DCC_MAX_RANKS];         // kp
  const void* residual[DCC_MAX_RANKS];  // rows per output rank, or all null (no residual)
  void* y[DCC_MAX_RANKS];               // rows
  size_t rows, kp;
  int blocks;
#if DCC_CHECK_BOUNDS
  size_t ext[kNumBufKinds][DCC_MAX_RANKS];  // weight: kBufSend, y: kBufRecv, x: kBufX, residual: kBufResidual
#endif
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

static_assert(DCC_MAX_RANKS <= 32, "lane q of warp 0 serves output rank q");

// Lane q < N of warp 0: residual q's two rows of item v (0 without
// residuals).  Loaded when the item starts, so that the load overlaps the
// weight stream instead of adding a memory round trip to the epilogue.
__device__ __forceinline__ uint32_t load_residual(const DevComm& dc, const LinearArgs& a, int n, int lane,
                                                  size_t v) {
  return a.residual[0] != nullptr && lane < n && in_bounds(dc, a, kBufResidual, lane, v * 4, 4)
             ? static_cast<const uint32_t*>(a.residual[lane])[v]
             : 0u;
}

// Puts item v's two rows (fp32 sums y0, y1) into the N outputs: one packed
// rounding shared by every rank, or with residuals R(y + residual_q) for
// output q (res: the word load_residual returned), the residual joining the
// fp32 sum before the one rounding.  The same thread reads residual q and
// writes output q, so they may be the same buffer (the in-place
// residual-stream update).
template <typename T>
__device__ __forceinline__ void put_rows(const DevComm& dc, const LinearArgs& a, int n, int lane, size_t v,
                                         float y0, float y1, uint32_t res) {
  using L = Lanes<T>;
  if (a.residual[0] == nullptr) {
    const uint32_t packed = L::narrow2(y0, y1);
    if (lane < n && in_bounds(dc, a, kBufRecv, lane, v * 4, 4)) static_cast<uint32_t*>(a.y[lane])[v] = packed;
  } else if (lane < n && in_bounds(dc, a, kBufRecv, lane, v * 4, 4)) {
    const float2 r = L::widen2(res);
    static_cast<uint32_t*>(a.y[lane])[v] = L::narrow2(__fadd_rn(y0, r.x), __fadd_rn(y1, r.y));
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <typename T, int NT>
__global__ void __launch_bounds__(kFusedThreads) k_linear_allreduce(DevComm dc, LinearArgs a) {
  pdl_prologue();
  constexpr int R = kFusedRows, V = kFusedVecs;
  static_assert(R == 2, "the epilogue packs two rows per item");
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const size_t kv = a.kp / 8;  // 16-byte vectors per weight row
  const size_t items = a.rows / R;
  __shared__ float part_s[DCC_MAX_RANKS][R];
  size_t s0, s1;
  shard_vecs(items, n, rank, s0, s1);
  for (size_t v = s0 + blk; v < s1; v += B) {
    const uint32_t res = warp == 0 ? load_residual(dc, a, n, lane, v) : 0u;
    // warp w computes the partial products of ranks w, w + nwarps, ... for
    // the item's rows; the ranks' partials meet in shared memory
    for (int p = warp; p < n; p += nwarps) {
      const uint4* w = static_cast<const uint4*>(a.weight[p]) + v * R * kv;
      const uint4* x = static_cast<const uint4*>(a.x[p]);
      float part[R];
#pragma unroll
      for (int r = 0; r < R; ++r) part[r] = 0.0f;
      for (size_t k0 = 0; k0 < kv; k0 += 32 * V) {
        uint4 wv[R][V], xv[V];
#pragma unroll
        for (int j = 0; j < V; ++j) {
          const size_t k = k0 + j * 32 + lane;
          const bool in = k < kv;
          xv[j] = in && in_bounds(dc, a, kBufX, p, k * 16, 16) ? ld_vec(x + k) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int r = 0; r < R; ++r)
            wv[r][j] = in && in_bounds(dc, a, kBufSend, p, ((v * R + r) * kv + k) * 16, 16) ? ld_vec(w + r * kv + k)
                                                                                            : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < V; ++j)
#pragma unroll
          for (int r = 0; r < R; ++r) dot8_acc<T>(part[r], wv[r][j], xv[j]);
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float sum = warp_sum(part[r]);
        if (lane == 0) part_s[p][r] = sum;
      }
    }
    __syncthreads();
    // one thread per row adds the ranks' partials in rank order; the packed
    // rows go to all N outputs
    if (warp == 0) {
      float acc = 0.0f;
      if (lane < R) {
        acc = part_s[0][lane];
        for (int p = 1; p < n; ++p) acc = __fadd_rn(acc, part_s[p][lane]);
      }
      const float y0 = __shfl_sync(0xffffffffu, acc, 0), y1 = __shfl_sync(0xffffffffu, acc, 1);
      put_rows<T>(dc, a, n, lane, v, y0, y1, res);
    }
    // kept even after the CTA's last item: skipping it there measured slower
    // on GB300 (32.4 vs 26.2 us at 8 ranks x 8192 rows x kp 1024)
    __syncthreads();
  }
}

template <typename T>
const void* linear_allreduce_kernel(int n);

}  // namespace dcc
