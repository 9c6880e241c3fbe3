// fused_bulk.cuh -- the row-parallel linear layer + AllReduce of fused.cuh
// with its weight stream staged in shared memory by the bulk copy engine
// (TMA, non-tensor cp.async.bulk), for long rows.
//
//   y_r[i] = R( sum_p  sum_k W_p[i][k] x_p[k] [+ res_r[i]] )   for every rank r
//
// A matrix-vector product streams its weights once, so it is bound by how
// many bytes each SM keeps in flight.  Loads into registers cannot keep
// enough: on GB300 the thread-load kernel of fused.cuh holds 90 registers per
// thread, two CTAs per SM, and reads 5.4-5.8 TB/s.  Here one thread per CTA
// hands whole row chunks to the copy engine and the in-flight bytes sit in
// shared memory instead: 7.1 TB/s at kp = 8192 (8 ranks x 8192 rows).
//
// Schedule.  An item is kFusedBulkRows output rows.  Rank r's CTAs own shard
// r of the items, one item per CTA at a time (the two-shot owner schedule of
// k_linear_allreduce).  For its item a CTA walks the tiles (rank p, k-chunk
// c), p = 0..N-1, c = 0..ceil(kp / kFusedBulkChunk)-1: a tile is the item's
// rows of W_p between k = c*chunk and the chunk's end (one bulk copy per row)
// plus the same piece of x_p (one more), landing on the stage's mbarrier.
// Stages form a ring of kFusedBulkStages; thread 0 refills a stage once all
// warps have read it.  Warp w takes row w % kFusedBulkRows and every
// (8 / kFusedBulkRows)-th group of 32 vectors of the chunk, accumulates with
// fused multiply-adds, and at the end of rank p reduces across lanes with a
// fixed shuffle tree.  The epilogue adds the warps' partials of a row in warp
// order, then the ranks in rank order, rounds once, and lanes 0..N-1 put the
// packed rows into the N outputs.  Every output element is computed once, so
// every rank receives the same bits; the dot products are reordered relative
// to a sequential sum, so results are exact for small-integer data and
// otherwise within the fp32 dot-product error bound.
//
// Every mbarrier wait is bounded as in bulk.cuh: on the limit it records a
// timeout in the status word, waits (bounded) for its copies in flight and
// returns.
#pragma once
#include "bulk.cuh"
#include "fused.cuh"

namespace dcc {

constexpr int kFusedBulkRows = 2;       // output rows per item
constexpr int kFusedBulkChunk = 4096;   // elements of a row per tile (8 KiB of bf16)
constexpr int kFusedBulkStages = 2;
constexpr int kFusedBulkStageBytes = (kFusedBulkRows + 1) * kFusedBulkChunk * 2;

__host__ __device__ constexpr size_t fused_bulk_smem_bytes() {
  return 128 + (size_t)kFusedBulkStages * kFusedBulkStageBytes;
}

template <typename T, int NT>
__global__ void __launch_bounds__(kFusedThreads) k_linear_allreduce_bulk(DevComm dc, LinearArgs a) {
  pdl_prologue();
  constexpr int RI = kFusedBulkRows, ST = kFusedBulkStages;
  constexpr int ROWB = kFusedBulkChunk * 2;
  constexpr int NW = kFusedThreads / 32, PARTS = NW / RI;
  static_assert(NW % RI == 0 && RI == 2, "the epilogue packs two rows per item");
  const int n = NT > 0 ? NT : dc.n;
  const int B = a.blocks;
  const int rank = blockIdx.x / B, blk = blockIdx.x % B;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = warp % RI, part = warp / RI;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  unsigned char* stage0 = smem + 128;
  __shared__ float part_s[DCC_MAX_RANKS][NW];

  const size_t kp = a.kp;
  const int nch = (int)((kp + kFusedBulkChunk - 1) / kFusedBulkChunk);
  const int ntiles = n * nch;
  const size_t items = a.rows / RI;
  size_t s0, s1;
  shard_vecs(items, n, rank, s0, s1);
  auto chunk_elems = [&](int c) {
    const size_t k0 = (size_t)c * kFusedBulkChunk;
    return kp - k0 < (size_t)kFusedBulkChunk ? kp - k0 : (size_t)kFusedBulkChunk;
  };
  // thread 0: tile t of item v into stage u (global tile count g selects the stage)
  auto issue = [&](size_t v, int t, unsigned long long g) {
    const int u = (int)(g % ST), p = t / nch, c = t % nch;
    const uint32_t bytes = (uint32_t)(chunk_elems(c) * 2);
    unsigned char* st = stage0 + (size_t)u * kFusedBulkStageBytes;
    const size_t woff = (v * RI * kp + (size_t)c * kFusedBulkChunk) * 2, xoff = (size_t)c * kFusedBulkChunk * 2;
    bool ok = in_bounds(dc, a, kBufX, p, xoff, bytes);  // bounds-checked build: a bad tile loads nothing
    for (int r = 0; r < RI; ++r) ok = in_bounds(dc, a, kBufSend, p, woff + (size_t)r * kp * 2, bytes) && ok;
    mbar_arrive_expect_tx(&full[u], ok ? bytes * (RI + 1) : 0u);
    if (!ok) return;
    const char* w = static_cast<const char*>(a.weight[p]) + woff;
    for (int r = 0; r < RI; ++r) bulk_load(st + r * ROWB, w + (size_t)r * kp * 2, bytes, &full[u]);
    bulk_load(st + RI * ROWB, static_cast<const char*>(a.x[p]) + xoff, bytes, &full[u]);
  };

  if (threadIdx.x == 0) {
    for (int u = 0; u < ST; ++u) mbar_init(&full[u], 1);
    fence_mbar_init();
  }
  __syncthreads();
  // the ring runs across the CTA's items: g counts every tile this CTA has
  // consumed, h every tile it has issued
  unsigned long long g = 0, h = 0;
  bool failed = false;
  auto issue_next = [&](size_t& iv, int& it) {  // thread 0: next tile after (iv, it), in order
    if (iv >= s1) return;
    issue(iv, it, h++);
    if (++it == ntiles) {
      it = 0;
      iv += (size_t)B;
    }
  };
  size_t iv = s0 + (size_t)blk;
  int it = 0;
  if (threadIdx.x == 0)
    for (int u = 0; u < ST; ++u) issue_next(iv, it);

  for (size_t v = s0 + (size_t)blk; v < s1 && !failed; v += (size_t)B) {
    const uint32_t res = warp == 0 ? load_residual(dc, a, n, lane, v) : 0u;
    float acc = 0.0f;
    for (int t = 0; t < ntiles; ++t, ++g) {
      const int u = (int)(g % ST), p = t / nch, c = t % nch;
      const int nv = (int)(chunk_elems(c) / 8);
      failed = !mbar_wait(&full[u], (uint32_t)((g / ST) & 1), dc, rank, blk);
      if (!failed) {
        const uint4* wr = reinterpret_cast<const uint4*>(stage0 + (size_t)u * kFusedBulkStageBytes + row * ROWB);
        const uint4* xr = reinterpret_cast<const uint4*>(stage0 + (size_t)u * kFusedBulkStageBytes + RI * ROWB);
#pragma unroll 4
        for (int j = part * 32 + lane; j < nv; j += 32 * PARTS) dot8_acc<T>(acc, wr[j], xr[j]);
        if (c == nch - 1) {
          const float r = warp_sum(acc);
          if (lane == 0) part_s[p][warp] = r;
          acc = 0.0f;
        }
      }
      if (__syncthreads_or(failed)) {
        failed = true;
        break;
      }
      if (threadIdx.x == 0) issue_next(iv, it);
    }
    if (failed) break;
    // epilogue: lane r < RI sums row r over the warps, then over the ranks
    if (warp == 0) {
      float y = 0.0f;
      if (lane < RI) {
        for (int q = 0; q < n; ++q) {
          float rq = part_s[q][lane];
          for (int k = 1; k < PARTS; ++k) rq = __fadd_rn(rq, part_s[q][k * RI + lane]);
          y = q == 0 ? rq : __fadd_rn(y, rq);
        }
      }
      const float y0 = __shfl_sync(0xffffffffu, y, 0), y1 = __shfl_sync(0xffffffffu, y, 1);
      put_rows<T>(dc, a, n, lane, v, y0, y1, res);
    }
    __syncthreads();  // part_s is rewritten by the next item
  }
  if (failed && threadIdx.x == 0)  // let the copies in flight land before shared memory goes away
    for (; g < h; ++g) mbar_wait(&full[g % ST], (uint32_t)((g / ST) & 1), dc, rank, blk);
}

template <typename T>
const void* linear_allreduce_bulk_kernel(int n);

}  // namespace dcc
