// fused_mma.cuh -- the row-parallel linear layer over a batch of tokens fused
// with the sum AllReduce, on the fifth-generation tensor cores.
//
// The project summary ("How It Works") counts overlapping communication with
// computation among the channel interfaces' uses and its "Highlighted
// Details" single out AllReduce for tensor-parallel serving.  With several
// tokens per step (batched decode, speculative decoding, prefill chunks) the
// row-parallel layer is a contraction:
//
//   Y[t][i] = R( sum_p sum_k W_p[i][k] * X_p[t][k] ),  every rank receives Y
//
// W_p rows x kp (row-major), X_p tokens x kp (row-major), Y tokens x rows
// (token t's hidden vector contiguous).  Seen as one GEMM, D = A B^T with
// A = [W_0 | ... | W_{N-1}] (rows x N*kp) and B = [X_0 | ... | X_{N-1}]
// (tokens x N*kp): the ranks' shards are slices of the contraction
// dimension, and the AllReduce is the sum over them.
//
// Kernel.  A CTA owns a tile of up to 128 rows of Y (one accumulator: the
// MMA's M = 128, N = tokens rounded up to a multiple of 16, at most 256) or
// up to 256 rows (MACC = 2 accumulators sharing each token tile) for every
// token,
// and a slice of the contraction dimension; the KS CTAs of a thread-block
// cluster split the contraction (rank slices in rank order).  Per CTA (128
// threads in the pair form, two CTAs to an SM; 256 otherwise):
//   warp 0, one thread   TMA producer: per 64-element K block, the 128 x 64
//                         tile(s) of W_p and the tokens x 64 tile of X_p (all
//                         128-byte swizzled, K-major) onto a stage mbarrier;
//   warp 1, one thread   MMA issuer: four tcgen05.mma (K = 16 each) per
//                         stage and accumulator into fp32 accumulators in
//                         tensor memory, then tcgen05.commit frees the stage;
//   warp 2               allocates / frees the tensor-memory columns;
//   warps 2 and up       (with residuals) ask L2 for the epilogue's residual
//                         rows while the main loop runs;
//   all warps            epilogue (mma_epilogue): tcgen05.ld of the
//                         accumulators into shared memory, the split partials
//                         exchanged through each CTA's inbox, each CTA of the
//                         cluster adds the KS partials of its share of the
//                         tokens in split order, rounds once and stores 16
//                         bytes (8 rows) at a time into all N outputs.
// With a residual per output rank (the residual stream of the layer,
// h_q <- h_q + layer) output q gets R(sum + residual_q): the residual joins
// the fp32 sum before the one rounding, and the thread that reads residual q
// writes output q, so the two may be one buffer.
// Tokens beyond the batch and rows beyond the matrix are zero-filled by the
// tensor map and masked at the store.  The fp32 accumulation order inside
// the tensor core is the hardware's, so results are exact when every partial
// sum is exact (small-integer data) and otherwise within the error bound of
// an fp32 sum of N*kp exact products plus the one rounding.
//
// Every wait is bounded: a wait that runs out records a timeout in the
// status word; the thread stops issuing work but every thread still reaches
// both cluster barriers and the tensor memory is always freed.
#pragma once
#include <cuda.h>

#include "collectives.cuh"

namespace dcc {

// Threads per CTA, the kernel's THREADS: 256 (8 warps; the epilogue's loads
// and stores are latency-bound, so all eight take part, warps w and w + 4
// reading the same tensor-memory lanes in alternate 32-column chunks) with
// one CTA per SM, or 128 (the "pair" form: two CTAs per SM, each with half
// the shared memory, so the K split can be twice as deep at the same bytes
// in flight per SM).
constexpr int kMmaThreads = 256;
constexpr int kMmaPairThreads = 128;
// Shared memory for the stages: one CTA per SM, or two
constexpr unsigned kMmaStageBudget = 216u * 1024u;
constexpr unsigned kMmaPairStageBudget = 108u * 1024u;
constexpr int kMmaBM = 128;      // accumulator rows per CTA (TMEM lanes)
constexpr int kMmaBK = 64;       // K elements per stage (one 128-byte swizzle atom row)
constexpr int kMmaMaxTokens = 256;
constexpr int kMmaMaxSplit = 8;  // CTAs per cluster along K
#ifndef DCC_MMA_PLAIN_BATCH
#define DCC_MMA_PLAIN_BATCH 2  // epilogue items per thread per pass without residuals
#endif

struct MmaMaps {
  CUtensorMap w[DCC_MAX_RANKS];   // rows x kp, box 64 x bm (one accumulator) or 64 x 128
  CUtensorMap x[DCC_MAX_RANKS];   // tokens x kp, box 64 x ntile
  CUtensorMap w2[DCC_MAX_RANKS];  // several accumulators: the last one's box, 64 x (bm - 128 (macc - 1))
};

struct MmaArgs {
  void* y[DCC_MAX_RANKS];          // tokens x rows
  const void* res[DCC_MAX_RANKS];  // tokens x rows residuals (res[0] null: none)
  int tokens, rows, kp, ntile, ks, stages;
  int bm;                  // weight rows per CTA (multiple of 8, at most macc * kMmaBM)
  int macc;                // accumulators per CTA (the kernel's MACC): 1 or 2, 128 rows each but the last
  int rounds;              // epilogue rounds (token ranges exchanged one after another): 1, 2 or 4
  int fp16;                // element type: 0 bf16, 1 fp16
#if DCC_CHECK_BOUNDS
  size_t ext[kNumBufKinds][DCC_MAX_RANKS];
#endif
};

// a stage: macc weight tiles of 128 x 64 and the token tile ntile x 64
__host__ __device__ constexpr size_t mma_stage_bytes(int ntile, int macc) {
  return (size_t)macc * kMmaBM * kMmaBK * 2 + (size_t)ntile * kMmaBK * 2;
}
constexpr int kMmaMaxStages = 16;
// dynamic shared memory: 1 KiB for alignment, the stages, and the mbarriers
__host__ __device__ constexpr size_t mma_smem_bytes(int ntile, int stages, int macc) {
  return 1024 + (size_t)stages * mma_stage_bytes(ntile, macc) + 16 * (size_t)stages + 64;
}
// Stages: as many as fit in the budget (at most kMmaMaxStages) -- the weight
// stream is bound by the bytes in flight (on GB300 a loaded HBM read takes
// about 4 us, so saturating it takes some 28 MB in flight across the GPU) --
// and at least as many bytes as the fp32 partial tile the epilogue puts in
// their place.  The epilogue's inbox (the other splits' slices, see
// mma_epilogue) also needs room: mma_epilogue_fits says whether a K split
// leaves it, and the kernel checks it again before it writes.
inline int mma_stages(int ntile, int macc, unsigned budget = kMmaStageBudget) {
  const size_t st = mma_stage_bytes(ntile, macc);
  int s = (int)(budget / st);
  if (s > kMmaMaxStages) s = kMmaMaxStages;
  while ((size_t)s * st < (size_t)ntile * kMmaBM * 4) ++s;
  return s;
}

// The epilogue takes the tokens in `rounds` ranges of w = ntile / rounds
// (a multiple of 16 and of ks); a round's partial tile (w x 128 fp32) plus
// the inbox for the other ks - 1 splits' token slices must fit the stage
// buffers.
constexpr int kMmaMaxRounds = 4;
__host__ __device__ inline bool mma_round_fits(int ntile, int stages, int macc, int ks, int rounds) {
  if (rounds < 1 || rounds > kMmaMaxRounds || ntile % (16 * rounds) != 0) return false;
  const int w = ntile / rounds;
  if (w % ks != 0) return false;
  const size_t need = ((size_t)2 * w - (size_t)w / ks) * kMmaBM * 4;
  return need <= (size_t)stages * mma_stage_bytes(ntile, macc);
}
// the fewest rounds that fit, 0 if none does
__host__ __device__ inline int mma_epilogue_rounds(int ntile, int stages, int macc, int ks) {
  for (int r = 1; r <= kMmaMaxRounds; r *= 2)
    if (mma_round_fits(ntile, stages, macc, ks, r)) return r;
  return 0;
}
__host__ __device__ inline bool mma_epilogue_fits(int ntile, int stages, int macc, int ks) {
  return mma_epilogue_rounds(ntile, stages, macc, ks) > 0;
}

__device__ __forceinline__ uint32_t smem_addr_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mma_mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mma_mbar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mma_mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// bounded wait on a phase; gives up at once when another wait already failed
__device__ __forceinline__ bool mma_mbar_wait(uint32_t bar, uint32_t parity, const DevComm& dc, int rank,
                                              int blk) {
  if (mma_mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (unsigned it = 1;; ++it) {
    if (mma_mbar_try(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (ld_relaxed_gpu(dc.status) != 0ull) return false;
      if (global_timer_ns() - t0 > dc.timeout_ns) {
        atomicCAS(dc.status, 0ull, pack_status(kStatusTimeout, rank, rank, blk));
        return false;
      }
    }
  }
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// L2 eviction policies: the weights stream through once (evict first); the
// token tiles, read by every CTA, and the residuals, prefetched for the
// epilogue, stay (evict last)
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}
// asks L2 for `bytes` (a multiple of 16) at a 16-byte aligned global address
__device__ __forceinline__ void l2_prefetch_bytes(const void* p, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(p), "r"(bytes), "l"(policy)
               : "memory");
}
// asks L2 for a tile of a tensor map (no data comes back to the CTA)
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global [%0, {%1, %2}];" ::"l"(map), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void mma_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the two halves, for work in between (every thread of every CTA of the
// cluster executes each once per use, in the same order)
__device__ __forceinline__ void mma_cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void mma_cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte
// swizzled layout the tensor map writes: rows of 128 bytes, 8-row groups
// 1024 bytes apart (stride offset), descriptor version 1, swizzle mode 2.
__device__ __forceinline__ uint64_t mma_smem_desc(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: fp32 accumulator, A and B of the same
// 16-bit type (bf16 or fp16), both K-major, M = 128, N = ntile.
__device__ __forceinline__ uint32_t mma_instr_desc(int ntile, bool fp16) {
  const uint32_t ab = fp16 ? 0u : 1u;
  return (1u << 4) | (ab << 7) | (ab << 10) | ((uint32_t)(ntile >> 3) << 17) | ((uint32_t)(kMmaBM >> 4) << 24);
}

// 8 fp32 values rounded once to 8 packed 16-bit values (fp16 or bf16), and back
__device__ __forceinline__ uint4 mma_narrow8(const float* v, bool fp16) {
  if (fp16)
    return make_uint4(HalfLanes<__half2, F16Ops>::narrow2(v[0], v[1]), HalfLanes<__half2, F16Ops>::narrow2(v[2], v[3]),
                      HalfLanes<__half2, F16Ops>::narrow2(v[4], v[5]), HalfLanes<__half2, F16Ops>::narrow2(v[6], v[7]));
  return make_uint4(HalfLanes<__nv_bfloat162, Bf16Ops>::narrow2(v[0], v[1]),
                    HalfLanes<__nv_bfloat162, Bf16Ops>::narrow2(v[2], v[3]),
                    HalfLanes<__nv_bfloat162, Bf16Ops>::narrow2(v[4], v[5]),
                    HalfLanes<__nv_bfloat162, Bf16Ops>::narrow2(v[6], v[7]));
}
__device__ __forceinline__ void mma_widen8(uint4 w, bool fp16, float* v) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 f = fp16 ? F16Ops::widen2(u[k]) : Bf16Ops::widen2(u[k]);
    v[2 * k] = f.x;
    v[2 * k + 1] = f.y;
  }
}

// Epilogue of the tensor-core layer, for each accumulator h of the CTA:
//  1. each thread (row = TMEM lane) reads its row of the accumulator
//     (tcgen05.ld, 32 tokens at a time) into part[token][row] (fp32, local);
//  2. tokens are dealt out to the CTAs of the cluster in KSC equal slices of
//     T = NTILE / KSC; after a cluster barrier one thread sends slice o of
//     part (T x 128 fp32, contiguous) to CTA o with one bulk copy into its
//     inbox, completing on that CTA's inbox mbarrier.  The barrier is split:
//     a CTA arrives as soon as its main loop is over and its inbox armed,
//     writes part, then waits for the others (step 1 overlaps the wait for
//     the slowest CTA of the cluster: measured on GB300 at 8 x 8192 x 1024,
//     0.05-0.35 us less per layer from 1 to 256 tokens);
//  3. once its inbox is full each CTA adds, for 8 consecutive rows of one of
//     its tokens at a time, the KSC partials in split order (its own from
//     part, the others from the inbox: local shared memory only), rounds once
//     and stores 16 bytes into each of the N outputs (with residuals:
//     R(sum + residual_q) into output q; the thread that reads residual q
//     writes output q).
// part and the inbox reuse the stage buffers (part: NTILE x 128 floats, the
// inbox after it: (KSC - 1) x T x 128), so the copies start only once every
// CTA of the cluster is past its main loop (the barrier of step 2).
template <int KSC, int MACC, int THREADS, bool RES>
__device__ __forceinline__ void mma_epilogue(const DevComm& dc, const MmaArgs& a, uint32_t tmem, uint32_t acc_cols,
                                             float* part, uint32_t inbar, int n, unsigned split, int m0,
                                             int bm_last, bool acc_ok, int mtile) {
  // items per thread per pass: with residuals 4, whose loads then overlap;
  // without, 2 (measured on GB300 at 8 x 8192 x 1024: 0.2-0.5 us faster than
  // 4 from 1 to 256 tokens)
  constexpr int kBatch = RES ? 4 : DCC_MMA_PLAIN_BATCH;
  // a warp reaches the tensor-memory lanes 32 (warp mod 4) .. + 31 only
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, quad = warp & 3, row = quad * 32 + lane;
  // tokens in R ranges of W, each dealt out in KSC slices of T
  const int NTILE = a.ntile, R = a.rounds, W = NTILE / R, T = W / KSC;
  float* inbox = part + (size_t)W * kMmaBM;
  const uint32_t slice_bytes = (uint32_t)T * kMmaBM * 4u;
  bool ok = acc_ok;
  int phase = 0;
  for (int h = 0; h < MACC; ++h)
  for (int r = 0; r < R; ++r, ++phase) {
    const int w_lo = r * W, w_hi = w_lo + W;  // this round's tokens
    const int t_lo = w_lo + (int)split * T;   // this CTA's share of them
    // the previous round's copies refill the inboxes and part: every CTA is
    // done reading its own
    if (phase > 0) {
      if (KSC > 1) mma_cluster_sync();
      else __syncthreads();
    }
    // this CTA's stage buffers are free and its inbox armed: the others may
    // send (the inbox lies past part, which is written below meanwhile)
    if (KSC > 1) {
      if (threadIdx.x == 0) mma_mbar_expect(inbar, (uint32_t)(KSC - 1) * slice_bytes);
      mma_cluster_arrive();
    }
    // with 8 warps, warps w and w + 4 take alternate 32-column chunks; W is a
    // multiple of 16, so the last chunk may have 16 columns
    for (int c0 = w_lo + (warp >> 2) * 32; c0 < w_hi; c0 += 32 * (THREADS / 128)) {
      uint32_t v[32];
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)h * acc_cols + (uint32_t)c0;
      if (c0 + 32 <= w_hi) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]),
              "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
              "=r"(v[30]), "=r"(v[31])
            : "r"(taddr));
      } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(taddr));
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      const int cols = c0 + 32 <= w_hi ? 32 : 16;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < cols) part[(c0 - w_lo + j) * kMmaBM + row] = acc_ok ? __uint_as_float(v[j]) : 0.0f;
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    if (KSC > 1) {
      // the bulk copies read part through the async proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();     // part written
      mma_cluster_wait();  // every CTA of the cluster past its main loop, inboxes armed
      if (threadIdx.x == 0) {
        for (int o = 0; o < KSC; ++o) {
          if (o == (int)split) continue;
          const int slot = (int)split < o ? (int)split : (int)split - 1;  // my place in o's inbox
          uint32_t dst, bar;
          const uint32_t ldst = smem_addr_u32(inbox + (size_t)slot * T * kMmaBM);
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(ldst), "r"((uint32_t)o));
          asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(bar) : "r"(inbar), "r"((uint32_t)o));
          asm volatile(
              "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                  dst),
              "r"(smem_addr_u32(part + (size_t)o * T * kMmaBM)), "r"(slice_bytes), "r"(bar)
              : "memory");
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
      }
      ok = mma_mbar_wait(inbar, (uint32_t)(phase & 1), dc, mtile, (int)split) && ok;  // my inbox is full
    } else {
      __syncthreads();
    }

    const int mh = m0 + h * kMmaBM, bmh = h == MACC - 1 ? bm_last : kMmaBM;  // rows of accumulator h
    const int items = T * (kMmaBM / 8);
    // With residuals and items for less than kBatch passes of the threads, G
    // threads share an item, thread g of the group taking ranks g, g + G, ...:
    // their residual loads are in flight together instead of one rank after
    // another (each of the G adds the item's partials itself).  Otherwise
    // G = 1.
    int G = 1;
    if (RES) {
      G = THREADS * kBatch / items;
      if (G > n) G = n;
      if (G < 1) G = 1;
    }
    const int g = (int)threadIdx.x % G, lanes = THREADS / G;  // threads per item slot
    for (int w0 = (int)threadIdx.x / G; w0 < items && (int)threadIdx.x < lanes * G; w0 += lanes * kBatch) {
      float acc[kBatch][8];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int w = w0 + b * lanes;
        const int tl = w < items ? w / (kMmaBM / 8) : 0, r8 = (w % (kMmaBM / 8)) * 8;
#pragma unroll
        for (int s2 = 0; s2 < KSC; ++s2) {  // split order
          const float* src = s2 == (int)split ? &part[((int)split * T + tl) * kMmaBM + r8]
                                              : &inbox[((s2 < (int)split ? s2 : s2 - 1) * T + tl) * kMmaBM + r8];
          const float4 lo = *reinterpret_cast<const float4*>(src), hi = *reinterpret_cast<const float4*>(src + 4);
          const float v8[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[b][j] = s2 == 0 ? v8[j] : __fadd_rn(acc[b][j], v8[j]);
        }
      }
      // item b's place in the outputs (bytes), or -1 when it lies beyond the
      // batch or the matrix (rows come in multiples of 8, and bm too: all 8
      // rows or none)
      long long off[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int w = w0 + b * lanes;
        const int t = t_lo + w / (kMmaBM / 8), r8 = (w % (kMmaBM / 8)) * 8;
        off[b] = (w < items && t < a.tokens && r8 < bmh && mh + r8 < a.rows)
                     ? (long long)(((size_t)t * a.rows + (size_t)(mh + r8)) * 2)
                     : -1;
      }
      if constexpr (!RES) {  // one rounding shared by every output
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
          if (off[b] < 0) continue;
          const uint4 out = mma_narrow8(acc[b], a.fp16 != 0);
          for (int q = 0; q < n; ++q)
            if (in_bounds(dc, a, kBufRecv, q, (size_t)off[b], 16))
              st_vec(reinterpret_cast<uint4*>(static_cast<char*>(a.y[q]) + off[b]), out);
        }
      } else {
        // rank q+G's residuals are loaded before rank q's outputs are stored,
        // so two of this thread's ranks' loads are in flight at a time
        auto load_res = [&](int q, uint4* rv) {
#pragma unroll
          for (int b = 0; b < kBatch; ++b)
            rv[b] = off[b] >= 0 && in_bounds(dc, a, kBufResidual, q, (size_t)off[b], 16)
                        ? *reinterpret_cast<const uint4*>(static_cast<const char*>(a.res[q]) + off[b])
                        : make_uint4(0u, 0u, 0u, 0u);
        };
        uint4 cur[kBatch], nxt[kBatch];
        load_res(g, cur);
        for (int q = g; q < n; q += G) {
          if (q + G < n) load_res(q + G, nxt);
#pragma unroll
          for (int b = 0; b < kBatch; ++b) {
            if (off[b] < 0 || !in_bounds(dc, a, kBufRecv, q, (size_t)off[b], 16)) continue;
            float r[8], v[8];
            mma_widen8(cur[b], a.fp16 != 0, r);
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __fadd_rn(acc[b][j], r[j]);
            st_vec(reinterpret_cast<uint4*>(static_cast<char*>(a.y[q]) + off[b]), mma_narrow8(v, a.fp16 != 0));
          }
#pragma unroll
          for (int b = 0; b < kBatch; ++b) cur[b] = nxt[b];
        }
      }
    }
    // my copies have read part before it is overwritten or the CTA exits
    if (KSC > 1 && threadIdx.x == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
  (void)ok;
}

// MACC (accumulators per CTA) is a template parameter: with a run-time
// count the loops over the accumulators cost about 12 us per launch at 8 x
// 8192 x 1024 (measured on GB300: 40 vs 28 us).
//
// RES: the residual form (a.res set) is its own kernel, so the plain one
// carries none of its code (the epilogue's code is fetched cold once per
// launch: "no instruction" stalls at 2-5 per issue).  Measured on GB300 at
// 8 x 8192 x 1024 against one kernel for both: the plain layer 0.6-0.85 us
// faster from 1 to 256 tokens (21.2 against 21.8 us at 1 token), the
// residual one 0.1-0.55 us.
template <int NT, int MACC, int THREADS, bool RES>
__global__ void __launch_bounds__(THREADS, THREADS == kMmaPairThreads ? 2 : 1)
    k_linear_allreduce_mma(const __grid_constant__ MmaMaps maps, DevComm dc, MmaArgs a) {
  extern __shared__ unsigned char mma_raw[];
  __shared__ uint32_t tmem_slot;
  const int n = NT > 0 ? NT : dc.n;
  const uint32_t raw_u32 = smem_addr_u32(mma_raw);
  const uint32_t base = (raw_u32 + 1023u) & ~1023u;  // 128-byte swizzle wants 1024-byte alignment
  unsigned char* gbase = mma_raw + (base - raw_u32);
  const int S = a.stages, NTILE = a.ntile, KS = a.ks;
  const uint32_t a_bytes = kMmaBM * kMmaBK * 2, st_bytes = (uint32_t)mma_stage_bytes(NTILE, MACC);
  const uint32_t b_off = (uint32_t)MACC * a_bytes;      // the token tile follows the weight tiles
  const uint32_t bars = base + (uint32_t)S * st_bytes;  // full[S], empty[S], accumulator ready
  auto full = [&](int s) { return bars + 8u * (uint32_t)s; };
  auto empty = [&](int s) { return bars + 8u * (uint32_t)(S + s); };
  const uint32_t accf = bars + 16u * (uint32_t)S, inbar = accf + 8u;  // accumulator ready, epilogue inbox full
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned split = 0;
  if (KS > 1) asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(split));
  const int mtile = (int)blockIdx.x / KS, m0 = mtile * a.bm;
  // rows of the last accumulator (the others have 128 each)
  const int bm_last = a.bm - kMmaBM * (MACC - 1);
  // 64-column blocks per rank, the last one partial when kp is not a multiple
  // of 64: the TMA fills the columns past kp with zeros in the weight and the
  // token tiles alike, so they add nothing (and the transaction counts the
  // whole box)
  const int kpb = (a.kp + kMmaBK - 1) / kMmaBK, nb = n * kpb;
  const int b0 = (int)((long long)split * nb / KS), b1 = (int)((long long)(split + 1) * nb / KS);
  const int nk = b1 - b0;
  // columns of one accumulator (a power of two, at least 32); the second follows the first
  const uint32_t acc_cols = NTILE <= 32 ? 32u : NTILE <= 64 ? 64u : NTILE <= 128 ? 128u : 256u;
  const uint32_t ncols = acc_cols * (uint32_t)MACC;

  // The start is on the critical path of every launch (measured on GB300 at
  // 1 token: 1.1 us from entry to the first load with one thread doing all
  // of it): warp 0's lanes set up the mbarriers (full[S], empty[S], the
  // accumulator and inbox barriers, all one arrival, laid out back to back),
  // warp 2 allocates the tensor memory and warp 3 asks L2 for the first
  // weight tiles, side by side.
  if (warp == 0) {
    for (int j = lane; j < 2 * S + 2; j += 32) mma_mbar_init(bars + 8u * (uint32_t)j, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr_u32(&tmem_slot)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Launched with programmatic dependent launch, everything above overlaps
  // the end of the previous kernel on the stream, and so do L2 prefetches of
  // the first weight tiles (a prefetch returns nothing, so whatever that
  // kernel still writes lands in L2 before the loads below read it).  No data
  // is read before griddepcontrol.wait.
  if (warp == 3 && lane == 0)
    for (int i = 0; i < nk && i < S; ++i) {
      const int g = b0 + i;
      tma_prefetch_2d(&maps.w[g / kpb], (g % kpb) * kMmaBK, m0);
      for (int h = 1; h < MACC; ++h)
        tma_prefetch_2d(h == MACC - 1 ? &maps.w2[g / kpb] : &maps.w[g / kpb], (g % kpb) * kMmaBK, m0 + h * kMmaBM);
    }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_slot;

  if (warp == 0 && lane == 0) {  // TMA producer
    // the weight boxes are 128 rows for all accumulators but the last, which
    // has bm_last (tile rows beyond them are never written and only reach
    // accumulator rows the epilogue discards)
    const uint32_t tx = st_bytes - (uint32_t)(MACC * kMmaBM - a.bm) * (kMmaBK * 2);
    const uint64_t pol_w = l2_evict_first(), pol_x = l2_evict_last();
    for (int i = 0; i < nk; ++i) {
      const int s = i % S;
      if (i >= S && !mma_mbar_wait(empty(s), (uint32_t)(((i / S) - 1) & 1), dc, mtile, (int)split)) break;
      const int g = b0 + i, p = g / kpb, k0 = (g % kpb) * kMmaBK;
      const uint32_t sa = base + (uint32_t)s * st_bytes;
      mma_mbar_expect(full(s), tx);
      tma_load_2d_hint(sa, &maps.w[p], k0, m0, full(s), pol_w);
#pragma unroll
      for (int h = 1; h < MACC; ++h)
        tma_load_2d_hint(sa + (uint32_t)h * a_bytes, h == MACC - 1 ? &maps.w2[p] : &maps.w[p], k0, m0 + h * kMmaBM,
                         full(s), pol_w);
      tma_load_2d_hint(sa + b_off, &maps.x[p], k0, 0, full(s), pol_x);
    }
  } else if (RES && warp >= 2) {
    // idle during the main loop: ask L2 for the residual rows of this CTA's
    // epilogue (per rank and token, the tile's rows are contiguous), to be
    // kept there while the weights stream past
    const uint64_t pol = l2_evict_last();
    const int per_tok = n * MACC;
    // this CTA's epilogue tokens: in each of the rounds' ranges of W, its
    // slice of T (see mma_epilogue); a launch plan the epilogue rejects
    // prefetches nothing
    const int R = a.rounds >= 1 && a.rounds <= kMmaMaxRounds ? a.rounds : 1, W = NTILE / R,
              T = KS >= 1 && W % KS == 0 ? W / KS : 0;
    for (int j = threadIdx.x - 64; j < R * T * per_tok; j += THREADS - 64) {
      const int jt = j / per_tok, t = (jt / T) * W + (int)split * T + jt % T;
      const int q = (j % per_tok) / MACC, h = j % MACC;
      const int mh = m0 + h * kMmaBM, bmh = h == MACC - 1 ? bm_last : kMmaBM;
      const int nr = mh + bmh <= a.rows ? bmh : a.rows - mh;
      if (t >= a.tokens || nr <= 0) continue;
      const size_t off = ((size_t)t * a.rows + (size_t)mh) * 2;
      if (in_bounds(dc, a, kBufResidual, q, off, (size_t)nr * 2))
        l2_prefetch_bytes(static_cast<const char*>(a.res[q]) + off, (uint32_t)nr * 2u, pol);
    }
  } else if (warp == 1 && lane == 0) {  // MMA issuer
    const uint32_t idesc = mma_instr_desc(NTILE, a.fp16 != 0);
    for (int i = 0; i < nk; ++i) {
      const int s = i % S;
      if (!mma_mbar_wait(full(s), (uint32_t)((i / S) & 1), dc, mtile, (int)split)) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const uint32_t sa = base + (uint32_t)s * st_bytes, sb = sa + b_off;
#pragma unroll
      for (int kk = 0; kk < kMmaBK / 16; ++kk) {
        const uint64_t bd = mma_smem_desc(sb + (uint32_t)kk * 32u);
        const uint32_t accumulate = (i > 0 || kk > 0) ? 1u : 0u;
        for (int h = 0; h < MACC; ++h) {  // both accumulators share the token tile
          const uint64_t ad = mma_smem_desc(sa + (uint32_t)h * a_bytes + (uint32_t)kk * 32u);
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem + (uint32_t)h * acc_cols),
              "l"(ad), "l"(bd), "r"(idesc), "r"(accumulate)
              : "memory");
        }
      }
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(empty(s))
                   : "memory");
    }
    // arrives once every MMA issued above has completed (at once if none)
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(accf)
                 : "memory");
  }
  __syncwarp();

  const bool acc_ok = nk > 0 && mma_mbar_wait(accf, 0, dc, mtile, (int)split);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  float* part = reinterpret_cast<float*>(gbase);  // reuses the stage buffers (all loads consumed)
  // The epilogue's partial tile and inbox must fit the stage buffers and the
  // split must be one the epilogue knows: a launch that breaks this (the
  // host's shape search never makes one) is reported as an out-of-bounds
  // plan for the scratch space, and every CTA of the cluster skips the
  // epilogue alike, touching nothing outside its own shared memory.
  const bool plan_ok = (KS == 1 || KS == 2 || KS == 4 || KS == 8) && mma_round_fits(NTILE, S, MACC, KS, a.rounds);
  if (!plan_ok) {
    if (threadIdx.x == 0)
      atomicCAS(dc.status, 0ull, pack_bounds(mtile, kBufScratch, ((size_t)2 * NTILE) * kMmaBM * 4));
  } else {
    switch (KS) {
      case 1: mma_epilogue<1, MACC, THREADS, RES>(dc, a, tmem, acc_cols, part, inbar, n, split, m0, bm_last, acc_ok, mtile); break;
      case 2: mma_epilogue<2, MACC, THREADS, RES>(dc, a, tmem, acc_cols, part, inbar, n, split, m0, bm_last, acc_ok, mtile); break;
      case 4: mma_epilogue<4, MACC, THREADS, RES>(dc, a, tmem, acc_cols, part, inbar, n, split, m0, bm_last, acc_ok, mtile); break;
      default: mma_epilogue<8, MACC, THREADS, RES>(dc, a, tmem, acc_cols, part, inbar, n, split, m0, bm_last, acc_ok, mtile); break;
    }
  }
  __syncthreads();
  if (warp == 2) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols) : "memory");
}

const void* linear_allreduce_mma_kernel(int n, int macc, int threads, bool res);

}  // namespace dcc
