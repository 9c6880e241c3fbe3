// coll_fused_mma.cu -- kernels of the tensor-core linear layer + AllReduce
// (any rank count: the kernel reads it from the communicator): one
// accumulator in 128-thread CTAs (two per SM) or 256-thread CTAs (one per
// SM), two accumulators in 256-thread CTAs.
#include "fused_mma.cuh"

namespace dcc {
const void* linear_allreduce_mma_kernel(int, int macc, int threads) {
  if (macc == 2) return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 2, kMmaThreads>);
  if (threads == kMmaPairThreads) return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 1, kMmaPairThreads>);
  return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 1, kMmaThreads>);
}
}  // namespace dcc
