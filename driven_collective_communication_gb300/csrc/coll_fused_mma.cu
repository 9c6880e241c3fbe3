// coll_fused_mma.cu -- kernels of the tensor-core linear layer + AllReduce
// (any rank count: the kernel reads it from the communicator): one
// accumulator in 128-thread CTAs (two per SM) or 256-thread CTAs (one per
// SM), two accumulators in 256-thread CTAs; each without and with residuals.
#include "fused_mma.cuh"

namespace dcc {
const void* linear_allreduce_mma_kernel(int, int macc, int threads, bool res) {
  if (res) {
    if (macc == 2) return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 2, kMmaThreads, true>);
    if (threads == kMmaPairThreads) return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 1, kMmaPairThreads, true>);
    return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 1, kMmaThreads, true>);
  }
  if (macc == 2) return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 2, kMmaThreads, false>);
  if (threads == kMmaPairThreads) return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 1, kMmaPairThreads, false>);
  return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 1, kMmaThreads, false>);
}
}  // namespace dcc
