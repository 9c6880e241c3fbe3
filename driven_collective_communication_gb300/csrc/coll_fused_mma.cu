// coll_fused_mma.cu -- kernels of the tensor-core linear layer + AllReduce
// (any rank count: the kernel reads it from the communicator), with one or
// two accumulators per CTA.
#include "fused_mma.cuh"

namespace dcc {
const void* linear_allreduce_mma_kernel(int, int macc) {
  return macc == 2 ? reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 2>)
                   : reinterpret_cast<const void*>(&k_linear_allreduce_mma<0, 1>);
}
}  // namespace dcc
