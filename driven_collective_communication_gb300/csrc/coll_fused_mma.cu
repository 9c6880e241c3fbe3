// coll_fused_mma.cu -- kernel of the tensor-core linear layer + AllReduce
// (any rank count: the kernel reads it from the communicator).
#include "fused_mma.cuh"

namespace dcc {
const void* linear_allreduce_mma_kernel(int) { return reinterpret_cast<const void*>(&k_linear_allreduce_mma<0>); }
}  // namespace dcc
