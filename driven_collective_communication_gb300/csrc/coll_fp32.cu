// coll_fp32.cu -- kernels of the sum collectives for fp32 elements.
#include "instantiate.cuh"

namespace dcc {
template <>
const void* reduce_kernel<float>(int kind, int n) {
  return reduce_kernel_impl<float>(kind, n);
}
}  // namespace dcc
