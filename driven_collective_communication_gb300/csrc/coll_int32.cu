// coll_int32.cu -- kernels of the sum collectives for int32 elements.
#include "instantiate.cuh"

namespace dcc {
template <>
const void* reduce_kernel<int32_t>(int kind, int n) {
  return reduce_kernel_impl<int32_t>(kind, n);
}
}  // namespace dcc
