// coll_fp16.cu -- kernels of the sum collectives for fp16 elements.
#include "instantiate.cuh"

namespace dcc {
template <>
const void* reduce_kernel<__half>(int kind, int n) {
  return reduce_kernel_impl<__half>(kind, n);
}
template <>
const void* linear_allreduce_kernel<__half>(int n) {
  return linear_kernel_impl<__half>(n);
}
}  // namespace dcc
