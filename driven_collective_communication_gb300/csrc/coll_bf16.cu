// coll_bf16.cu -- kernels of the sum collectives for bf16 elements.
#include "instantiate.cuh"

namespace dcc {
template <>
const void* reduce_kernel<__nv_bfloat16>(int kind, int n) {
  return reduce_kernel_impl<__nv_bfloat16>(kind, n);
}
template <>
const void* linear_allreduce_kernel<__nv_bfloat16>(int n) {
  return linear_kernel_impl<__nv_bfloat16>(n);
}
}  // namespace dcc
