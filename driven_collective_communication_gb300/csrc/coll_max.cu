// coll_max.cu -- MAX AllReduce and ReduceScatter kernels of the four element types.
#include "instantiate_op.cuh"

namespace dcc {
template <>
const void* reduce_op_kernel<int32_t, kOpMax>(int kind, int n) {
  return reduce_op_kernel_impl<int32_t, kOpMax>(kind, n);
}
template <>
const void* reduce_op_kernel<float, kOpMax>(int kind, int n) {
  return reduce_op_kernel_impl<float, kOpMax>(kind, n);
}
template <>
const void* reduce_op_kernel<__half, kOpMax>(int kind, int n) {
  return reduce_op_kernel_impl<__half, kOpMax>(kind, n);
}
template <>
const void* reduce_op_kernel<__nv_bfloat16, kOpMax>(int kind, int n) {
  return reduce_op_kernel_impl<__nv_bfloat16, kOpMax>(kind, n);
}
}  // namespace dcc
