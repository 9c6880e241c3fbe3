// coll_min.cu -- MIN AllReduce and ReduceScatter kernels of the four element types.
#include "instantiate_op.cuh"

namespace dcc {
template <>
const void* reduce_op_kernel<int32_t, kOpMin>(int kind, int n) {
  return reduce_op_kernel_impl<int32_t, kOpMin>(kind, n);
}
template <>
const void* reduce_op_kernel<float, kOpMin>(int kind, int n) {
  return reduce_op_kernel_impl<float, kOpMin>(kind, n);
}
template <>
const void* reduce_op_kernel<__half, kOpMin>(int kind, int n) {
  return reduce_op_kernel_impl<__half, kOpMin>(kind, n);
}
template <>
const void* reduce_op_kernel<__nv_bfloat16, kOpMin>(int kind, int n) {
  return reduce_op_kernel_impl<__nv_bfloat16, kOpMin>(kind, n);
}
}  // namespace dcc
