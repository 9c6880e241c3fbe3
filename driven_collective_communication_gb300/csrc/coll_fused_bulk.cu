// coll_fused_bulk.cu -- kernel table of the bulk-copy-fed linear layer + AllReduce.
#include "fused_bulk.cuh"

namespace dcc {
template <typename T>
static const void* linear_bulk_impl(int n) {
  switch (n) {
    case 1: return reinterpret_cast<const void*>(&k_linear_allreduce_bulk<T, 1>);
    case 2: return reinterpret_cast<const void*>(&k_linear_allreduce_bulk<T, 2>);
    case 4: return reinterpret_cast<const void*>(&k_linear_allreduce_bulk<T, 4>);
    case 8: return reinterpret_cast<const void*>(&k_linear_allreduce_bulk<T, 8>);
    case 16: return reinterpret_cast<const void*>(&k_linear_allreduce_bulk<T, 16>);
    default: return reinterpret_cast<const void*>(&k_linear_allreduce_bulk<T, 0>);
  }
}
template <>
const void* linear_allreduce_bulk_kernel<__nv_bfloat16>(int n) {
  return linear_bulk_impl<__nv_bfloat16>(n);
}
template <>
const void* linear_allreduce_bulk_kernel<__half>(int n) {
  return linear_bulk_impl<__half>(n);
}
}  // namespace dcc
