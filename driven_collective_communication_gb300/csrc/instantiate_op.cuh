// instantiate_op.cuh -- MAX / MIN kernel table of one reduction (included by
// coll_max.cu and coll_min.cu, which compile in parallel).
#pragma once
#include "collectives.cuh"

namespace dcc {

template <typename T, int OP, int NT>
const void* pick_op_kernel(int kind) {
  switch (kind) {
    case kOneShot: return reinterpret_cast<const void*>(&k_allreduce_oneshot<T, NT, false, OP>);
    case kTwoShot: return reinterpret_cast<const void*>(&k_allreduce_twoshot<T, NT, false, OP>);
    case kReduceScatter: return reinterpret_cast<const void*>(&k_reduce_scatter<T, NT, false, OP>);
    default: return nullptr;
  }
}

template <typename T, int OP>
const void* reduce_op_kernel_impl(int kind, int n) {
  switch (kind) {  // entry barrier: runtime-N instances serve every rank count
    case kOneShotEB: return reinterpret_cast<const void*>(&k_allreduce_oneshot<T, 0, true, OP>);
    case kTwoShotEB: return reinterpret_cast<const void*>(&k_allreduce_twoshot<T, 0, true, OP>);
    case kReduceScatterEB: return reinterpret_cast<const void*>(&k_reduce_scatter<T, 0, true, OP>);
    default: break;
  }
  // compile-time N for the power-of-two rank counts; the runtime-N instance
  // serves the others (fewer kernels to build for the rarer reductions)
  switch (n) {
    case 2: return pick_op_kernel<T, OP, 2>(kind);
    case 4: return pick_op_kernel<T, OP, 4>(kind);
    case 8: return pick_op_kernel<T, OP, 8>(kind);
    case 16: return pick_op_kernel<T, OP, 16>(kind);
    default: return pick_op_kernel<T, OP, 0>(kind);
  }
}

}  // namespace dcc
