// instantiate.cuh -- kernel table of one element type (included by one .cu per type,
// so the four types compile in parallel).
#pragma once
#include "bulk.cuh"
#include "fused.cuh"
#include "ll.cuh"

namespace dcc {

template <typename T, int NT>
const void* pick_kernel(int kind) {
  switch (kind) {
    case kOneShot: return reinterpret_cast<const void*>(&k_allreduce_oneshot<T, NT>);
    case kTwoShot: return reinterpret_cast<const void*>(&k_allreduce_twoshot<T, NT>);
    case kTwoShotScratch: return reinterpret_cast<const void*>(&k_allreduce_twoshot_scratch<T, NT>);
    case kReduceScatter: return reinterpret_cast<const void*>(&k_reduce_scatter<T, NT>);
    case kTwoShotBulk: return reinterpret_cast<const void*>(&k_allreduce_twoshot_bulk<T, NT>);
    case kOneShotLL: return reinterpret_cast<const void*>(&k_allreduce_oneshot_ll<T, NT>);
    case kOneShotEB: return reinterpret_cast<const void*>(&k_allreduce_oneshot<T, NT, true>);
    case kTwoShotEB: return reinterpret_cast<const void*>(&k_allreduce_twoshot<T, NT, true>);
    case kTwoShotScratchEB: return reinterpret_cast<const void*>(&k_allreduce_twoshot_scratch<T, NT, true>);
    case kReduceScatterEB: return reinterpret_cast<const void*>(&k_reduce_scatter<T, NT, true>);
    default: return nullptr;
  }
}

template <typename T>
const void* reduce_kernel_impl(int kind, int n) {
  switch (n) {
    case 1: return pick_kernel<T, 1>(kind);
    case 2: return pick_kernel<T, 2>(kind);
    case 3: return pick_kernel<T, 3>(kind);
    case 4: return pick_kernel<T, 4>(kind);
    case 5: return pick_kernel<T, 5>(kind);
    case 6: return pick_kernel<T, 6>(kind);
    case 7: return pick_kernel<T, 7>(kind);
    case 8: return pick_kernel<T, 8>(kind);
    case 16: return pick_kernel<T, 16>(kind);
    default: return pick_kernel<T, 0>(kind);
  }
}

template <typename T>
const void* linear_kernel_impl(int n) {
  switch (n) {
    case 1: return reinterpret_cast<const void*>(&k_linear_allreduce<T, 1>);
    case 2: return reinterpret_cast<const void*>(&k_linear_allreduce<T, 2>);
    case 4: return reinterpret_cast<const void*>(&k_linear_allreduce<T, 4>);
    case 8: return reinterpret_cast<const void*>(&k_linear_allreduce<T, 8>);
    case 16: return reinterpret_cast<const void*>(&k_linear_allreduce<T, 16>);
    default: return reinterpret_cast<const void*>(&k_linear_allreduce<T, 0>);
  }
}

}  // namespace dcc
