// coll_allgather.cu -- AllGather kernel table (a bit copy; element type only sets the size).
#include "allgather.cuh"
#include "bulk.cuh"

namespace dcc {
template <bool EB>
static const void* allgather_impl(int n) {
  switch (n) {
    case 1: return reinterpret_cast<const void*>(&k_allgather<1, EB>);
    case 2: return reinterpret_cast<const void*>(&k_allgather<2, EB>);
    case 4: return reinterpret_cast<const void*>(&k_allgather<4, EB>);
    case 8: return reinterpret_cast<const void*>(&k_allgather<8, EB>);
    case 16: return reinterpret_cast<const void*>(&k_allgather<16, EB>);
    default: return reinterpret_cast<const void*>(&k_allgather<0, EB>);
  }
}
const void* allgather_kernel(int n, bool eb) { return eb ? allgather_impl<true>(n) : allgather_impl<false>(n); }
const void* allgather_bulk_kernel(int n) {
  switch (n) {
    case 1: return reinterpret_cast<const void*>(&k_allgather_bulk<1>);
    case 2: return reinterpret_cast<const void*>(&k_allgather_bulk<2>);
    case 4: return reinterpret_cast<const void*>(&k_allgather_bulk<4>);
    case 8: return reinterpret_cast<const void*>(&k_allgather_bulk<8>);
    case 16: return reinterpret_cast<const void*>(&k_allgather_bulk<16>);
    default: return reinterpret_cast<const void*>(&k_allgather_bulk<0>);
  }
}
}  // namespace dcc
