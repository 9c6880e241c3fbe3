// coll_allgather.cu -- AllGather kernel table (a bit copy; element type only sets the size).
#include "allgather.cuh"
#include "bulk.cuh"

namespace dcc {
const void* allgather_kernel(int n) {
  switch (n) {
    case 1: return reinterpret_cast<const void*>(&k_allgather<1>);
    case 2: return reinterpret_cast<const void*>(&k_allgather<2>);
    case 4: return reinterpret_cast<const void*>(&k_allgather<4>);
    case 8: return reinterpret_cast<const void*>(&k_allgather<8>);
    case 16: return reinterpret_cast<const void*>(&k_allgather<16>);
    default: return reinterpret_cast<const void*>(&k_allgather<0>);
  }
}
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
