// sync_kernels.cuh -- entry points of the ring-barrier and primitive kernels.
#pragma once

namespace dcc {
const void* ring_barrier_kernel();  // (DevComm, int iters); grid N x 32, cooperative
const void* ring_barrier_cluster_kernel();  // (DevComm, int iters); one cluster of N x 32 (N <= 8)
const void* channel_put_kernel();   // (DevComm, PrimArgs); grid 2 x 256, cooperative
const void* channel_get_kernel();   // (DevComm, PrimArgs); grid 1 x 256
}  // namespace dcc
