/* allreduce_8_ranks.c -- calling libdcc from C: an 8-rank bf16 sum
 * AllReduce over caller-owned device buffers on one GPU.
 *
 * Build: gcc -std=c11 -I include -I $CUDA_HOME/include -c allreduce_8_ranks.c
 *        and link with -L driven_collective_communication_gb300 -ldcc -lcudart.
 */
#include <cuda_runtime.h>
#include "dcc.h"

int allreduce_8_ranks(void* const* send, void* const* recv, size_t count, cudaStream_t s) {
  /* send[r], recv[r]: device buffers of count bf16 elements, 16-byte aligned */
  dcc_comm_t c;
  int rc = dcc_comm_create(8, &c);
  if (rc) return rc;
  for (int r = 0; r < 8; ++r) {
    dcc_register_buffer(c, r, DCC_BUF_INPUT, send[r], count * 2);
    dcc_register_buffer(c, r, DCC_BUF_OUTPUT, recv[r], count * 2);
  }
  for (int a = 0; a < 8; ++a)
    for (int b = 0; b < 8; ++b)
      if (a != b) dcc_memory_channel_make(c, a, b);
  rc = dcc_allreduce(c, send, recv, count, DCC_BF16, DCC_ALGO_AUTO, (dcc_stream_t)s);
  if (!rc) rc = dcc_comm_check(c, (dcc_stream_t)s);   /* synchronises s, reads the device status */
  dcc_comm_destroy(c);
  return rc;   /* 0 or a dcc_result_t; dcc_error_string(rc) names it */
}
