/*
 * dcc.h -- C ABI of libdcc, GB300-native virtual-rank collectives.
 *
 * N "virtual ranks" live on one GPU: rank r owns its own input, output and
 * scratch allocations in HBM, and in every collective kernel rank r is a group
 * of CTAs.  Ranks talk through MemoryChannels -- the memory-mapped channel of
 * the MSCCL++ README ("PortChannel and MemoryChannel"): GPU threads read and
 * write the peer's memory directly, and synchronise with signal/flush/wait
 * ("On-GPU Communication Interfaces: Channels").  As that section describes,
 * the host side creates the channels and a device copy of them exists before
 * the first launch.  The collectives are the usual sum collectives that point
 * (3) of the MSCCL++ abstract offers as ready-made algorithms; AllReduce is
 * the one the project summary singles out ("Highlighted Details":
 * tensor-parallel LLM serving).
 *
 * Conventions for every function below:
 *  - Return value: DCC_OK (0) or a negative dcc_result_t.  dcc_error_string()
 *    names it.  A host-side error returns before anything is launched.
 *  - Pointers named dev_* / send / recv are DEVICE addresses on the GPU the
 *    communicator was created on; the arrays that hold them (send[], recv[])
 *    are HOST arrays of n_ranks entries.  Pointers named host_* are host
 *    addresses (pinned memory recommended).
 *  - Ownership: the caller owns every data buffer and every stream.  The
 *    library owns only what dcc_comm_create allocates (semaphores, waiter
 *    counters, the channel table, the status word) and frees it in
 *    dcc_comm_destroy.  No data-path call allocates memory.
 *  - Streams: dcc_stream_t is a cudaStream_t passed as an opaque pointer;
 *    NULL is the legacy default stream.  Collectives are asynchronous on it.
 *  - Device failures (a wait that gave up) do not abort the process: the
 *    kernel records them in a status word and returns; dcc_comm_check reads it.
 *  - Layout: every buffer is a dense 1-D array of `count` elements of the
 *    given type, native (little-endian) storage; bf16 and fp16 are raw 16-bit
 *    IEEE patterns.  Data pointers must be 16-byte aligned.
 *  - Threading: a communicator is not thread-safe; serialise calls on it.
 *  - Concurrency on the GPU: kernels that synchronise ranks (in-place
 *    ONE_SHOT, TWO_SHOT_SCRATCH, ONE_SHOT_LL, the ring barrier, the channel
 *    primitives, anything with the entry barrier on) use the communicator's
 *    semaphores and waiter counts; two of them must not run at the same time
 *    on one communicator (issue them on one stream, or use one communicator
 *    per stream).  Kernels that never wait (out-of-place ONE_SHOT, TWO_SHOT,
 *    ReduceScatter, AllGather, the fused linear layer) may overlap freely.
 *  - Stream order with programmatic dependent launch: the kernels that never
 *    wait launch so that they may begin while the previous kernel on the
 *    stream finishes, and wait on the device for it to complete before they
 *    touch memory (dcc_set_pdl); the order a stream gives is kept either way.
 *  - Reductions: the sum everywhere; MAX and MIN through dcc_allreduce_op /
 *    dcc_reduce_scatter_op; the fused layer optionally adds a residual per
 *    rank (dcc_linear_allreduce_residual).
 */
#ifndef DCC_H
#define DCC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DCC_MAX_RANKS 16            /* virtual ranks per communicator */
#define DCC_MAX_BLOCKS_PER_RANK 128 /* CTAs per rank of a kernel that synchronises ranks */
#define DCC_MAX_WINDOWS 8           /* registered windows per (rank, kind) */

typedef struct dcc_comm* dcc_comm_t;
typedef void* dcc_stream_t; /* cudaStream_t */

typedef enum {
  DCC_OK = 0,
  DCC_ERR_INVALID_ARG = -1,    /* bad rank, count, enum value, NULL, overlap */
  DCC_ERR_NOT_REGISTERED = -2, /* a data range lies outside the rank's windows */
  DCC_ERR_MISALIGNED = -3,     /* a data pointer is not 16-byte aligned */
  DCC_ERR_NO_CHANNEL = -4,     /* a (src, dst) channel the call needs was never made */
  DCC_ERR_CUDA = -5,           /* a CUDA runtime call failed */
  DCC_ERR_LAUNCH = -6,         /* the grid cannot be co-resident on this GPU */
  DCC_ERR_TIMEOUT = -7,        /* a device wait gave up (sticky for the communicator) */
  DCC_ERR_UNSUPPORTED = -8,    /* valid request the library does not implement */
  DCC_ERR_BOUNDS = -9          /* bounds-checked build: a kernel access fell outside the call's
                                  range; any build: a tensor-core layer launch whose epilogue would
                                  not fit its shared memory (the library's own shape search never
                                  makes one; nothing is written) -- sticky for the communicator */
} dcc_result_t;

typedef enum { DCC_INT32 = 0, DCC_FP32 = 1, DCC_FP16 = 2, DCC_BF16 = 3 } dcc_dtype_t;

/* Reduction of dcc_allreduce_op / dcc_reduce_scatter_op.  SUM is the
 * reduction of the pages' collectives; MAX and MIN are not on the pages and
 * follow the IEEE 754-2019 maximum / minimum operations (see dcc_allreduce_op). */
typedef enum { DCC_OP_SUM = 0, DCC_OP_MAX = 1, DCC_OP_MIN = 2 } dcc_red_op_t;

typedef enum {
  DCC_ALGO_AUTO = 0,   /* pick by message size from the measured crossover table */
  DCC_ALGO_ONE_SHOT = 1, /* every rank gets all N inputs and reduces its whole output */
  DCC_ALGO_TWO_SHOT = 2, /* rank r reduces shard r, then puts it into all N outputs */
  DCC_ALGO_TWO_SHOT_SCRATCH = 3, /* rank r reduces shard r into its scratch, signal/wait,
                                    then every rank gets all shards from the scratches */
  DCC_ALGO_TWO_SHOT_BULK = 4, /* TWO_SHOT through shared-memory tiles moved by the bulk
                                 asynchronous copy engine (TMA): bulk gets, bulk puts */
  DCC_ALGO_ONE_SHOT_LL = 5 /* ONE_SHOT with a low-latency packet protocol: data and flag travel
                              in the same 16-byte store, no signal/wait round trip; messages of
                              at most DCC_LL_MAX_BYTES per rank */
} dcc_algo_t;

#define DCC_LL_MAX_BYTES (256u << 10) /* largest message per rank of DCC_ALGO_ONE_SHOT_LL */

typedef enum { DCC_BUF_INPUT = 0, DCC_BUF_OUTPUT = 1, DCC_BUF_SCRATCH = 2 } dcc_buf_kind_t;

/* ------------------------------------------------------------------------ */
/* Set-up: the host-side objects of the README's "Host-Side Communication   */
/* Proxy" example (bootstrap + Communicator + connection set-up), collapsed */
/* into one process that owns all N virtual ranks.                          */
/* ------------------------------------------------------------------------ */

/* Create a communicator of n_ranks (1..DCC_MAX_RANKS) virtual ranks on the
 * CUDA device that is current on the calling thread.  Allocates and zeroes the
 * semaphore block, waiter counters, channel table and status word (the only
 * device memory the library owns).  *out receives the handle.  Errors:
 * INVALID_ARG (n_ranks out of range, out NULL; checked before any CUDA call),
 * CUDA (no device / allocation failed). */
int dcc_comm_create(int n_ranks, dcc_comm_t* out);

/* Synchronise the device, free everything dcc_comm_create allocated, and free
 * the handle.  NULL is a no-op. */
int dcc_comm_destroy(dcc_comm_t c);

/* Register [dev_ptr, dev_ptr + bytes) as a window of `kind` for `rank`.  Every
 * data range a collective touches must lie inside one window of that rank
 * (INPUT or OUTPUT kind for send/recv buffers; SCRATCH for the two-shot
 * scratch algorithm).  Up to DCC_MAX_WINDOWS per (rank, kind).  The first
 * INPUT and OUTPUT windows of a rank are the local/remote memory its channels
 * bind (see dcc_channel_put/get).  Errors: INVALID_ARG (rank, kind, NULL,
 * bytes == 0, table full), MISALIGNED (dev_ptr not 16-byte aligned). */
int dcc_register_buffer(dcc_comm_t c, int rank, dcc_buf_kind_t kind, void* dev_ptr,
                        size_t bytes);

/* Make the MemoryChannel from src_rank to dst_rank (idempotent): src may then
 * put into / get from dst's memory and signal dst's inbound semaphore for
 * src; dst waits on it through its own channel to src.  A collective over N
 * ranks needs the channel for every ordered pair r != p; the ring barrier
 * needs r -> (r+1) mod N.  Channels are uploaded to the device lazily before
 * the next launch.  Errors: INVALID_ARG (rank out of range, src == dst). */
int dcc_memory_channel_make(dcc_comm_t c, int src_rank, int dst_rank);

/* ------------------------------------------------------------------------ */
/* Collectives (sum; MAX / MIN through the _op calls).  Per element, ranks  */
/* are added in order 0..N-1 starting                                       */
/* from rank 0's value; fp32/fp16/bf16 accumulate in fp32 and round once    */
/* (round-to-nearest-even) to the output type; int32 wraps.  Results are    */
/* therefore the same bits for every algorithm and every launch shape.      */
/* ------------------------------------------------------------------------ */

/* AllReduce: recv[r][i] = sum_p send[p][i] for every rank r, i < count.
 * send[r] == recv[r] is in-place for rank r; any other overlap between the
 * ranges is rejected.  algo selects the schedule (AUTO uses the crossover
 * table, see dcc_select_algo).  count == 0 is a no-op.  Errors: INVALID_ARG,
 * NOT_REGISTERED, MISALIGNED, NO_CHANNEL, LAUNCH, CUDA, TIMEOUT (a previous
 * device failure on this communicator). */
int dcc_allreduce(dcc_comm_t c, void* const* send, void* const* recv, size_t count,
                  dcc_dtype_t t, dcc_algo_t a, dcc_stream_t s);

/* ReduceScatter: recv[r][j] = sum_p send[p][r*recv_count + j], j < recv_count.
 * send[p] holds N*recv_count elements.  Ranges must not overlap. */
int dcc_reduce_scatter(dcc_comm_t c, void* const* send, void* const* recv, size_t recv_count,
                       dcc_dtype_t t, dcc_stream_t s);

/* AllReduce with a chosen reduction: recv[r][i] = op over p of send[p][i],
 * ranks combined in order 0..N-1.  DCC_OP_SUM is exactly dcc_allreduce.
 * DCC_OP_MAX / DCC_OP_MIN: the MSCCL++ pages describe sum collectives only;
 * these take the IEEE 754-2019 maximum / minimum -- a NaN in any rank gives
 * the type's canonical quiet NaN (fp32 0x7fc00000, fp16 0x7e00, bf16 0x7fc0),
 * -0 orders below +0, and otherwise the result is the bits of the largest /
 * smallest input (no rounding); int32 takes the signed maximum / minimum.
 * They run on the ONE_SHOT and TWO_SHOT schedules: AUTO picks between those
 * two by size as for the sum (two-shot where the sum would take another
 * schedule); any other explicit algo returns DCC_ERR_UNSUPPORTED.  Buffers,
 * in-place rules and errors as dcc_allreduce; an op outside dcc_red_op_t is
 * INVALID_ARG. */
int dcc_allreduce_op(dcc_comm_t c, void* const* send, void* const* recv, size_t count,
                     dcc_dtype_t t, dcc_red_op_t op, dcc_algo_t a, dcc_stream_t s);

/* ReduceScatter with a chosen reduction (same semantics as dcc_allreduce_op):
 * recv[r][j] = op over p of send[p][r*recv_count + j].  DCC_OP_SUM is exactly
 * dcc_reduce_scatter. */
int dcc_reduce_scatter_op(dcc_comm_t c, void* const* send, void* const* recv, size_t recv_count,
                          dcc_dtype_t t, dcc_red_op_t op, dcc_stream_t s);

/* AllGather: recv[p][q*send_count + j] = send[q][j] for all p, q, j < send_count.
 * recv[p] holds N*send_count elements.  Ranges must not overlap.  A bit copy:
 * t only fixes the element size.  Thread copies with eight 16-byte loads in
 * flight per thread and evict-first stores; DCC_AG_BULK=1 in the environment
 * at communicator creation sends inputs of at least 64 KiB per rank (a
 * multiple of 16 bytes) through the bulk-copy (TMA) kernel instead. */
int dcc_allgather(dcc_comm_t c, void* const* send, void* const* recv, size_t send_count,
                  dcc_dtype_t t, dcc_stream_t s);

/* Host-buffer AllReduce: host_recv[r] = sum_p host_send[p], as one
 * stream-ordered operation on s.  Two ways, same bits as dcc_allreduce:
 *  - zero copy (default when every host buffer is pinned memory the GPU can
 *    address, algo AUTO or TWO_SHOT; DCC_ZERO_COPY=0 turns it off): the
 *    two-shot kernel reads the host inputs and writes the host outputs over
 *    the host link directly; dev_send / dev_recv are checked but not touched;
 *  - staged: host_send[r] -> dev_send[r], dcc_allreduce(dev_send, dev_recv),
 *    dev_recv[r] -> host_recv[r], pipelined in 8 MiB-per-rank chunks: chunk i
 *    is copied in on the communicator's copy-in stream (one cudaMemcpyAsync
 *    per rank), reduced on s and copied out on its copy-out stream, so both
 *    copy directions and the kernels overlap.
 * The device buffers follow dcc_allreduce's rules; the host buffers must stay
 * valid until s has drained (pageable host memory makes the copies
 * synchronous). */
int dcc_allreduce_from_host(dcc_comm_t c, const void* const* host_send, void* const* host_recv,
                            void* const* dev_send, void* const* dev_recv, size_t count,
                            dcc_dtype_t t, dcc_algo_t a, dcc_stream_t s);

/* Row-parallel linear layer fused with the AllReduce (tensor-parallel decode;
 * the project summary's overlap of communication with computation): rank p holds
 * weight[p] (rows x kp, row-major) and x[p] (kp elements), and every rank
 * receives y[r][i] = R(sum_p sum_k weight[p][i*kp + k] * x[p][k]), i < rows.
 * One kernel, which puts the result into all N outputs; fp16/bf16; rows and
 * kp multiples of 8 (UNSUPPORTED otherwise); 16-byte aligned, registered,
 * outputs disjoint from every input.  Exact when every fp32 partial sum is
 * exact (small-integer data), else within the fp32 dot-product error bound of
 * the kernel that ran, before the final rounding.  The kernel, by kp:
 *  - up to 3584: the tensor-core kernel of dcc_linear_allreduce_tokens with
 *    one token (the tensor core's accumulation order, then the K-split
 *    partials in split order);
 *  - above: rank r's CTAs compute shard r of the rows with fp32 dot products
 *    in a fixed lane/shuffle order, the ranks' partials added in rank order,
 *    the weights streamed through shared memory by bulk copies (TMA);
 *  - on request the same with thread loads instead of bulk copies.
 * DCC_FUSED_KERNEL=thread|bulk|tensor (DCC_FUSED_BULK=0 / 1 for the first
 * two) in the environment at communicator creation forces one. */
int dcc_linear_allreduce(dcc_comm_t c, void* const* weight, void* const* x, void* const* y, size_t rows,
                         size_t kp, dcc_dtype_t t, dcc_stream_t s);

/* The same layer with a residual per output rank (the tensor-parallel
 * residual stream, h <- h + layer(h)): y[r][i] = R( sum_p sum_k W_p[i][k]
 * x_p[k] + residual[r][i] ).  The residual joins the fp32 sum before the one
 * rounding (the reading taken for the fused epilogue; the pages give none).
 * residual[r] holds rows elements of t, registered and 16-byte aligned like
 * y[r]; residual[r] == y[r] updates the residual in place, any other overlap
 * with an output is rejected.  Shapes, kernels, results on small-integer data
 * and errors as dcc_linear_allreduce; residual NULL is INVALID_ARG. */
int dcc_linear_allreduce_residual(dcc_comm_t c, void* const* weight, void* const* x, void* const* residual,
                                  void* const* y, size_t rows, size_t kp, dcc_dtype_t t, dcc_stream_t s);

/* The same row-parallel layer for a batch of tokens, on the tensor cores
 * (batched decode, speculative decoding, prefill chunks): rank p holds
 * weight[p] (rows x kp, row-major) and x[p] (tokens x kp, row-major: token
 * t's slice of the contraction dimension at x[p] + t*kp), and every rank
 * receives
 *   y[r][t*rows + i] = R( sum_p sum_k weight[p][i*kp + k] * x[p][t*kp + k] ),
 * y[r] holding tokens x rows elements, row-major.  One kernel: tiles of up
 * to 128 rows of y (up to 256 with two accumulators), tcgen05 MMAs on bf16 /
 * fp16 operands loaded by TMA with fp32 accumulation in tensor memory, the
 * contraction split across the CTAs of a thread-block cluster whose partials
 * meet through bulk copies between their shared memories, one rounding, and
 * the result put into all N outputs.  The launch is planned for three forms
 * (128-thread CTAs two to an SM with a deeper split; 256-thread CTAs one to
 * an SM with one accumulator, or with two): of the first two the one whose
 * grid fits one wave, whose epilogue takes one round and whose split is
 * deepest runs, the third only where it alone fits one wave (with 8192 rows:
 * the first up to 96 tokens, the second above);
 * DCC_MMA_FORM=pair|one|two at communicator creation forces a form (results
 * as above in every form).
 * fp16 or bf16; tokens
 * 1..256, kp and rows multiples of 8 (UNSUPPORTED otherwise; a kp that is
 * not a multiple of 64 ends in a partial 64-column block, zero-filled by the
 * TMA); 16-byte aligned, registered, outputs disjoint from every input.
 * Exact when every fp32 partial sum is exact (small-integer data), otherwise
 * within the fp32 dot-product error bound plus the one rounding (the tensor
 * core's accumulation order).  Errors as dcc_linear_allreduce. */
int dcc_linear_allreduce_tokens(dcc_comm_t c, void* const* weight, void* const* x, void* const* y, size_t tokens,
                                size_t rows, size_t kp, dcc_dtype_t t, dcc_stream_t s);

/* The batched layer with a residual per output rank (the residual stream of
 * a multi-token step, h <- h + layer(h)):
 *   y[r][t*rows + i] = R( sum_p sum_k weight[p][i*kp + k] * x[p][t*kp + k]
 *                         + residual[r][t*rows + i] ).
 * The residual joins the fp32 sum before the one rounding (the reading taken
 * for the fused epilogue; the pages give none).  residual[r] holds tokens x
 * rows elements of t laid out like y[r], registered and 16-byte aligned;
 * residual[r] == y[r] updates the residual in place, any other overlap with
 * an output is rejected.  Shapes, kernel, results on small-integer data and
 * errors as dcc_linear_allreduce_tokens; residual NULL is INVALID_ARG. */
int dcc_linear_allreduce_tokens_residual(dcc_comm_t c, void* const* weight, void* const* x, void* const* residual,
                                         void* const* y, size_t tokens, size_t rows, size_t kp, dcc_dtype_t t,
                                         dcc_stream_t s);

/* Ring barrier (the README's two-rank barrier, "signal, flush, wait", chained
 * around all N ranks): per iteration rank 0 signals rank 1 and waits for rank
 * N-1; rank r > 0 waits for rank r-1 and then signals rank (r+1) mod N.  One
 * kernel runs all `iters` (>= 0) iterations.  With at most 8 ranks the ranks
 * are the CTAs of one thread-block cluster and each signal is a cluster-scope
 * release arrive on the next rank's shared-memory barrier (DCC_RING_CLUSTER=0
 * at communicator creation keeps the global-memory semaphores); either way
 * the channels' signal counters advance by one per iteration and hop. */
int dcc_ring_barrier(dcc_comm_t c, int iters, dcc_stream_t s);

/* Synchronise s, read the device status word and return DCC_OK or the first
 * device failure (DCC_ERR_TIMEOUT).  A failure is sticky: the semaphores are
 * unbalanced afterwards, so the communicator must be destroyed. */
int dcc_comm_check(dcc_comm_t c, dcc_stream_t s);

/* After dcc_comm_check returned a failure: the rank, peer and block of the
 * wait that gave up (any pointer may be NULL).  INVALID_ARG if none.
 * For DCC_ERR_BOUNDS (the bounds-checked build, libdcc_checked.so, compiled
 * with DCC_CHECK_BOUNDS=1: every data access of the collectives and the fused
 * layer is checked against the byte range the call gave each pointer; the
 * first access outside is skipped and recorded, and the kernel runs to its
 * normal end): *rank = the buffer's rank, *peer = the buffer (0 send / weight,
 * 1 recv / y, 2 scratch, 3 x, 4 residual), *block = the offending byte offset
 * from that pointer / 16 (saturating at INT_MAX). */
int dcc_comm_error_detail(dcc_comm_t c, int* rank, int* peer, int* block);

/* Name of a dcc_result_t (static storage). */
const char* dcc_error_string(int code);

/* ------------------------------------------------------------------------ */
/* AllReduce without any allocation.  The MSCCL++ pages have no counterpart */
/* to this entry point; it exists for callers that cannot call cudaMalloc   */
/* when they need the collective -- a framework whose caching allocator     */
/* owns all device memory, a serving loop that cannot afford cudaMalloc's   */
/* implicit device synchronisation, a deployment with a fixed audited       */
/* memory budget -- and so cannot create a communicator.                    */
/* ------------------------------------------------------------------------ */

#define DCC_NOALLOC_MAX_BYTES (4u << 20) /* largest message per rank: 4 MiB */

/* Two-shot AllReduce through scratch (DCC_ALGO_TWO_SHOT_SCRATCH semantics and
 * bits) over n_ranks (1..DCC_MAX_RANKS) virtual ranks on the current device,
 * with no communicator, no registration and no channel set-up.  The caller
 * passes inputs and outputs only (send[r] == recv[r] is in place; other
 * overlaps are rejected; 16-byte alignment as for dcc_allreduce).  All
 * working memory -- reduced shards, semaphores, waiter counts, status word --
 * lives in one fixed device array of DCC_NOALLOC_MAX_BYTES plus 1.25 MiB that
 * every GPU that loads the library holds until the process exits.
 *  - Never allocates: no cudaMalloc/cudaFree or other allocating call.
 *  - The first call on a device (of this function or dcc_noalloc_check) sets
 *    that device up once: it resolves the array's device address, zeroes its
 *    synchronisation part and synchronises the device; make that first call
 *    before any stream capture.  Later calls only launch the kernel.
 *  - Calls share the array: calls that overlap on the GPU (on different
 *    streams, or from several host threads) race and must not be issued.
 *    Nothing is cleared between calls: a call that completes leaves every
 *    semaphore it used balanced (as many waits as signals), which is all the
 *    next call needs.
 *  - A device wait that runs out (the same bounded waits as the communicator
 *    path; limit DCC_WAIT_TIMEOUT_US, read at set-up) leaves that call's
 *    outputs incomplete and records the failure in the array's status word.
 *    It stays recorded, and outputs of later calls carry no guarantee, until
 *    dcc_noalloc_check has reported it.
 * Errors: INVALID_ARG (n_ranks, NULL, dtype, overlap), MISALIGNED,
 * UNSUPPORTED (count * element size > DCC_NOALLOC_MAX_BYTES), LAUNCH, CUDA. */
int dcc_allreduce_noalloc(int n_ranks, void* const* send, void* const* recv, size_t count,
                          dcc_dtype_t t, dcc_stream_t s);

/* Failure report of dcc_allreduce_noalloc on the current device.  Synchronises
 * s (the stream of the calls to check), reads the array's status word (a copy
 * into host memory; nothing is allocated) and returns DCC_OK, or
 * DCC_ERR_TIMEOUT with the rank, peer and block of the first wait that gave up
 * (any pointer may be NULL).  After a failure it zeroes the array's
 * synchronisation part (and synchronises the device), so the next call starts
 * clean.  Errors: CUDA. */
int dcc_noalloc_check(dcc_stream_t s, int* rank, int* peer, int* block);

/* ------------------------------------------------------------------------ */
/* MemoryChannel primitives on their own (README, "On-GPU Communication     */
/* Interfaces: Channels": put copies from local to remote memory; signal,   */
/* flush, wait synchronise a pair of ranks).  The channel src -> dst binds  */
/* src's first INPUT window as local source, src's first OUTPUT window as   */
/* local destination, dst's first INPUT window as remote source and dst's  */
/* first OUTPUT window as remote destination.                              */
/* ------------------------------------------------------------------------ */

/* put: dst.OUTPUT[remote_off, +bytes) <- src.INPUT[local_off, +bytes), by one
 * CTA of warp-cooperative 16-byte vector stores; then, if signal != 0, flush
 * and signal dst, and dst's CTA waits for that signal before the kernel ends.
 * Offsets and bytes must be multiples of 16 and inside the windows. */
int dcc_channel_put(dcc_comm_t c, int src_rank, int dst_rank, size_t remote_off,
                    size_t local_off, size_t bytes, int signal, dcc_stream_t s);

/* get: src.OUTPUT[local_off, +bytes) <- dst.INPUT[remote_off, +bytes). */
int dcc_channel_get(dcc_comm_t c, int src_rank, int dst_rank, size_t remote_off,
                    size_t local_off, size_t bytes, dcc_stream_t s);

/* Copy the semaphore state of block slot `block` to the host: inbound[d*N+s]
 * = signals rank d has received from rank s; expected[d*N+s] = waits rank d
 * has completed on rank s.  Each array holds N*N uint64 (NULL to skip).
 * Synchronises s. */
int dcc_comm_read_semaphores(dcc_comm_t c, int block, uint64_t* inbound, uint64_t* expected,
                             dcc_stream_t s);

/* ------------------------------------------------------------------------ */
/* PortChannels and the host-side proxy (README, "PortChannel and           */
/* MemoryChannel", "Host-Side Communication Proxy").  One GPU thread pushes */
/* 16-byte triggers {fst, snd} into a FIFO in pinned host memory; a proxy   */
/* thread of the communicator pops them and carries them out: PUT = a      */
/* cudaMemcpyAsync device-to-device on a copy engine from the source rank's */
/* first INPUT window to the destination rank's first OUTPUT window; SIGNAL */
/* and FLUSH = value writes the GPU polls (bounded).  Copies and signals to */
/* rank d run in FIFO order on proxy stream d % K (K = 4, or               */
/* DCC_PROXY_STREAMS = 1..8 at the proxy's first start), so K copy engines  */
/* work at once; a FLUSH is written after every stream's earlier work.  A   */
/* trigger whose fst is non-zero with bit 63 clear is a custom trigger for  */
/* the installed handler.  Windows must not change while the proxy runs.    */
/* The GPU must not multiplex a proxy stream onto the hardware queue of a   */
/* kernel that waits for it: with many streams set                          */
/* CUDA_DEVICE_MAX_CONNECTIONS=32 before the CUDA context exists.           */
/* ------------------------------------------------------------------------ */

typedef void (*dcc_trigger_handler_t)(uint64_t fst, uint64_t snd, void* user);

/* Start / stop the proxy thread (ProxyService startProxy/stopProxy).  The first
 * start allocates the FIFO (pinned host memory), the completion words and the
 * proxy's streams; every start loads all of libdcc's kernels into the context.
 * PortChannel kernels wait on the proxy's CUDA calls: a host call that waits
 * for the running kernels (the first launch of a kernel under lazy module
 * loading, a device-wide synchronisation) stalls the proxy until the waiting
 * kernel's limit runs out.  Load the application's own kernels before running
 * PortChannel kernels (e.g. CUDA_MODULE_LOADING=EAGER).  Stop reads how many triggers GPU threads have claimed
 * (call it after the pushing kernels have finished), lets the thread carry
 * those out (at most 5 s), joins it, waits for the proxy's copies, and returns
 * DCC_OK or the first error a trigger hit (NOT_REGISTERED, CUDA). */
int dcc_proxy_start(dcc_comm_t c);
int dcc_proxy_stop(dcc_comm_t c);

/* Install the handler for custom triggers (custom proxy); proxy stopped.
 * fn runs on the proxy thread, in FIFO order.  NULL removes it. */
int dcc_proxy_set_handler(dcc_comm_t c, dcc_trigger_handler_t fn, void* user);

/* Triggers the proxy has taken so far, and how many were custom.  Returns the
 * proxy's first error (or DCC_OK).  INVALID_ARG before the first start. */
int dcc_proxy_stats(dcc_comm_t c, uint64_t* processed, uint64_t* custom);

/* Diagnostic snapshot (synchronous): words[0..5] = FIFO head (claimed by GPU
 * threads), tail (taken by the proxy), flush word, triggers processed, custom
 * triggers, first error; then N*N port signal counts [dst][src] and N*N
 * completed port waits [dst][src].  nwords >= 6 + 2*N*N. */
int dcc_proxy_state(dcc_comm_t c, uint64_t* words, int nwords);

/* PortChannel put: one GPU thread of src pushes PUT (+SIGNAL if signal != 0)
 * for dst.OUTPUT[remote_off, +bytes) <- src.INPUT[local_off, +bytes); with
 * flush != 0 it then waits until the proxy has carried the copy out; with
 * signal != 0 a thread of dst waits for the signal.  Offsets and bytes are
 * multiples of 16.  Needs a running proxy (INVALID_ARG otherwise). */
int dcc_port_put(dcc_comm_t c, int src_rank, int dst_rank, size_t remote_off, size_t local_off,
                 size_t bytes, int signal, int flush, dcc_stream_t s);

/* AllGather through PortChannels (copy engines driven by the proxy):
 * recv[p][q*send_count + j] = send[q][j].  send[q] must lie in rank q's first
 * INPUT window and recv[p] in rank p's first OUTPUT window; send_count *
 * element size must be a multiple of 16.  Same result as dcc_allgather. */
int dcc_port_allgather(dcc_comm_t c, void* const* send, void* const* recv, size_t send_count,
                       dcc_dtype_t t, dcc_stream_t s);

/* Push `count` (<= 32) custom triggers {fst[i], snd[i]} from one GPU thread
 * (snd may be NULL: zeros).  fst[i] must be non-zero with bit 63 clear. */
int dcc_fifo_push(dcc_comm_t c, const uint64_t* fst, const uint64_t* snd, int count, dcc_stream_t s);

/* ------------------------------------------------------------------------ */
/* Tuning and test knobs.                                                   */
/* ------------------------------------------------------------------------ */

/* Wait limit of every device-side wait, microseconds (default 2,000,000, or
 * DCC_WAIT_TIMEOUT_US from the environment at create time). */
int dcc_set_wait_timeout_us(dcc_comm_t c, uint64_t us);

/* CTAs per rank for the collectives; 0 = choose by size (default, or
 * DCC_BLOCKS_PER_RANK from the environment).  Kernels that synchronise ranks
 * clamp it to one co-resident wave and DCC_MAX_BLOCKS_PER_RANK; streaming
 * kernels that never wait otherwise size their grid to cover the work. */
int dcc_set_blocks_per_rank(dcc_comm_t c, int blocks);

/* Entry barrier (off by default; also DCC_ENTRY_BARRIER=1 in the environment
 * at creation).  When on, every CTA of the AllReduce (ONE_SHOT, TWO_SHOT,
 * TWO_SHOT_SCRATCH), ReduceScatter and AllGather kernels first signals the
 * CTAs of its block slot in every other rank ("my input is ready") and waits
 * for their signals before it touches peer memory -- the step a multi-GPU
 * collective needs before reading a peer's input (MSCCL++ README, "Channels":
 * signal/wait).  On one GPU stream order already orders the ranks' inputs
 * before the kernel, so the barrier only adds its cost.  Those kernels then
 * launch cooperatively with at most one wave of CTAs; ONE_SHOT_LL and
 * TWO_SHOT_BULK have no entry barrier and return DCC_ERR_UNSUPPORTED while it
 * is on.  A wait that runs out is reported by dcc_comm_check. */
int dcc_set_entry_barrier(dcc_comm_t c, int on);

/* Programmatic dependent launch (on by default; DCC_PDL=0 in the environment
 * at creation turns it off).  The kernels whose CTAs never wait on one
 * another -- out-of-place ONE_SHOT, TWO_SHOT, TWO_SHOT_BULK, ReduceScatter,
 * AllGather and the fused linear layer, each without the entry barrier -- are
 * launched with programmatic stream serialization: the launch may begin while
 * the previous kernel on the stream is still finishing, and the kernel's
 * first instruction waits until that kernel has completed and its writes are
 * visible, so stream order is kept.  This hides most of the gap between
 * dependent launches (the next kernel must be launched the same way to gain
 * from it in turn).  Synchronising kernels always launch in plain stream
 * order.  Errors: INVALID_ARG (c NULL). */
int dcc_set_pdl(dcc_comm_t c, int on);

/* AUTO picks ONE_SHOT for out-of-place messages of at most `bytes` per rank
 * and TWO_SHOT above, for this dtype, on this communicator.  The default is
 * dcc_auto_threshold(n_ranks, t). */
int dcc_set_algo_threshold(dcc_comm_t c, dcc_dtype_t t, size_t bytes);

/* The default of that threshold for a communicator of n_ranks (1..16) and
 * dtype t: the measured crossover table compiled into the library (one-shot
 * up to the largest measured size at which it was never slower than
 * two-shot, CUDA-graph-amortised, on GB300).  Pure host logic, no GPU.
 * Errors: INVALID_ARG (n_ranks, t, bytes NULL). */
int dcc_auto_threshold(int n_ranks, dcc_dtype_t t, size_t* bytes);

/* The algorithm AUTO would run for this request (pure host logic). */
int dcc_select_algo(dcc_comm_t c, size_t count, dcc_dtype_t t, dcc_algo_t* out);

/* Test knob: rank `rank` skips every signal it would send (-1 = off), so its
 * peers' waits run out and report DCC_ERR_TIMEOUT.  Nothing faults. */
int dcc_debug_skip_signal(dcc_comm_t c, int rank);

/* Launch shape a collective would use: CTAs per rank and threads per CTA
 * (0 when no launch is needed).  Pure host logic except the occupancy query. */
int dcc_launch_shape(dcc_comm_t c, size_t count, dcc_dtype_t t, dcc_algo_t a, int* blocks_per_rank,
                     int* threads);

/* Two-shot shard of `rank` for `count` elements of `elem_bytes` each over
 * n_ranks ranks, in elements: [*begin, *end).  Shards are whole 16-byte
 * vectors; the last rank also takes the remainder.  Pure host logic, no GPU. */
int dcc_shard_range(size_t count, int n_ranks, int rank, size_t elem_bytes, size_t* begin,
                    size_t* end);

/* Library version string (static storage). */
const char* dcc_version(void);

/* Compute capability the library's device code was built for, as the CUDA
 * runtime reports it for every kernel of the library on the current device
 * (binaryVersion, e.g. 103 for sm_103a).  *version receives it when all
 * kernels agree.  Errors: INVALID_ARG (version NULL), CUDA (no device, or a
 * kernel that cannot load), UNSUPPORTED (kernels built for different
 * architectures). */
int dcc_kernel_binary_version(int* version);

#ifdef __cplusplus
}
#endif
#endif /* DCC_H */
