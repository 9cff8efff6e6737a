/*
 * rar.h -- C ABI of the ring AllReduce library (librar.so) for one GB300.
 *
 * N "virtual ranks" live in one GPU: every rank's send buffer, receive buffer
 * and connector FIFOs are ordinary device memory of that GPU, and one kernel
 * launch runs all ranks at once (one thread block per (rank, channel); for
 * large Simple and LL128 messages two blocks per (rank, channel), each moving
 * a fixed part of every step, when twice the grid fits the device's SMs).
 *
 * Pages the operations follow (cited by title and section):
 *   [C23] "NCCL 专家课程 23：Device Kernel、Primitives、Step/Credit 与 LL Flag"
 *   [C12] "NCCL 专家课程 12：Ring AllReduce 逐步推导、真实 Ring 与 Channel 并行"
 *   [NOTES] "NCCL" notes (cishoon.github.io), sections "2 CUDA stream",
 *           "5 Symmetric Memory"
 *   [OS89] "perf(osar): all-reduce 5커널 → 3커널 (가드·웨이트 프롤로그 융합) - #89"
 *
 * Conventions for every entry point:
 *  - Pointers named *buf*, workspace and the arrays they point to are DEVICE
 *    memory of the current CUDA device, owned by the caller; the library
 *    allocates nothing and keeps no pointer after a call returns.
 *  - Arrays of pointers (sendbufs, recvbufs) and ring_order are HOST arrays of
 *    nranks entries, read during the call only.
 *  - `stream` is a cudaStream_t (passed as void*). Work is enqueued on it and
 *    the call returns without waiting ([NOTES] "2 CUDA stream"). NULL means
 *    the legacy default stream, which serialises with other streams.
 *  - Argument errors are reported synchronously by the return value and
 *    enqueue nothing. Failures found on the device (a wait that ran out of
 *    time, a workspace not initialised for this call) are written to a status
 *    word in the workspace and read with rar_get_status().
 *  - Thread safety: calls that share a workspace must be ordered on one
 *    stream; calls on different workspaces are independent.
 *  - Environment: RAR_TRACE (set, and not "0") makes every call print its
 *    resolved geometry to stderr once its arguments have passed the checks
 *    that precede the workspace check (grid, block -> channel, each channel's
 *    range, loops and first chunk, chunk and slice sizes), and the kernel it
 *    launches; RAR_SPIN_TIMEOUT_NS sets the default time limit of every wait
 *    (rar_set_spin_timeout_ns overrides it).
 */
#ifndef RAR_H
#define RAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define RAR_API __attribute__((visibility("default")))
#else
#define RAR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rar_status {
  RAR_OK = 0,
  RAR_ERR_ARG = 1,         /* a bad argument: sizes, enums, chunkSteps, buffSize, aliasing */
  RAR_ERR_RING = 2,        /* ring_order is not one ring over all ranks ([C12] "Graph 如何变成完整 ring") */
  RAR_ERR_ALIGN = 3,       /* a buffer or the workspace is not 16-byte aligned */
  RAR_ERR_WORKSPACE = 4,   /* workspace too small, or not initialised for this configuration */
  RAR_ERR_CORESIDENCY = 5, /* the (rank, channel) blocks cannot all be resident at once */
  RAR_ERR_CUDA = 6,        /* a CUDA runtime call failed */
  RAR_ERR_TIMEOUT = 7,     /* device: a wait ran past its time limit; the kernel gave up */
  RAR_ERR_ABORT = 8,       /* device: the workspace was aborted by an earlier failure */
  RAR_ERR_BOUNDS = 9       /* device, debug library only: a slice fell outside its buffers */
} rar_status;

typedef enum rar_dtype { RAR_F32 = 0, RAR_BF16 = 1 } rar_dtype;
typedef enum rar_redop { RAR_SUM = 0 } rar_redop;
typedef enum rar_proto { RAR_LL = 0, RAR_LL128 = 1, RAR_SIMPLE = 2 } rar_proto;

#define RAR_NCCL_STEPS 8    /* slots of every connector FIFO ([C23] "Simple 的 Credit 与 Step") */
#define RAR_MAX_RANKS 32
#define RAR_MAX_CHANNELS 64 /* bits of channelMask */

/*
 * Bytes of device workspace a ring AllReduce with these parameters needs.
 * buffSize 0 selects the protocol's default (Simple 4 MiB, LL 512 KiB,
 * LL128 4915200 bytes). Layout: a 4 KiB header (status word, abort flag, the
 * configuration it was initialised for, a per-block trace), then a 256-byte
 * head/tail record per connection (with a second head/tail pair for the
 * second part of a two-block launch), then one FIFO of buffSize bytes per
 * connection; a connection is one (channel, ring edge) pair, so there are
 * nranks * popcount(channelMask) of each. Returns 0 for invalid arguments.
 */
RAR_API size_t rar_workspace_bytes(int nranks, uint64_t channelMask, rar_proto proto, size_t buffSize);

/*
 * Prepare a workspace for ring AllReduce calls with this (nranks,
 * channelMask, proto, buffSize): zeroes it (FIFO lines, step counters,
 * status, abort flag) and records the configuration in its header.
 * Enqueued on `stream`. Must be called once before the first rar_allreduce
 * on a workspace, again after switching any of these four parameters, and
 * again after the device reported RAR_ERR_TIMEOUT or RAR_ERR_ABORT.
 * workspace must be 256-byte aligned.
 */
RAR_API rar_status rar_workspace_init(void* workspace, size_t workspaceBytes, int nranks,
                              uint64_t channelMask, rar_proto proto, size_t buffSize,
                              void* stream);

/*
 * Ring AllReduce (sum) over nranks virtual ranks: afterwards every
 * recvbufs[r][i] holds the sum over all ranks q of sendbufs[q][i].
 *
 * Method ([C12] "runRing 的数据切分" .. "源码步骤五", [C23] "Ring AllReduce 到
 * Primitive"): the channels of channelMask split the buffer into contiguous
 * ranges; each channel moves its range in loops of nranks chunks; in each loop
 * the rank at ring index i runs 2*nranks-1 rows -- send, nranks-2 x
 * recvReduceSend, recvReduceCopySend, nranks-2 x recvCopySend, recv -- on
 * chunk (i - s - 1) mod nranks at row s, exchanging data only with its ring
 * neighbours through per-connection FIFOs of RAR_NCCL_STEPS slots under the
 * chosen protocol ([C23] "Simple 的 Credit 与 Step", "LL：Data 与 Flag 同 Line",
 * "LL128：15/16 Payload").
 *
 * Result: the partial sum of chunk c starts with the input of ring index
 * c+1 and each following rank adds its input, the owner (index c) last; for
 * bf16 the partial sums travel as binary32 and are rounded once to bf16 by
 * the owner. The value is fully determined by (inputs, ring_order,
 * channelMask, proto, buffSize, chunkSteps) and is identical on every rank.
 *
 * sendbufs, recvbufs: host arrays of nranks device pointers, 16-byte aligned,
 *   count elements each. recvbufs[r] == sendbufs[r] (in place) is allowed;
 *   any other overlap between buffers is RAR_ERR_ARG.
 * count: elements per rank; 0 enqueues nothing and returns RAR_OK.
 * dtype: RAR_F32 or RAR_BF16. op: RAR_SUM.
 * ring_order: host array of nranks user ranks in ring order (next direction);
 *   must be a permutation of 0..nranks-1, else RAR_ERR_RING.
 * channelMask: non-zero; block n of each rank serves the n-th set bit
 *   ([C23] "Kernel 如何把 Block 映射到 Channel").
 * proto: RAR_SIMPLE, RAR_LL or RAR_LL128.
 * buffSize: FIFO bytes per connection (0 = default); a multiple of 4096.
 *   Must match the workspace.
 * chunkSteps: FIFO steps per Simple chunk: 1, 2 or 4 (8 would fill the whole
 *   credit window with one chunk and deadlock the ring); LL and LL128 use one
 *   step per chunk but still require 1, 2 or 4.
 * workspace: initialised by rar_workspace_init for the same nranks,
 *   channelMask, proto and buffSize; workspaceBytes >= rar_workspace_bytes().
 *   Its step counters carry over from call to call, so FIFO contents never
 *   need clearing between calls.
 * Errors: RAR_ERR_ARG, RAR_ERR_RING, RAR_ERR_ALIGN, RAR_ERR_WORKSPACE,
 *   RAR_ERR_CORESIDENCY, RAR_ERR_CUDA (synchronous); RAR_ERR_TIMEOUT,
 *   RAR_ERR_WORKSPACE, RAR_ERR_ABORT later through rar_get_status().
 */
RAR_API rar_status rar_allreduce(const void* const* sendbufs, void* const* recvbufs, int nranks,
                         size_t count, rar_dtype dtype, rar_redop op, const int* ring_order,
                         uint64_t channelMask, rar_proto proto, size_t buffSize, int chunkSteps,
                         void* workspace, size_t workspaceBytes, void* stream);

/* Flags of rar_allreduce_ex. */
#define RAR_FLAG_DIRECT 1u /* Simple: all-gather hops write the next rank's output directly */

/*
 * rar_allreduce with one ring order per channel and with options.
 *
 * ring_orders: host array of nrings x nranks user ranks; nrings is 1 (every
 *   channel uses the same ring, as in rar_allreduce) or popcount(channelMask)
 *   (dense channel n uses ring n, as NCCL gives each channel its own ring
 *   permutation: [C12] "GRAPH 重建：N=4", "为什么 channels 会重复"). Each ring
 *   must be a permutation of 0..nranks-1, else RAR_ERR_RING; another nrings
 *   is RAR_ERR_ARG. Ring orders may change from call to call on one workspace.
 * flags: 0 or RAR_FLAG_DIRECT (Simple only, else RAR_ERR_ARG). With
 *   RAR_FLAG_DIRECT the all-gather hops use direct writes ([C23] "发布顺序与
 *   Fence": direct read/write skip FIFO slots, barriers and progress stay): a
 *   rank that sends a final value stores it straight into the next rank's
 *   receive buffer and publishes its tail; the receiver waits for the tail and
 *   forwards from its own receive buffer. No FIFO slot is used for those hops,
 *   so the sender takes no credit for them. The result is identical to the
 *   FIFO path. In place stays allowed (a rank's input chunk is always read
 *   before any peer's direct write to it, since each chunk's partial sum passes
 *   through every rank first).
 * Every other argument, and every error, as for rar_allreduce.
 */
RAR_API rar_status rar_allreduce_ex(const void* const* sendbufs, void* const* recvbufs, int nranks,
                                    size_t count, rar_dtype dtype, rar_redop op,
                                    const int* ring_orders, int nrings, uint64_t channelMask,
                                    rar_proto proto, size_t buffSize, int chunkSteps, unsigned flags,
                                    void* workspace, size_t workspaceBytes, void* stream);

/*
 * ReduceScatter (sum) and AllGather on the ring: the two halves of the ring
 * AllReduce ([C12] "Ring AllReduce 不只是“绕一圈”": AllReduce is ReduceScatter
 * followed by AllGather; "源码步骤三": the owner row is the last recv+reduce of
 * the first and the first send of the second) run as collectives of their own,
 * each with nranks rows per chunk loop instead of 2*nranks-1:
 *   ReduceScatter  send, recvReduceSend x (nranks-2), recvReduceCopy
 *   AllGather      copySend, recvCopySend x (nranks-2), recv
 * A block is `count` elements (recvcount, sendcount). The channels split the
 * block range exactly as rar_allreduce splits a rank's buffer; a chunk loop
 * moves one chunk of every block: the chunk with ring index c is that range of
 * the block of the user rank at ring index c on the channel's ring.
 *
 * rar_reduce_scatter: sendbufs[r] holds nranks blocks (nranks*recvcount
 *   elements), block b for user rank b; recvbufs[r] receives block r reduced
 *   over all ranks, in binary32, in ring order starting after r and ending with
 *   r's own input (the AllReduce fold of a chunk owned by r), rounded once for
 *   bf16. Partial sums cross the hops as binary32.
 * rar_all_gather: sendbufs[r] holds one block (sendcount elements);
 *   recvbufs[r] (nranks*sendcount elements) receives block b = sendbufs[b],
 *   bit for bit.
 * Buffers: device pointers, 16-byte aligned; a receive buffer may not overlap
 *   another receive buffer or another rank's send buffer; a rank's own pair
 *   may overlap only in the in-place shape (ReduceScatter: recvbufs[r] ==
 *   sendbufs[r] + r*recvcount elements; AllGather: sendbufs[r] == recvbufs[r] +
 *   r*sendcount elements); anything else is RAR_ERR_ARG. A block of a count
 *   that is not a multiple of 16/sizeof(T) is moved element by element
 *   (correct, slower).
 * proto: RAR_SIMPLE (else RAR_ERR_ARG). flags: 0, or RAR_FLAG_DIRECT for
 *   rar_all_gather only (its hops write the next rank's receive buffer
 *   directly, as in rar_allreduce_ex); RAR_FLAG_DIRECT with rar_reduce_scatter
 *   is RAR_ERR_ARG.
 * ring_orders, nrings, channelMask, buffSize, chunkSteps, workspace, stream
 * and every error as for rar_allreduce_ex; the workspace is the one
 * rar_workspace_init prepares for (nranks, channelMask, proto, buffSize), and
 * its step counters carry over between calls of any of the three collectives.
 */
RAR_API rar_status rar_reduce_scatter(const void* const* sendbufs, void* const* recvbufs, int nranks,
                                      size_t recvcount, rar_dtype dtype, rar_redop op,
                                      const int* ring_orders, int nrings, uint64_t channelMask,
                                      rar_proto proto, size_t buffSize, int chunkSteps, unsigned flags,
                                      void* workspace, size_t workspaceBytes, void* stream);
RAR_API rar_status rar_all_gather(const void* const* sendbufs, void* const* recvbufs, int nranks,
                                  size_t sendcount, rar_dtype dtype, const int* ring_orders, int nrings,
                                  uint64_t channelMask, rar_proto proto, size_t buffSize, int chunkSteps,
                                  unsigned flags, void* workspace, size_t workspaceBytes, void* stream);

/*
 * One-shot AllReduce (sum) over nranks virtual ranks ([OS89], the single
 * kernel form; [NOTES] "5 Symmetric Memory": a rank reads its peers' buffers
 * by pointer): every rank reads all peers' inputs and reduces them itself,
 * in binary32, in user-rank order 0..nranks-1, rounding once for bf16:
 *   recvbufs[r][i] = T(((x_0[i] + x_1[i]) + x_2[i]) + ... + x_{n-1}[i]).
 * sendbufs, recvbufs: host arrays of nranks device pointers, 16-byte aligned,
 *   count elements each; a receive buffer may not overlap any send buffer
 *   (the ranks read each other's inputs while writing their outputs) nor
 *   another receive buffer, else RAR_ERR_ARG.
 * dtype: RAR_BF16 or RAR_F32; op: RAR_SUM; count 0 returns RAR_OK.
 * Needs no workspace and waits on nothing. Errors: RAR_ERR_ARG,
 * RAR_ERR_ALIGN, RAR_ERR_CUDA.
 */
RAR_API rar_status rar_oneshot(const void* const* sendbufs, void* const* recvbufs, int nranks,
                       size_t count, rar_dtype dtype, rar_redop op, void* stream);

/*
 * Staged one-shot AllReduce (sum), the single-kernel form of [OS89] (the
 * "5 kernels -> 3" review and its one-kernel follow-up): per call every rank
 * copies its input into a staging slot of the workspace, the last of the
 * rank's blocks to finish copying (found with a monotonic done counter that
 * every launch advances by exactly its fixed grid) publishes the rank's
 * sequence number, every block waits for all ranks' numbers, then each rank
 * reduces the nranks staged copies:
 *   recvbufs[r][i] = T(((x_0[i] + x_1[i]) + x_2[i]) + ... + x_{n-1}[i])
 * in binary32, in user-rank order, rounded once for bf16 (the same value as
 * rar_oneshot). A slot is reused every 4 calls and only after every rank has
 * acknowledged reading it (the guard). Nothing is reset between calls, so a
 * CUDA graph of calls may be replayed any number of times.
 *
 * rar_oneshot_workspace_bytes: bytes of a workspace for calls of up to
 *   max_count elements of dtype over nranks ranks (0 for invalid arguments):
 *   a 4 KiB header, 640 B of counters per rank, 4 slots per rank.
 * rar_oneshot_workspace_init: zero the header and counters, record the
 *   configuration (nranks, dtype, max_count, and the grid, 4 * SMs / nranks
 *   blocks per rank on the current device); enqueued on `stream`. Errors:
 *   RAR_ERR_ARG, RAR_ERR_WORKSPACE (null or too small), RAR_ERR_ALIGN (not
 *   256-byte aligned), RAR_ERR_CUDA.
 * rar_oneshot_staged: sendbufs/recvbufs as for rar_oneshot, except that in
 *   place (recvbufs[r] == sendbufs[r]) is allowed: every rank reads only the
 *   staged copies. count 0 returns RAR_OK and advances nothing. The workspace
 *   must have been initialised for (nranks, dtype) with max_count >= count on
 *   this device, else the kernel reports RAR_ERR_WORKSPACE through
 *   rar_get_status(); a wait that runs out of time (rar_set_spin_timeout_ns)
 *   reports RAR_ERR_TIMEOUT and leaves the workspace aborted (re-initialise).
 *   The launch is cooperative: RAR_ERR_CORESIDENCY if it cannot be resident.
 */
RAR_API size_t rar_oneshot_workspace_bytes(int nranks, size_t max_count, rar_dtype dtype);
RAR_API rar_status rar_oneshot_workspace_init(void* workspace, size_t workspaceBytes, int nranks,
                                              size_t max_count, rar_dtype dtype, void* stream);
RAR_API rar_status rar_oneshot_staged(const void* const* sendbufs, void* const* recvbufs, int nranks,
                                      size_t count, rar_dtype dtype, rar_redop op, void* workspace,
                                      size_t workspaceBytes, void* stream);

/*
 * Bytes of the device array behind rar_allreduce_static(). Every GPU that
 * loads this library holds one such array until the process exits.
 */
#define RAR_STATIC_WORKSPACE_BYTES (16u << 20)

/*
 * rar_allreduce() for callers that cannot allocate device memory -- for
 * example a plug-in whose host application owns all device memory through
 * its own allocator, or code on a latency-critical path that may not call
 * cudaMalloc or cudaFree because those calls can synchronise the whole
 * device. This entry point allocates nothing: its workspace is a library
 * array of RAR_STATIC_WORKSPACE_BYTES in device memory (see above). The pages
 * have no counterpart to it. The caller still passes the send and receive
 * buffers; every other argument means what it means for rar_allreduce().
 *
 * - Arguments are checked first, with the codes of rar_allreduce() and in
 *   its order; then a call whose workspace (rar_workspace_bytes(nranks,
 *   channelMask, proto, buffSize)) would exceed RAR_STATIC_WORKSPACE_BYTES
 *   is refused with RAR_ERR_WORKSPACE. A refused call makes no CUDA call and
 *   enqueues nothing; so does an empty call (count 0, RAR_OK).
 * - The first call on a device looks up the array's device address on that
 *   device (it must be the current device). Make that first call before any
 *   stream capture begins.
 * - All calls share the one array, which keeps the last call's contents.
 *   Each call first clears, on `stream`, what it needs cleared: the header,
 *   status and step counters, and for LL and LL128 also the FIFO lines of
 *   the bytes it uses (Simple writes each FIFO byte before reading it). No
 *   state carries over between calls.
 * - Calls that overlap on the GPU -- on different streams, or from threads
 *   whose calls are not ordered on one stream -- race on the array and give
 *   wrong results. Order them on one stream.
 * - A device failure of a call (a wait that ran out of time) cannot be read
 *   back: the status word lives in the array, whose address this entry point
 *   does not expose, and the next call clears it. Callers that need the
 *   status use rar_allreduce() with a workspace of their own.
 */
RAR_API rar_status rar_allreduce_static(const void* const* sendbufs, void* const* recvbufs,
                                        int nranks, size_t count, rar_dtype dtype, rar_redop op,
                                        const int* ring_order, uint64_t channelMask,
                                        rar_proto proto, size_t buffSize, int chunkSteps,
                                        void* stream);

/*
 * Wait for `stream`, then return the device status word of `workspace`
 * (RAR_OK if no kernel reported a failure) and clear it. After
 * RAR_ERR_TIMEOUT the workspace stays aborted (later calls report
 * RAR_ERR_ABORT) until rar_workspace_init.
 */
RAR_API rar_status rar_get_status(void* workspace, void* stream);

/* Static text for a status code. */
RAR_API const char* rar_strerror(rar_status status);

/*
 * Time limit, in nanoseconds, of every wait inside the kernels (a wait for
 * data, for a credit, or for another role of the same block). When it runs
 * out the block records RAR_ERR_TIMEOUT, raises the workspace's abort flag,
 * and every block leaves its loops, so the launch always completes. Applies
 * to launches enqueued after the call. Default 2 s; 0 restores the default.
 */
RAR_API void rar_set_spin_timeout_ns(uint64_t ns);

/*
 * Test hook for failure detection: fault 0 = none (default); 1 = every
 * receiver skips publishing its head, so each sender runs out of credit
 * after RAR_NCCL_STEPS steps and waits until the time limit; 2 = in
 * rar_oneshot_staged, no rank acknowledges its reads, so the fifth call's
 * guard (4 slots per rank) waits until the time limit. No GPU fault
 * happens: the waits end, every block leaves, the launch completes, and
 * rar_get_status() reports RAR_ERR_TIMEOUT. 3 = in the debug library
 * (librar_debug.so) only, the device-side bounds check of the ring kernels
 * sees every slice one buffer further on than it is (the slice's own
 * accesses keep their offsets), so the first slice is refused and
 * rar_get_status() reports RAR_ERR_BOUNDS; the release library ignores 3.
 * Applies to launches enqueued after the call.
 */
RAR_API void rar_debug_set_fault(int fault);

/*
 * Test mode of the LL flags ([C23] "LL：Data 与 Flag 同 Line": a test macro
 * makes the flag wrap at 0x100, and a cleanup keeps the wrap correct).
 * flag_max 0 (default): the production flag, step + 1 as 32 bits. A power of
 * two in [64, 2^31]: LL flags are (step + 1) mod flag_max, and on the last
 * RAR_NCCL_STEPS steps of every flag_max / 2 steps a sender also rewrites
 * every line of its FIFO slot past its slice with the current flag, so no
 * line is ever older than half a period when it is read and none can carry
 * the flag of a later step. Results are unchanged. Applies to LL launches
 * enqueued after the call; a workspace used under one mode must be
 * re-initialised (rar_workspace_init) before calls under the other. Returns
 * RAR_ERR_ARG (and changes nothing) for any other flag_max.
 */
RAR_API rar_status rar_debug_set_ll_flag_wrap(uint32_t flag_max);

/*
 * The geometry a ring AllReduce call would use, computed on the host with
 * no device work (the "TRACE" view of [C23] "Kernel 如何把 Block 映射到
 * Channel" and [C12] "runRing 的数据切分"). out receives, in order:
 *   out[0] step bytes, out[1] full-chunk elements, out[2] steps per slice,
 *   out[3] slices per chunk, out[4] C = popcount(channelMask), out[5]
 *   elements per channel, then C channel ids (dense order), then for each
 *   dense channel its (gridOffset, channelCount), then for each dense
 *   channel its number of loops.
 * out must hold 6 + 4*C entries. Returns the status of argument checks.
 */
RAR_API rar_status rar_describe_geometry(int nranks, size_t count, rar_dtype dtype, uint64_t channelMask,
                                 rar_proto proto, size_t buffSize, int chunkSteps, int64_t* out);

#ifdef __cplusplus
}
#endif

#endif /* RAR_H */
