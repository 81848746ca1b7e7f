/*
 * rr.h -- C ABI of the reduce/gather data movement inside a custom collective,
 * for one GB300 (sm_103a) GPU.
 *
 * W "ranks" are emulated on one GPU: each rank's registered buffer is a plain
 * device pointer into this GPU's own HBM, standing in for the peer (IPC /
 * symmetric-memory) buffers a real multi-GPU collective would address.  One
 * call launches one kernel that runs all W ranks' per-GPU work as W groups of
 * blocks; the groups order themselves through a signal pad of generation
 * flags in the same HBM.  No NCCL, no peer access and no host synchronisation
 * happen on any call below except rr_signal_pad_create/_destroy/_status.
 *
 * Conventions for every entry point:
 *  - Pointer arrays (inputs, rank_bufs, outputs) are HOST arrays of W device
 *    pointers.  They are read during the call only (copied by value into the
 *    kernel's parameters), so the caller may reuse them as soon as the call
 *    returns.  The pointed-to device buffers are owned by the caller and must
 *    stay valid until the work completes on `stream`.
 *  - Every device pointer must be 16-byte aligned (RR_ERR_ALIGNMENT).  It may
 *    point anywhere inside a larger allocation.  Any element count is
 *    accepted, not only multiples of the 16-byte vector.
 *  - Buffers are dense: rank r's data is `numel` consecutive elements.
 *  - Outputs must not overlap any input, rank buffer or other output
 *    (RR_ERR_ALIAS); rank buffers must not overlap each other.
 *  - Argument errors are returned synchronously, before anything is
 *    enqueued.  A barrier that times out on the device is recorded in the
 *    pad (sticky) and read back with rr_signal_pad_status.
 *  - Calls are asynchronous with respect to the host and ordered on
 *    `stream` (a cudaStream_t; 0 is the legacy default stream).  A pad may be
 *    used by one stream at a time: concurrent collectives need separate
 *    pads, because a pad's flag slots and generation counter are shared
 *    state (the lesson of the shared per-slot flag in "ccl: hierarchical
 *    cross-node AllGather (intra-node SDMA + inter-node RDMA) #441", the
 *    commit on concurrent param-contiguous scatters).  Each call is one
 *    cooperative kernel launch that is also programmatic: it may be launched
 *    while the work before it on `stream` drains, and waits on the device
 *    for that work to complete before touching memory, so stream order is
 *    kept; the kernel lets the next launch on `stream` start early, which a
 *    following launch uses only if it is programmatic too.
 *  - Reductions accumulate in binary32 in rank order 0, 1, ..., W-1, starting
 *    from rank 0's value, and round once to the element type (round to
 *    nearest, ties to even; no flush of subnormals).  int32 sums wrap modulo
 *    2^32.  Gathers copy raw bits.
 */
#ifndef RR_H
#define RR_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RR_MAX_WORLD 16   /* largest W */
#define RR_MAX_SPLITS 256 /* largest number of params in one param-contiguous call */

typedef enum { RR_BF16 = 0, RR_FP16 = 1, RR_FP32 = 2, RR_INT32 = 3 } rr_dtype;

typedef enum {
    RR_OK = 0,
    RR_ERR_INVALID_ARG = 1,       /* null pointer, W out of range, negative size, ... */
    RR_ERR_UNSUPPORTED_DTYPE = 2,
    RR_ERR_ALIGNMENT = 3,         /* a device pointer is not 16-byte aligned */
    RR_ERR_ALIAS = 4,             /* buffers overlap where they must not */
    RR_ERR_TOO_MANY_BLOCKS = 5,   /* the pad was created for fewer blocks per rank */
    RR_ERR_CUDA = 6,              /* a CUDA runtime call failed; see rr_last_error */
    RR_ERR_TIMEOUT = 7,           /* a device-side barrier wait ran out of time */
    RR_ERR_WRONG_DEVICE = 8       /* the current device is not the pad's device */
} rr_status;

/* Barriers inside one call, used to name a barrier in fault injection and in
 * the diagnostic of a timeout. */
typedef enum {
    RR_BARRIER_ARRIVE = 0, /* start, no staging: block 0 of every rank announces arrival */
    RR_BARRIER_STAGE = 1,  /* start, copy_mode: block b of every rank has staged its chunk */
    RR_BARRIER_MID = 2,    /* two-shot: block b of every rank has reduced its owned chunk */
    RR_BARRIER_END = 3     /* end: block b of every rank is done with every peer buffer */
} rr_barrier;

/* Options of a pad (rr_signal_pad_set_option / rr_signal_pad_get_option). */
typedef enum {
    RR_OPT_TIMEOUT_NS = 0,      /* barrier wait limit in ns (default 2e9) */
    RR_OPT_BLOCKS_PER_RANK = 1, /* 0 = automatic (default); else a fixed block count per rank */
    RR_OPT_GATHER_ENGINE = 2,   /* 0 = automatic (TMA bulk copies when a call moves at least
                                   256 MiB, shards read plus outputs written, or 8 MiB with two
                                   or more kept outputs, and every split
                                   boundary is a multiple of 16 bytes; 128-bit loads/stores
                                   otherwise), 1 = 128-bit loads/stores,
                                   2 = TMA bulk copies, 3 = the GPU's copy engines: one
                                   cudaMemcpyAsync per (output, rank, param) slot and no
                                   kernel, so no SM is taken from concurrent compute
                                   ("ccl: hierarchical cross-node AllGather (intra-node SDMA
                                   + inter-node RDMA) #441", PR description: the intra-node
                                   gather on copy engines overlaps a concurrent GEMM).  The
                                   copies are ordered by the stream alone: they pass no
                                   barrier and ignore a pending timeout on the pad */
    RR_OPT_INJECT_SKIP = 3,     /* fault injection: -1 = off; else rank*4 + barrier: that rank
                                   never emits that barrier's flags, so peers time out */
    RR_OPT_ROUND_BYTES = 4,     /* bytes per rank per round of a pipelined chunk; 0 = automatic.
                                   Bulk-copy copy_mode kernels: the piece of each range staged
                                   and published as one unit (automatic: at most 16 KiB, cut
                                   so that every block of a rank gets the same number of
                                   pieces where granules allow).  Load/store
                                   kernels: the round of a block's chunk (automatic 64 KiB
                                   one-shot, 8 KiB per range two-shot).  Grown where a block
                                   would pass 65535 rounds */
    RR_OPT_REDUCE_ENGINE = 5,   /* 0 = automatic (copy_mode: bulk-copy staging for the one-shot
                                   when W >= 4, W x bytes per rank >= 64 MiB and one or at most
                                   W/4 outputs are kept, for the push two-shot when W = 2 or
                                   from 8 MiB per rank; copy_mode off: bulk-copy loads for the
                                   one-shot when W > 8 and W x bytes per rank >= 128 MiB, 512 MiB
                                   with more than half the outputs kept; loads/stores otherwise),
                                   1 = 128-bit loads/stores, 2 = bulk-copy (TMA)
                                   engine: copy_mode off, the one-shot's loads stream into a
                                   shared-memory ring; copy_mode on, a producer warp stages the
                                   inputs by bulk copies while the other warps reduce (the
                                   two-shot then uses the push allgather) */
    RR_OPT_TWOSHOT_MODE = 6,    /* two-shot allgather phase: 0 = automatic (push), 1 = pull (every rank
                                   copies the other owners' reduced chunks after the MID
                                   barrier), 2 = push (each owner stores its reduced chunk into
                                   every output; no MID barrier) */
    RR_OPT_DEVICE_GENERATION = 7, /* 0 = each call takes its generation from a host counter
                                   (default); 1 = from a counter in device memory that the
                                   last block of each call advances, so that calls captured
                                   in a CUDA graph stay correct on every replay.  Switching
                                   synchronises the device; the pad must be idle */
    RR_OPT_DEBUG_ITERATIONS = 8, /* test mode, default 1: each call runs n complete calls inside
                                   one launch, iteration k with generation g + k, so the barriers
                                   that separate one call from the next are crossed without a
                                   kernel boundary (as on several GPUs, where there is none).
                                   Iteration k uses the inputs, outputs and (copy_mode off) rank
                                   buffers advanced by k * S bytes, S = the per-call size of that
                                   pointer rounded up to 16 bytes (allgather outputs: W * shard
                                   bytes rounded up); with copy_mode on every iteration stages
                                   into the same rank buffers, so a rank that restaged before a
                                   peer finished reading would corrupt that peer's result.
                                   Every buffer must hold all n slices.  bf16 reductions on the
                                   automatic engines (push two-shot) and the gather kernels
                                   (not the copy engines); needs device generation off */
    RR_OPT_DEBUG_SKEW_NS = 9,   /* test mode, default 0 (max 1e6): before iteration k every block
                                   of rank r sleeps ((r + k) mod W) * skew ns, so the ranks reach
                                   every barrier out of step.  Non-zero selects the test-mode
                                   kernels even with one iteration */
    /* read-only */
    RR_OPT_GENERATION = 16,     /* generation flag value of the last call (device-generation
                                   mode: reads the device counter, synchronising the device) */
    RR_OPT_LAST_GRID = 17,      /* blocks launched by the last call */
    RR_OPT_LAST_BLOCKS_PER_RANK = 18,
    RR_OPT_LAST_ENGINE = 19,    /* engine the last call used (1 = loads/stores, 2 = bulk copies,
                                   3 = copy engines) */
    RR_OPT_WORLD_SIZE = 20,
    RR_OPT_MAX_BLOCKS_PER_RANK = 21
} rr_option;

typedef struct rr_signal_pad rr_signal_pad; /* opaque, owned by the library */

/*
 * rr_signal_pad_create -- allocate the signal pad of one communicator.
 *
 * The pad is the array of 32-bit generation flags that the ranks' blocks
 * exchange, as the `uint32_t** signals` of multi_gpu_barrier / block_barrier
 * in "Question and suggestions about custom allreduce" (sglang discussion
 * 2918), leizhao1234's first post: dimension 0 listens, the last dimension
 * emits.  Layout here: [W listener][4 barriers][2 parities][blocks][W emitter]
 * uint32 words on the current device, then [W listener][2][blocks][W emitter]
 * uint64 round flags, then a status block.  Each call takes the next
 * generation value g (a host counter, never 0) and writes g into slots of
 * parity g & 1, so consecutive calls never share a slot (the same post picks
 * the half of the arrival flags to use from the flag's parity).  Barriers
 * passed once per round of a pipelined chunk (copy_mode staging, the two-shot
 * middle) use the 64-bit round flags instead: values that only grow, from a
 * 64-bit call counter, waited on as "at least".
 *
 * world_size: W, 1..RR_MAX_WORLD.  max_blocks_per_rank: upper bound on
 * blocks per rank any call on this pad may use (0 = 1024).  timeout_ns:
 * barrier wait limit (0 = 2 s).  Allocates and zeroes device memory and
 * synchronises the device once.  *out receives the pad.
 */
rr_status rr_signal_pad_create(int world_size, int max_blocks_per_rank, uint64_t timeout_ns,
                               rr_signal_pad **out);

/*
 * Free the pad's device memory (synchronises the device first).  NULL is a
 * no-op.  No passage on the pages covers the pad's lifecycle: the sglang
 * discussion's signal arrays are set up once per communicator and live as
 * long as it does, which is what create / destroy bracket here.
 */
rr_status rr_signal_pad_destroy(rr_signal_pad *pad);

/*
 * Synchronise `stream`, then return the pad's sticky device status: RR_OK, or
 * RR_ERR_TIMEOUT if any barrier wait of an earlier call ran out of time.
 * Reading the status clears it.  While a timeout is pending, every later call
 * on the pad exits at its first barrier without writing outputs.
 * rr_signal_pad_timeout_info gives where the first timeout happened.
 * No passage on the pages covers it: their barrier loops spin without a
 * bound ("Question and suggestions about custom allreduce", sglang discussion
 * 2918, multi_gpu_barrier / block_barrier), and this library bounds every
 * wait and reports the failure here instead of hanging the GPU.
 */
rr_status rr_signal_pad_status(rr_signal_pad *pad, cudaStream_t stream);

/* Where the last cleared timeout happened: barrier, waiting rank, block, and
 * the generation of the call.  Valid after rr_signal_pad_status returned
 * RR_ERR_TIMEOUT. */
rr_status rr_signal_pad_timeout_info(rr_signal_pad *pad, int *barrier, int *rank, int *block,
                                     uint32_t *generation);

rr_status rr_signal_pad_set_option(rr_signal_pad *pad, rr_option opt, int64_t value);
rr_status rr_signal_pad_get_option(rr_signal_pad *pad, rr_option opt, int64_t *value);

/*
 * rr_allreduce_oneshot -- every rank reads all W rank buffers and writes the
 * element-wise sum to its own output.
 *
 * Source: "Question and suggestions about custom allreduce" (sglang discussion
 * 2918), the trt_reduce_internal.cu block comment quoted in yizhang2077's
 * reply: each block (1) copies its chunk from local_input to the shareable
 * buffer when copy_mode is on, (2) waits for the same block on every other
 * GPU, (3) pulls the chunk from every GPU, sums it and writes local_output;
 * with copy_mode off step 1 is skipped and only the arrival of every GPU is
 * awaited.
 *
 * inputs:    W device pointers, rank r's local input (numel elements).  Read
 *            only when copy_mode != 0 (may be NULL otherwise).
 * rank_bufs: W device pointers, rank r's registered buffer (numel elements).
 *            copy_mode != 0: the kernel stages inputs[r] into rank_bufs[r]
 *            (overwritten).  copy_mode == 0: rank_bufs[r] already holds rank
 *            r's data and is only read.
 * outputs:   W device pointers, rank r's output (numel elements).  An entry
 *            may be NULL: that rank's output is not materialised (its blocks
 *            still stage, signal, and lend their bandwidth to the
 *            materialised outputs of the same chunk).  At least one non-NULL.
 * numel:     elements per rank (>= 0; 0 returns RR_OK without a launch).
 * dtype:     RR_BF16, RR_FP16, RR_FP32 (binary32 accumulate) or RR_INT32.
 * Barriers: ARRIVE (copy_mode off) or STAGE (copy_mode on) before the
 * reduction, END after it, so that when the call completes on `stream` no rank
 * still reads any peer buffer.
 */
rr_status rr_allreduce_oneshot(const void *const *inputs, void *const *rank_bufs,
                               void *const *outputs, int world_size, int64_t numel,
                               rr_dtype dtype, int copy_mode, rr_signal_pad *pad,
                               cudaStream_t stream);

/*
 * rr_allreduce_twoshot -- reduce-scatter then allgather: rank r owns segment
 * S_r of the message, reduces it from all W rank buffers into outputs[r][S_r],
 * and after a barrier copies every other owner's reduced segment
 * outputs[c][S_c] into outputs[r][S_c].
 *
 * Source: "Question and suggestions about custom allreduce" (sglang discussion
 * 2918), leizhao1234's opening post (two-shot needs an arrival barrier and a
 * block barrier between its two phases), and the owned-slice partition of
 * multimem_all_reduce_kernel in "triton_multimem_all_reduce.py"
 * (symm-mem-recipes): rank r covers 128-bit units [r*C, (r+1)*C) with
 * C = ceil(units / W).  Here the owned segments are C 16-byte vectors (rounded
 * up to whole 256-byte granules), the last segment short or empty, and the
 * elements after the last whole vector are owned by rank W-1.
 *
 * Arguments as rr_allreduce_oneshot, except that every outputs[r] is required.
 * Two allgather modes (RR_OPT_TWOSHOT_MODE): push (default), where each owner
 * stores its reduced chunk into every output, as the owner-side multicast
 * store of the Triton kernel does; pull, where each rank copies the other
 * owners' reduced chunks out of their outputs after the MID barrier.
 * Barriers: ARRIVE or STAGE, MID (pull only), END.  Results are bit-identical
 * to the one-shot.
 *
 * In place: with copy_mode off, outputs[r] may equal rank_bufs[r] (exactly,
 * for any subset of r); the sum then replaces the rank buffers, as the Triton
 * kernel's in-place allreduce does.  (Every chunk is read from all buffers
 * and written by the same block; in pull mode the MID barrier orders every
 * owner's reads before the overwrite.)  The one-shot never runs in place: a
 * peer may still be reading the buffer being overwritten.
 */
rr_status rr_allreduce_twoshot(const void *const *inputs, void *const *rank_bufs,
                               void *const *outputs, int world_size, int64_t numel,
                               rr_dtype dtype, int copy_mode, rr_signal_pad *pad,
                               cudaStream_t stream);

/*
 * rr_allgather -- all_gather_into_tensor, rank-major: every materialised
 * output q receives rank r's buffer at element offset r * numel_per_rank.
 *
 * Source: "ccl: hierarchical cross-node AllGather (intra-node SDMA +
 * inter-node RDMA) #441", the PR description (an all_gather_into_tensor-
 * compatible collective, bit-exact for bf16/fp16/fp32/int32).  Each rank
 * pushes its own shard into every materialised output, as that PR's gather
 * pushes straight into the destination.
 *
 * rank_bufs: W device pointers, rank r's shard (numel_per_rank elements).
 * outputs:   W device pointers to W*numel_per_rank elements each, or NULL
 *            (not materialised); at least one non-NULL.
 * Raw bits are copied (any dtype; NaN payloads survive).  Barriers: ARRIVE,
 * END (every push into an output has landed before its rank completes).
 */
rr_status rr_allgather(const void *const *rank_bufs, void *const *outputs, int world_size,
                       int64_t numel_per_rank, rr_dtype dtype, rr_signal_pad *pad,
                       cudaStream_t stream);

/*
 * rr_allgather_param_contiguous -- FSDP-style allgather into a [param][rank]
 * output: rank r's shard is the concatenation of its pieces of params
 * 0..S-1 (piece s has E_s = split_sizes[s] elements and starts at
 * O_s = E_0 + ... + E_{s-1}); the piece lands at element O_s*W + r*E_s of
 * every materialised output.
 *
 * Source: "ccl: hierarchical cross-node AllGather (intra-node SDMA +
 * inter-node RDMA) #441", the commit adding enqueue_param_contiguous (rank r
 * lands at O_s*W + r*E_s, from "dtype-elem splits"), and the following commit
 * that loops all blocks and splits inside one launch instead of one launch
 * per (node block, param).  One call here is one launch over every
 * (rank, param) slot.  The node grouping G of that PR does not change where
 * anything lands, so it is not an argument.
 *
 * split_sizes: HOST array of num_splits (0..RR_MAX_SPLITS) element counts,
 *              each >= 0.  rank_bufs[r] holds sum(E_s) elements.
 * outputs:     W device pointers to W*sum(E_s) elements each, or NULL.
 * Raw bits are copied.  Barriers: ARRIVE, END.
 */
rr_status rr_allgather_param_contiguous(const void *const *rank_bufs, void *const *outputs,
                                        int world_size, const int64_t *split_sizes,
                                        int num_splits, rr_dtype dtype, rr_signal_pad *pad,
                                        cudaStream_t stream);

/*
 * rr_allgather_list -- torch.distributed.all_gather with list output: output
 * q is a list of W separate buffers, and buffer r of every materialised list
 * receives rank r's shard.
 *
 * Source: "ccl: hierarchical cross-node AllGather (intra-node SDMA +
 * inter-node RDMA) #441", the commit adding HierAllGather.all_gather
 * (tensor_list, tensor) on the same path as all_gather_into_tensor, bit-exact
 * against torch for bf16/fp16/fp32/int32.  The same kernels as rr_allgather
 * run it (one launch); only each slot's destination differs.
 *
 * rank_bufs:    W device pointers, rank r's shard (numel_per_rank elements).
 * output_lists: HOST array of W*W device pointers; entry q*W + r is buffer r
 *               of rank q's list (numel_per_rank elements).  Row q is either
 *               all non-NULL (materialised) or all NULL; at least one row is
 *               materialised.  No buffer may overlap another or a rank buffer.
 * Raw bits are copied.  Barriers: ARRIVE, END (none with the copy engines).
 */
rr_status rr_allgather_list(const void *const *rank_bufs, void *const *output_lists, int world_size,
                            int64_t numel_per_rank, rr_dtype dtype, rr_signal_pad *pad,
                            cudaStream_t stream);

/*
 * rr_allreduce_oneshot_noalloc -- rr_allreduce_oneshot for callers that may
 * not allocate device memory.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * such as engine plugins whose enqueue runs inside a memory budget fixed
 * ahead of time, frameworks that hand every byte of device memory to their
 * own pool, and code on a latency-critical path where cudaMalloc's implicit
 * device synchronisation would stall the GPU.  Those callers cannot create a
 * signal pad (rr_signal_pad_create calls cudaMalloc).  This call uses instead
 * a fixed signal pad that the library holds in a static device array of
 * 96 KiB + 32 bytes, present on every GPU that loads the library until the
 * process exits.  It calls no cudaMalloc, cudaFree or allocating routine.
 *
 * Arguments, results and errors are those of rr_allreduce_oneshot without
 * the pad.  Limits: world_size 1..8 (larger W returns RR_ERR_INVALID_ARG
 * with a message naming the limit) and at most 32 blocks per rank (chosen
 * automatically).  The first call on a device looks up the array's device
 * address with that device current; make that first call before any stream
 * capture.  A call made while `stream` is being captured into a CUDA graph
 * returns RR_ERR_INVALID_ARG: each call takes a new flag generation from a
 * host counter, and a replayed launch would repeat it.  After a
 * cudaDeviceReset of a device, calls on it are not supported (the address
 * looked up by the first call is void).  Every call on a device shares the
 * one array: calls that overlap on the GPU (different streams, or other
 * threads) race on it, so serialise them.  Each call clears the array's
 * status words on `stream` before its kernel.  A barrier that times out (only
 * if the GPU cannot keep all ranks' blocks running at once for 2 s) stops the
 * kernel early with incomplete outputs and is recorded in those words: read
 * it with rr_allreduce_oneshot_noalloc_status.
 */
rr_status rr_allreduce_oneshot_noalloc(const void *const *inputs, void *const *rank_bufs,
                                       void *const *outputs, int world_size, int64_t numel,
                                       rr_dtype dtype, int copy_mode, cudaStream_t stream);

/*
 * rr_allreduce_oneshot_noalloc_status -- the device status of the allocation-
 * free one-shot on the current device, read without allocating.
 *
 * The pages have no counterpart (it belongs to rr_allreduce_oneshot_noalloc).
 * Synchronises `stream`, copies the status words of the static array into a
 * local host array and returns RR_OK, or RR_ERR_TIMEOUT (rr_last_error says
 * which barrier, rank, block and generation) if a barrier wait of the last
 * call enqueued before the read ran out of time; reading clears it.  Returns
 * RR_OK when no call has been made on the device.  Calls no cudaMalloc,
 * cudaFree or allocating routine.
 */
rr_status rr_allreduce_oneshot_noalloc_status(cudaStream_t stream);

/* Name of a status code (static string). */
const char *rr_status_string(rr_status s);

/* Human-readable detail of the last error returned on this host thread
 * (static thread-local buffer; empty after a successful call). */
const char *rr_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* RR_H */
