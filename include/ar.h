/*
 * ar.h -- C ABI of libar.so: an all-reduce over P ranks emulated as P separate
 * buffers in one GPU's memory.
 *
 * The operation ("NCCL, NIXL, and Distributed GPU Communication", section
 * "All-reduce"): every rank's buffer is reduced elementwise with sum, min or
 * max, and the single result is stored in every rank's receive buffer; DDP
 * then divides it by world_size (the fused `scale` below).  The call mirrors
 * the pages' host-side NCCL pattern ("NCCL and NVSHMEM -- two GPU communication
 * models, side by side", host-code example: ncclCommInitRank once, then
 * ncclAllReduce(sendbuff, recvbuff, count, datatype, op, comm, stream), then
 * cudaStreamSynchronize).  Because one process holds all P emulated ranks, the
 * rank id disappears and send / receive buffers become arrays of P pointers.
 *
 * Combination order (which partial sums are formed) is part of the result for
 * floating-point data:
 *   AR_ALGO_RING -- reduce-scatter of P chunks followed by all-gather ("NCCL,
 *     NIXL, ...", section "Reduce-scatter": all-reduce = reduce-scatter +
 *     all-gather; lecture_068 page, section 05: the ring takes 2(N-1) steps).
 *     The count is cut into P chunks of L = roundup(ceil(count/P), V) elements,
 *     V = 16 / sizeof(element); element e of chunk c is folded as
 *     x_c, then (+) x_{c+1}, ..., (+) x_{c+P-1} (ranks mod P).
 *   AR_ALGO_TREE -- the double binary tree ("NCCL and NVSHMEM ...", section
 *     "double binary tree": two complementary binary trees at once).  Labels
 *     1..P form an in-order binary tree rooted at the largest power of two <= P
 *     (label v with lowbit b >= 2 has children v - b/2 and v + h, h the largest
 *     of b/2, b/4, ..., 1 with v + h <= P).  Tree 0 puts rank r at label r+1,
 *     tree 1 puts it one label earlier (label v -> rank v mod P).  A node's
 *     value is ((own (+) left) (+) right).  Elements [0, H) follow tree 0 and
 *     [H, count) tree 1, H = min(count, roundup(ceil(count/2), V)).
 *   AR_ALGO_LL -- the small-message protocol of "Demystifying NVSHMEM" (the
 *     collectives paragraph: LL packs data and its arrival flag into one
 *     atomic write): each rank's 4-byte payload words are staged as 8-byte
 *     {payload, flag = per-call epoch} words, reducers poll the flags (bounded
 *     spin) and fold in the RING order, so LL == RING bit for bit.
 *   AR_ALGO_LL128 -- LL's medium-message sibling (same paragraph of
 *     "Demystifying NVSHMEM"): each rank's bytes are staged in 128-byte lines
 *     of 120 payload bytes and one flag word (the epoch).  A 128-byte store is
 *     not guaranteed to be seen whole by the PTX memory model, so a line is
 *     published with a release store of its flag after the payload, and read
 *     after an acquire of the flag.  Ring order: LL128 == RING bit for bit.
 *     Up to the LL128 limit (1 MiB per rank by default, AR_LL128_MAX_BYTES).
 *   AR_ALGO_HIER -- the hierarchical all-reduce (lecture_068 page, section 06:
 *     reduce-scatter inside each node, ring all-reduce between nodes,
 *     all-gather inside each node) for P = G groups of Q consecutive ranks
 *     (Q set by AR_OPT_HIER_GROUP, default 8).  Element e of intra-group
 *     chunk c1 (Q chunks of L1 = roundup(ceil(count/Q), V)) is folded inside
 *     each group g from local rank c1: part_g = x_{g,c1} (+) ... (+)
 *     x_{g,c1+Q-1}; the G partials of chunk c1 (len1 elements, cut into G
 *     sub-chunks of roundup(ceil(len1/G), V)) are then folded from group c2,
 *     e's sub-chunk: part_{c2} (+) ... (+) part_{c2+G-1}.  G = 1 or Q = 1 is
 *     the plain ring.  Never chosen by AUTO.
 *   AR_ALGO_AUTO -- LL when count * sizeof(element) <= the LL limit (64 KiB by
 *     default), RING above it (NCCL picks tree for small and ring for large
 *     messages by itself: "NCCL and NVSHMEM ...", the ring / tree paragraph);
 *     after ar_tune, the measured fastest algorithm for the size instead.
 * Accumulation: fp32 for fp32 and bf16 data (bf16 rounded once, to nearest
 * even, at the end), two's-complement wrap-around for int32.  Min / max keep
 * the earlier operand of a tie in fold order.
 *
 * Threading: a communicator is not thread-safe, and only one ar_allreduce may
 * be in flight on it at a time (calls on one stream are ordered, so that is
 * the normal case); two concurrent collectives need two communicators
 * ("Demystifying NVSHMEM": two concurrent collectives on one PE may not share
 * a team's internal resources).
 */
#ifndef AR_H_
#define AR_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque communicator.  Created once and reused across calls: creating one is
 * expensive, so it belongs outside the training loop ("NCCL, NIXL, and
 * Distributed GPU Communication", the checklist item on communicator
 * creation). */
typedef struct ar_comm* ar_comm_t;

typedef enum {
    AR_SUCCESS = 0,
    AR_ERR_INVALID_ARG = 1,  /* bad pointer, alignment, overlap, size or enum value     */
    AR_ERR_CUDA = 2,         /* a CUDA runtime call failed (no device, launch failure)   */
    AR_ERR_UNSUPPORTED = 3,  /* valid but not provided: scale != 1 for int32 / min / max,
                                LL above the LL limit                                    */
    AR_ERR_TIMEOUT = 4,      /* device side: a flag or mbarrier wait hit its limit      */
    AR_ERR_OOM = 5           /* ar_init could not allocate its device memory            */
} ar_status_t;

typedef enum { AR_FLOAT32 = 0, AR_BFLOAT16 = 1, AR_INT32 = 2 } ar_dtype_t;
typedef enum { AR_SUM = 0, AR_MIN = 1, AR_MAX = 2 } ar_op_t;
typedef enum {
    AR_ALGO_AUTO = 0,
    AR_ALGO_RING = 1,
    AR_ALGO_TREE = 2,
    AR_ALGO_LL = 3,
    AR_ALGO_HIER = 4,
    AR_ALGO_LL128 = 5
} ar_algo_t;

/* Largest number of emulated ranks one communicator takes. */
#define AR_MAX_RANKS 256

/* Size buckets measured by ar_tune: per-rank sizes 8 B, 16 B, ..., 16 MiB. */
#define AR_TUNE_BUCKETS 22

/*
 * Creates a communicator for `nranks` emulated ranks (1 .. AR_MAX_RANKS) on
 * the calling thread's current CUDA device and stores it in *out.  Allocates
 * the LL staging area (nranks * LL limit * 2 bytes: 8-byte words carrying
 * 4-byte payloads), the LL128 staging area (nranks * LL128 limit * 128/120
 * bytes), a device status word and the tree schedules; reads the
 * environment defaults AR_DEBUG, AR_LL_MAX_BYTES, AR_LL128_MAX_BYTES and
 * AR_LL_SPIN_LIMIT.
 * Synchronous.  Errors: AR_ERR_INVALID_ARG (out == NULL or nranks out of
 * range), AR_ERR_CUDA (no usable device), AR_ERR_OOM.  On error *out is NULL.
 */
ar_status_t ar_init(int nranks, ar_comm_t* out);

/*
 * All-reduce of P = nranks buffers (definition and orders above).
 *   sendbufs  host array of P device pointers; sendbufs[r] holds rank r's
 *             `count` elements.  Read only.
 *   recvbufs  host array of P device pointers; recvbufs[r] receives the
 *             `count`-element result.  recvbufs[r] == sendbufs[r] (in place)
 *             is allowed; so is any exact aliasing of two buffers.  Buffers
 *             that overlap without starting at the same address are rejected.
 *   count     elements per rank; 0 is a no-op returning AR_SUCCESS.
 *   scale     multiplies the reduced value once, in fp32, before the final
 *             rounding (1.0f = none; 1/P gives the DDP mean).  Only for
 *             AR_SUM on AR_FLOAT32 / AR_BFLOAT16; otherwise it must be 1.0f.
 *   stream    a cudaStream_t (NULL = legacy default stream).
 * The caller owns every buffer; the pointer arrays are read during the call
 * only.  Every pointer must be 16-byte aligned device memory of the
 * communicator's device, and that device must be current.
 * Asynchronous: returns after enqueueing one kernel on `stream` (none when
 * count == 0).  Argument errors return synchronously (AR_ERR_INVALID_ARG,
 * AR_ERR_UNSUPPORTED) before anything is enqueued; launch failures return
 * AR_ERR_CUDA; device-side errors (a wait limit) are reported later by
 * ar_get_status.
 * Launch order: a call without an SM cap (AR_OPT_MAX_BLOCKS) is launched with
 * programmatic dependent launch, so its kernel may become resident while the
 * kernel before it on `stream` drains; it waits on the device until that
 * kernel has completed and its writes are visible before it reads or writes
 * any buffer, so the stream's order holds.  Every kernel of the library also
 * lets the kernel after it start early the same way: a kernel of the caller's
 * that is launched with programmatic stream serialization after a call must
 * wait (cudaGridDependencySynchronize) before it reads the call's results,
 * as the CUDA programming model requires of any such kernel.
 * CUDA graphs: every algorithm may be captured and replayed (the buffers
 * are then fixed).  The LL / LL128 epoch lives in device memory and each
 * launch takes the next value itself, so a replayed call never matches an
 * earlier call's staged words.  Calls on one communicator must still run one
 * at a time on the GPU (one stream, or streams ordered by events): they share
 * the staging areas and the epoch.
 */
ar_status_t ar_allreduce(ar_comm_t comm, const void* const* sendbufs, void* const* recvbufs,
                         size_t count, ar_dtype_t dtype, ar_op_t op, ar_algo_t algo,
                         float scale, void* stream);

/*
 * Device-side status of the calls made so far on `comm`: AR_SUCCESS or
 * AR_ERR_TIMEOUT (an LL / LL128 flag wait or a TMA-kernel mbarrier wait gave
 * up; that call's output is incomplete).  The collective runs asynchronously
 * on the caller's stream and is complete only after a stream synchronize
 * ("NCCL and NVSHMEM -- two GPU communication models, side by side", the
 * host-code example), so an error found while it runs can only be read
 * afterwards; reporting a wait that ran out instead of hanging follows the
 * fail-fast default and the timeout advice of the lecture_068 page, section 08
 * (debug and stability).
 * Reads and clears the device status word with a synchronous copy, so call it
 * after synchronizing the streams the calls ran on.  AR_ERR_CUDA if the copy
 * fails, AR_ERR_INVALID_ARG for a NULL comm.
 */
ar_status_t ar_get_status(ar_comm_t comm);

/* Static, human-readable name of a status code (never NULL).  The pages have
 * no counterpart: it exists so that callers and the AR_DEBUG trace can log a
 * status by name, the observability that the lecture_068 page, section 08,
 * asks of a communication library (NCCL_DEBUG=INFO as the first tool). */
const char* ar_get_error_string(ar_status_t status);

/* Frees the communicator's device memory.  Synchronizes the device first.
 * NULL is accepted (no-op).  The pages' host-code example creates the
 * communicator once (ncclCommInitRank) and never shows its teardown; the
 * checklist of "NCCL, NIXL, and Distributed GPU Communication" says a
 * communicator is set up once and reused, never created and destroyed inside
 * the training loop -- so this call belongs at shutdown. */
ar_status_t ar_destroy(ar_comm_t comm);

/*
 * Algorithm the call would run for these arguments: AR_ALGO_AUTO resolves to
 * AR_ALGO_LL when count * sizeof(dtype) <= the LL limit, else AR_ALGO_RING;
 * a forced algorithm is returned as is.  Host only, touches no device.
 */
ar_status_t ar_select_algo(ar_comm_t comm, size_t count, ar_dtype_t dtype, ar_algo_t algo,
                           ar_algo_t* chosen);

/* Per-communicator options (take effect on the next call; host only except
 * AR_OPT_LL_EPOCH). */
typedef enum {
    AR_OPT_LL_MAX_BYTES = 0,     /* LL limit in bytes per rank, 16 .. the size given
                                    at ar_init (default 65536 or AR_LL_MAX_BYTES)       */
    AR_OPT_LL_SPIN_LIMIT = 1,    /* polls of one LL / LL128 flag, or of one mbarrier
                                    phase in the TMA kernel, before AR_ERR_TIMEOUT
                                    (>= 1)                                          */
    AR_OPT_DEBUG = 2,            /* nonzero: one line per call on stderr               */
    AR_OPT_LL_SKIP_PRODUCER = 3, /* test hook: the LL / LL128 kernels skip staging and
                                    the TMA kernel's producer issues no copies, so
                                    every wait runs out and reports AR_ERR_TIMEOUT   */
    AR_OPT_HIER_GROUP = 4,       /* AR_ALGO_HIER ranks per group: a divisor of P
                                    (default 8; a call whose P it does not divide
                                    returns AR_ERR_UNSUPPORTED)                       */
    AR_OPT_LL128_MAX_BYTES = 6,  /* LL128 limit in bytes per rank, 16 .. the size given
                                    at ar_init (default 1 MiB or AR_LL128_MAX_BYTES)   */
    AR_OPT_AUTO_TUNED = 7,       /* nonzero: AUTO follows the table measured by
                                    ar_tune; 0: the fixed LL-up-to-the-limit rule
                                    (default; ar_tune sets it to 1)                  */
    AR_OPT_MAX_BLOCKS = 5,       /* > 0: ring / tree / hierarchical / reduce-scatter /
                                    all-gather kernels launch at most this many
                                    thread blocks (grid-stride), leaving the other
                                    SMs to kernels on other streams; 0 = no cap
                                    (default).  Below the SM count, ring / tree
                                    all-reduces and reduce-scatters with P <= 8
                                    run the kernel AR_OPT_CAPPED_KERNEL names,
                                    one block per SM (the TMA pipeline needs at
                                    least 4 KiB per rank per block, else the
                                    whole-GPU load/store kernel runs, capped);
                                    more
                                    ranks, and the hierarchical order, run the
                                    pipelined kernel in 768-thread blocks, one
                                    per SM; all-gathers of whole 16-byte pieces
                                    with at least 32 KiB per block run a TMA
                                    bulk-copy pipeline.  Results do not change.    */
    AR_OPT_CAPPED_KERNEL = 9,    /* kernel that P <= 8 ring / tree all-reduces and
                                    reduce-scatters run when AR_OPT_MAX_BLOCKS is
                                    below the SM count: AR_CAPPED_WIDE (default;
                                    1024-thread load/store blocks, one per SM --
                                    measured fastest alone) or AR_CAPPED_TMA (the
                                    TMA bulk-copy pipeline -- measured fastest
                                    beside GEMMs on the other SMs).  The initial
                                    value comes from the environment variable
                                    AR_CAPPED_KERNEL=wide|tma at ar_init.  Results
                                    do not change.                                 */
    AR_OPT_LL_EPOCH = 8          /* test hook: sets the last epoch used by LL and
                                    LL128 (0 .. 2^32 - 2; the next call uses
                                    value + 1; the call that uses 2^32 - 1 clears
                                    the staging area and restarts at 1).  Writes
                                    device memory synchronously: synchronize the
                                    communicator's streams first.                 */
} ar_option_t;

/* Values of AR_OPT_CAPPED_KERNEL. */
#define AR_CAPPED_WIDE 0
#define AR_CAPPED_TMA 1

ar_status_t ar_set_option(ar_comm_t comm, ar_option_t option, long long value);

/*
 * Measures which algorithm is fastest on this device for this communicator's
 * rank count and makes AUTO use the result.  NCCL picks among ring, tree and
 * its protocols by message size and hardware, and the crossover has to be
 * measured per platform ("NCCL and NVSHMEM -- two GPU communication models,
 * side by side": the ring / tree paragraph and exercise 6, force each
 * algorithm and find the crossover; "Demystifying NVSHMEM": selection is a
 * rule table, not an analytic model).  For every per-rank size 8 B * 2^i,
 * i < AR_TUNE_BUCKETS, it times RING, TREE, LL and LL128 (fp32 sum, 20 calls
 * back to back, within the LL / LL128 limits) and keeps the fastest; AUTO
 * then rounds a call's size up to a bucket and uses its entry.
 *   table  optional (table_len entries): the chosen algorithm per bucket.
 * Synchronous; allocates and frees 2 * nranks * 16 MiB of scratch buffers and
 * a stream.  Errors: AR_ERR_INVALID_ARG, AR_ERR_OOM, AR_ERR_CUDA, or the
 * status of a failed measurement call (the previous AUTO rule is kept).
 */
ar_status_t ar_tune(ar_comm_t comm, ar_algo_t* table, int table_len);

/*
 * Reduce-scatter ("NCCL, NIXL, and Distributed GPU Communication", section
 * "Reduce-scatter": the ranks' values are reduced and the result is split
 * into P shards, rank s receiving shard s).
 *   sendbufs  P device pointers to P * recvcount elements each (rank r's
 *             full vector)
 *   recvbufs  P device pointers to recvcount elements: recvbufs[s] receives
 *             reduced shard s
 * Shard s is folded in the ring order of all-reduce chunk s (x_s, then
 * x_{s+1}, ..., x_{s+P-1}); so when recvcount * sizeof(element) is a
 * multiple of 16, reduce-scatter followed by all-gather equals ar_allreduce
 * with AR_ALGO_RING bit for bit ("all-reduce = reduce-scatter + all-gather").
 * op, scale, stream, asynchrony and errors as for ar_allreduce.  Pointers
 * need only element alignment here; when every pointer and recvcount *
 * sizeof(element) are multiples of 16 bytes the 16-byte vector kernel runs,
 * otherwise an element-wise kernel with the same order.  Buffers may share
 * memory only when identical or in place (recvbufs[r] == sendbufs[r] +
 * r * recvcount elements).  recvcount == 0 is a no-op.
 */
ar_status_t ar_reduce_scatter(ar_comm_t comm, const void* const* sendbufs, void* const* recvbufs,
                              size_t recvcount, ar_dtype_t dtype, ar_op_t op, float scale,
                              void* stream);

/*
 * All-gather (same page, section "All-gather": every rank receives all
 * ranks' pieces, k ranks of N values giving k x N values on every rank).
 *   sendbufs  P device pointers to sendcount elements (rank s's piece)
 *   recvbufs  P device pointers to P * sendcount elements: every rank
 *             receives piece s at element offset s * sendcount
 * A copy (no arithmetic; dtype only sets the element size).  Pointers need
 * only element alignment (16-byte vectors are used when every pointer and
 * sendcount * sizeof(element) are multiples of 16).  Buffers may share memory
 * only when identical or in place (sendbufs[r] == recvbufs[r] + r * sendcount
 * elements).  Stream, asynchrony and errors as for ar_allreduce; sendcount
 * == 0 is a no-op.
 */
ar_status_t ar_all_gather(ar_comm_t comm, const void* const* sendbufs, void* const* recvbufs,
                          size_t sendcount, ar_dtype_t dtype, void* stream);

/*
 * LL all-reduce that allocates nothing.  (The pages have no counterpart: this
 * entry point exists for callers of this library that cannot allocate device
 * memory -- code whose device memory belongs to a framework's pool, code in a
 * latency-critical loop where cudaMalloc / cudaFree may synchronize the
 * device, code that may not allocate after start-up -- and so cannot hold a
 * communicator, whose ar_init allocates the LL staging area.)
 *
 * Same result as ar_allreduce(..., AR_ALGO_LL, ...) on the same arguments (the
 * ring combination order).  The staging area and the status word live in one
 * fixed array compiled into libar.so (about 1 MiB per GPU that loads the
 * library, held until the process exits), so it serves at most
 * AR_NOALLOC_MAX_RANKS ranks and AR_NOALLOC_MAX_BYTES bytes per rank; larger
 * requests return AR_ERR_UNSUPPORTED.  No cudaMalloc, cudaFree or allocating
 * library call is made.
 *   nranks        1 .. AR_NOALLOC_MAX_RANKS emulated ranks
 *   sendbufs,     host arrays of nranks device pointers, as for ar_allreduce
 *   recvbufs      (16-byte aligned, no partial overlap; exact aliasing allowed)
 *   count, dtype, op, scale, stream   as for ar_allreduce
 *   device_status NULL: asynchronous, returns after enqueueing the kernel.
 *                 Non-NULL: waits for `stream`, then stores AR_SUCCESS or
 *                 AR_ERR_TIMEOUT (a flag wait ran out in this or an earlier
 *                 call on this device) and clears the device status word.
 * The first call on each device looks up the array's device address with that
 * device current.  If that lookup fails (AR_ERR_CUDA), nothing is cached: the
 * next call on the device tries again.  Every call
 * on a device shares the one array: calls that overlap on the GPU (for example
 * on two streams at once) race and must not be issued.
 * Errors: AR_ERR_INVALID_ARG (bad pointer, alignment, overlap, enum, NaN
 * scale), AR_ERR_UNSUPPORTED (limits above, scale on int32 / min / max),
 * AR_ERR_CUDA (launch or status read failed).
 */
#define AR_NOALLOC_MAX_RANKS 8
#define AR_NOALLOC_MAX_BYTES 65536

ar_status_t ar_allreduce_ll_noalloc(int nranks, const void* const* sendbufs, void* const* recvbufs,
                                    size_t count, ar_dtype_t dtype, ar_op_t op, float scale,
                                    void* stream, int* device_status);

#ifdef __cplusplus
}
#endif

#endif /* AR_H_ */
