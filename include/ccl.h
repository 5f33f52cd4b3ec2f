/*
 * ccl.h -- C ABI of the single-GPU ring-collective library (libccl.so).
 *
 * N "ranks" are simulated on one GPU: each rank is a buffer in device memory
 * (normally a slice of one arena allocation).  Every collective computes the
 * exact data semantics of the textbook ring algorithm on the device:
 *
 *   ReduceScatter phase, step s = 0..N-2: rank i sends chunk (i-s) mod N to
 *   rank i+1 and adds the chunk (i-1-s) mod N arriving from rank i-1 into its
 *   own copy; AllGather phase: rank i forwards chunk (i+1-s) mod N and stores
 *   chunk (i-s) mod N.  (Collectives and sharded matmul, "ring ReduceScatter"
 *   and "ring AllGather"; AllReduce survey, "Algorithm 1: Ring AllReduce",
 *   phase 1 and 2; Collective Communication, Algorithm 1.)
 *
 * Chunk c of a K-element buffer holds len_c = K/N + (c < K mod N) elements
 * starting at off_c = sum_{d<c} len_d (the pages split evenly; the first
 * K mod N chunks take the remainder).  Chunk c is therefore folded in the order
 * x_c, x_{c+1}, ..., x_{c-1} (ranks mod N): each hop is one IEEE fp32 operation
 * rounded to nearest-even, followed by a round to the buffer type (identity for
 * fp32, round-to-nearest-even for bf16).  A NaN result is the canonical quiet
 * NaN (fp32 0x7FFFFFFF, bf16 0x7FFF).  AVG sums around the ring, then divides
 * the finished chunk once by N in fp32 before the gather, so every rank gets
 * identical bits.  AVG_PREMUL is NCCL's pre-multiplied average (Collective
 * Communication, libraries section on NCCL): every contribution is first
 * multiplied in fp32 by the correctly rounded reciprocal of N and rounded to
 * the buffer type, the scaled values are summed around the ring as SUM does,
 * and nothing is divided at the end.  It differs from AVG in the last bits for
 * N not a power of two (the same bits for N a power of two, barring
 * subnormals); its partial sums stay near the inputs' magnitude, where the
 * plain sum that AVG divides can overflow first.  MAX is NaN if
 * either side is NaN, else the larger, and
 * +0 against -0 gives +0; MIN likewise takes the smaller, and -0 wins the tie
 * (the pages list sum, min and max as the reductions: Collective
 * Communication, table of the six core primitives).
 *
 * Common conventions
 *   - Pointer arrays (send[], recv[], ptrs[]) are HOST arrays of nranks DEVICE
 *     pointers.  The caller owns every buffer; the library never frees them.
 *     A pointer to zero elements may be NULL (a ReduceScatter or Scatter
 *     output, or an AllGather or Gather input, for an empty chunk when
 *     count < nranks; a zero-length bucket tensor; an empty AllToAllv
 *     buffer), as may the entries a call ignores (noted per call); every other
 *     pointer a call uses must not be NULL (CCL_ERR_INVALID_ARG).
 *   - All entry points that take a stream are asynchronous: they validate
 *     their arguments on the host, enqueue kernels on `stream` (0 = legacy
 *     default stream) and return.  Completion is stream completion
 *     (Collective Communication, section on correctness: a non-blocking return
 *     means work in flight, not work done).
 *   - Argument errors are returned before anything is enqueued: NULL pointers,
 *     nranks outside [1, CCL_MAX_RANKS], counts that overflow, unknown dtype,
 *     op or mode, root out of range, and buffers that partially overlap
 *     (CCL_ERR_OVERLAP).  A CUDA launch error is returned as CCL_ERR_CUDA.
 *     Nothing aborts or traps.
 *   - count == 0 is a no-op returning CCL_OK; nranks == 1 is a copy (or
 *     nothing, in place).
 *   - In-place: send[r] == recv[r] is allowed for every rank.  Any other
 *     overlap between two buffers that the same call writes and reads is an
 *     error, except the in-place forms noted per call.
 *   - CCL_MODE_FUSED computes the ring's end state in one pass over memory (one
 *     launch).  CCL_MODE_STEP executes the ring's 2(N-1) steps one launch per
 *     step, in stream order, for validating the schedule; it gives identical
 *     bits and is slower.
 *   - CUDA graphs.  Fused-mode collectives, ccl_allreduce_algo,
 *     ccl_allreduce_compressed and ccl_check_identical enqueue only kernels
 *     whose arguments travel by value and allocate nothing, so they may be
 *     captured; a graph replays them on the pointers it was captured with.
 *     ccl_allreduce_compressed sets up its kernel (shared-memory opt-in) on
 *     its first call on a device: make that call before capturing.  In step
 *     mode, AllReduce, AllGather, Broadcast, Gather, Scatter and AllToAll(v)
 *     allocate nothing either and may be captured.  Step-mode ReduceScatter,
 *     Reduce and bucket AllReduce use a library-cached device workspace that
 *     a first or larger call allocates (and frees the old one): capture them
 *     only after a call at least as large has run on that device outside the
 *     capture, and while the graph may still be replayed make no larger such
 *     call and no ccl_finalize (either frees the memory the graph uses).
 *     ccl_reduce_scatter_step_static may be captured after its set-up call
 *     (count = 0).  ccl_allreduce_host refuses capture.
 *   - That step-mode workspace is one per device, shared by every call:
 *     step-mode ReduceScatter, Reduce or bucket AllReduce calls whose work
 *     overlaps on the GPU (different streams, different host threads) race on
 *     it and must be serialised.  Fused calls share nothing.
 *   - The environment variable CCL_MODE (or ccl_set_mode_override) can force
 *     one mode on every call that takes a mode argument; a forced step mode
 *     brings the step-mode rules above with it.  See "Settings" below.
 */
#ifndef CCL_H
#define CCL_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CCL_MAX_RANKS 1024
#define CCL_DEFAULT_BUCKET_BYTES (25u * 1024u * 1024u)
/* Size of the fixed device working space of ccl_reduce_scatter_step_static. */
#define CCL_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)

typedef enum { CCL_FP32 = 0, CCL_BF16 = 1 } ccl_dtype_t;
typedef enum {
    CCL_SUM = 0,
    CCL_AVG = 1,
    CCL_MAX = 2,
    CCL_PROD = 3,
    CCL_MIN = 4,
    CCL_AVG_PREMUL = 5 /* AllReduce, ReduceScatter, Reduce, bucket and host-buffer calls; ring order only */
} ccl_op_t;
typedef enum { CCL_MODE_FUSED = 0, CCL_MODE_STEP = 1 } ccl_mode_t;
typedef enum {
    CCL_ALGO_RING = 0,
    CCL_ALGO_HALVING_DOUBLING = 1,
    CCL_ALGO_TREE = 2,
    CCL_ALGO_HIERARCHICAL = 3
} ccl_algo_t;
typedef enum { CCL_COMP_INT8_BLOCK = 0, CCL_COMP_THRESHOLD = 1, CCL_COMP_TOPK = 2 } ccl_compressor_t;
typedef enum {
    CCL_OK = 0,
    CCL_ERR_INVALID_ARG = 1,
    CCL_ERR_UNSUPPORTED = 2,
    CCL_ERR_OVERLAP = 3,
    CCL_ERR_CUDA = 4,
    CCL_ERR_NO_MEMORY = 5,
    CCL_ERR_TIMEOUT = 6,
    CCL_ERR_CHECK_FAILED = 7
} ccl_status_t;

/* ------------------------------------------------------------------ */
/* Collectives                                                         */
/* ------------------------------------------------------------------ */

/* AllReduce: every rank ends with the reduction of all ranks' buffers
 * (Collectives and sharded matmul, "Reduce and AllReduce"; Collective
 * Communication, table of the six core primitives: y_i = sum_j x_j for all i).
 * send[r], recv[r]: `count` elements each.  In place when send[r] == recv[r].
 * Result: the ring fold of chunk c starting at rank c, on every rank. */
ccl_status_t ccl_allreduce(const void *const *send, void *const *recv, int nranks, size_t count,
                           ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode, cudaStream_t stream);

/* ReduceScatter: rank r receives chunk r of the reduction (Collectives and
 * sharded matmul, "Scatter and ReduceScatter": the sum of block r goes only to
 * rank r).  send[r]: `count` elements; recv[r]: len_r elements.  The fold
 * order is the AllReduce's (start at rank r), so ReduceScatter followed by
 * AllGather is bit-identical to AllReduce.  In place when
 * recv[r] == send[r] + off_r elements. */
ccl_status_t ccl_reduce_scatter(const void *const *send, void *const *recv, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode, cudaStream_t stream);

/* AllGather: send[r] holds len_r elements (chunk r of a `count`-element
 * result); every recv[q] receives all `count` elements, chunks in rank order
 * (Collectives and sharded matmul, "Gather and AllGather").  In place when
 * send[r] == recv[r] + off_r elements. */
ccl_status_t ccl_allgather(const void *const *send, void *const *recv, int nranks, size_t count,
                           ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream);

/* Broadcast: every recv[q] receives root's `count` elements
 * (Collectives and sharded matmul, "Broadcast").  Only send[root] is read;
 * other send[] entries may be NULL.  Step mode chains root -> root+1 -> ...
 * one hop per launch. */
ccl_status_t ccl_broadcast(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                           ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream);

/* AllToAll, uniform blocks: send[i] holds nranks blocks of `count` elements
 * ordered by destination; recv[j] receives nranks blocks ordered by source:
 * recv[j][i*count + t] = send[i][j*count + t] ("rank = row, block = column:
 * a transpose", Collectives and sharded matmul, "AllToAll"; Collective
 * Communication, Figure 5).  send and recv buffers must not overlap. */
ccl_status_t ccl_alltoall(const void *const *send, void *const *recv, int nranks, size_t count,
                          ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream);

/* AllToAllv: counts is a HOST array of nranks*nranks element counts,
 * counts[i*nranks + j] = elements rank i sends to rank j.  send[i] holds its
 * blocks ordered by destination, recv[j] its blocks ordered by source, both at
 * prefix-sum displacements (explicit per-destination counts and displacements,
 * Collective Communication, section on correctness).  Step mode follows the
 * pairwise schedule: at step k rank i sends to (i+k) mod N (Distributed LLM
 * collectives, "Pairwise algorithm"). */
ccl_status_t ccl_alltoallv(const void *const *send, void *const *recv, int nranks, const size_t *counts,
                           ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream);

/* Bucket-fused gradient AllReduce (Collective Communication, "Bucket fusion").
 * Each rank registers ntensors gradient tensors in forward order:
 * ptrs[r*ntensors + t] is rank r's tensor t (numels[t] elements, HOST array).
 * The tensors are laid end to end in REVERSE registration order, the stream is
 * cut into buckets of bucket_bytes (0 = the default bucket size: 25 MiB,
 * CCL_DEFAULT_BUCKET_BYTES, unless CCL_BUCKET_MB or
 * ccl_set_default_bucket_bytes changed it; the last bucket is partial and a
 * tensor may span buckets) and every bucket is
 * ring-AllReduced on its own, with its own N-chunk partition.  In place on the
 * tensors; nothing is copied into a staging bucket (the kernel reads and writes
 * the pieces where they are). */
ccl_status_t ccl_bucket_allreduce(void *const *ptrs, const size_t *numels, int ntensors, int nranks,
                                  size_t bucket_bytes, ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode,
                                  cudaStream_t stream);

/* Reduce: only recv[root] receives the reduction, the other ranks' buffers
 * are not touched (Collectives and sharded matmul, "Reduce and AllReduce";
 * Lesson 3, core concepts: AllReduce equals a Reduce followed by a Broadcast).
 * The root receives exactly the AllReduce's bits.  send[r]: `count` elements;
 * recv[root]: `count` elements; recv[r] for r != root is ignored (may be
 * NULL).  In place when send[root] == recv[root].  Step mode runs the ring's
 * ReduceScatter phase through a cached workspace, then brings each finished
 * chunk to the root. */
ccl_status_t ccl_reduce(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                        ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode, cudaStream_t stream);

/* Gather: recv[root] receives every rank's slice concatenated in rank order
 * (Lesson 3, core concepts: "Gather"; Collectives and sharded matmul, "Gather
 * and AllGather").  send[r] holds len_r elements (chunk r of `count`);
 * recv[r] for r != root is ignored.  In place when
 * send[root] == recv[root] + off_root elements; more generally, any send[r]
 * may already sit at its own place, recv[root] + off_r elements (its chunk is
 * then copied onto itself). */
ccl_status_t ccl_gather(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                        ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream);

/* Scatter: send[root]'s `count` elements are split into the N chunks and
 * chunk r goes to recv[r] (len_r elements) (Lesson 3, core concepts: "Scatter",
 * the inverse of Gather; Collectives and sharded matmul, "Scatter and
 * ReduceScatter").  send[r] for r != root is ignored.  In place when
 * recv[root] == send[root] + off_root elements; more generally, any recv[r]
 * may already sit at its own place, send[root] + off_r elements (its chunk is
 * then copied onto itself). */
ccl_status_t ccl_scatter(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                         ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream);

/* Bucket AllReduce overlapped with the backward pass (Collective
 * Communication, "Layer-wise overlap": a gradient hook per parameter starts a
 * bucket's AllReduce as soon as the bucket is full, while the backward pass
 * goes on).  ccl_bucketer_create takes the same tensors, layout and bucket
 * size as ccl_bucket_allreduce and plans the buckets once (the tensors stay
 * owned by the caller and must outlive the bucketer).  Each step, the caller
 * calls ccl_bucketer_mark_ready for every tensor once its gradient is final
 * on every rank, with an event recorded after it on the compute stream (or
 * NULL if comm_stream is already ordered after that work).  The call makes
 * comm_stream wait for that event (so the event need only be valid during the
 * call; mark tensors in the order they are produced, or a later wait delays
 * an earlier-filled bucket), and when all the tensors a bucket touches are
 * ready it enqueues the bucket's fused ring reduction on comm_stream.  Results
 * are bit-identical to ccl_bucket_allreduce.  ccl_bucketer_reset starts the
 * next step. */
typedef struct ccl_bucketer ccl_bucketer_t;
/* max_ctas > 0 caps each bucket kernel's grid so the reduction, which is
 * bound by memory bandwidth, runs beside the backward pass's compute-bound
 * kernels on part of the GPU instead of claiming every SM; 0 launches one CTA
 * per tile.  The bits do not depend on it. */
ccl_status_t ccl_bucketer_create(void *const *ptrs, const size_t *numels, int ntensors, int nranks,
                                 size_t bucket_bytes, ccl_dtype_t dtype, ccl_op_t op, int max_ctas,
                                 ccl_bucketer_t **out);
ccl_status_t ccl_bucketer_mark_ready(ccl_bucketer_t *b, int tensor, cudaEvent_t ready, cudaStream_t comm_stream);
ccl_status_t ccl_bucketer_reset(ccl_bucketer_t *b);
/* Buckets planned and buckets enqueued so far in this step. */
ccl_status_t ccl_bucketer_status(ccl_bucketer_t *b, size_t *nbuckets, size_t *launched);
ccl_status_t ccl_bucketer_destroy(ccl_bucketer_t *b);

/* AllReduce under another schedule's summation order, in one pass (fused).
 * Each schedule adds the contributions in its own order, so each gives its own
 * rounded bits; this call reproduces them exactly.
 *   CCL_ALGO_RING: the ring of ccl_allreduce (identical result).
 *   CCL_ALGO_HALVING_DOUBLING: round k pairs rank i with i XOR 2^k, k = 0, 1,
 *     ... (Collective Communication, "Recursive halving-doubling (butterfly)");
 *     for N not a power of two the first 2r ranks, r = N - 2^floor(log2 N), are
 *     first added pairwise (2v, 2v+1) (Distributed LLM collectives, "Recursive
 *     Halving-Doubling").  Per element: a balanced tree, adjacent leaves first.
 *   CCL_ALGO_TREE: binomial tree to rank 0, level k adding rank i + 2^k into
 *     rank i, then broadcast (Collective Communication, "Tree AllReduce").
 *   CCL_ALGO_HIERARCHICAL: ring ReduceScatter inside groups of group_size
 *     consecutive ranks, ring AllReduce among the groups' representatives,
 *     ring AllGather inside the groups (AllReduce survey, two-level table);
 *     group_size must divide nranks (1 or nranks gives the flat ring).
 * AVG divides the finished sum once by N; CCL_AVG_PREMUL is accepted with
 * CCL_ALGO_RING only (CCL_ERR_UNSUPPORTED otherwise).  Buffers as
 * ccl_allreduce (in place when send[r] == recv[r]).  group_size is ignored
 * except for CCL_ALGO_HIERARCHICAL. */
ccl_status_t ccl_allreduce_algo(const void *const *send, void *const *recv, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, ccl_algo_t algo, int group_size,
                                cudaStream_t stream);

/* Compressed AllReduce with error feedback (Collective Communication,
 * "Gradient compression": blockwise INT8 quantization, and "Error feedback and
 * residual accumulation", Definition 1.4).  grads[r]: `count` elements of
 * dtype, in place; residuals[r]: `count` fp32 per rank, zero before the first
 * step, carried by the caller from step to step.  Each rank compresses
 * u = g + e and keeps e' = u - v:
 *   CCL_COMP_INT8_BLOCK (block = 64 or 128): s = max|u| / 127 over each
 *     block, q = round(u / s) (ties to even), v = q * s;
 *   CCL_COMP_THRESHOLD (the greedy 1-bit compressor of the pages' Tables 3
 *     and 4): v = 1 when u >= threshold, else 0.
 * The transmitted v are AllReduced in ring order in fp32 (op CCL_SUM, or
 * CCL_AVG dividing once by N; CCL_AVG_PREMUL returns CCL_ERR_UNSUPPORTED) and
 * rounded once to dtype, written to every grads[r].  Up to 16 ranks; grads
 * and residuals must not overlap.  CCL_COMP_TOPK needs k and a work buffer:
 * it is ccl_allreduce_topk's (CCL_ERR_INVALID_ARG here).  One launch, two
 * with a partial last block. */
ccl_status_t ccl_allreduce_compressed(void *const *grads, float *const *residuals, int nranks, size_t count,
                                      ccl_dtype_t dtype, ccl_op_t op, ccl_compressor_t comp, int block,
                                      float threshold, cudaStream_t stream);

/* Top-k sparsified AllReduce with error feedback (Collective Communication,
 * "Top-k sparsification", and "Error feedback and residual accumulation",
 * Definition 1.4).  grads[r]: `count` elements of dtype, in place;
 * residuals[r]: `count` fp32 per rank, zero before the first step, carried by
 * the caller.  Each rank forms u = g + e (fp32) and sends v = u where |u| is
 * at least its k-th largest magnitude |u|_(k), else 0 -- every value tied
 * with the k-th is sent, so a rank may send more than k -- and keeps
 * e' = u - v.  Magnitudes are ordered as the bit patterns of |u|, so a NaN
 * counts as the largest and is always sent.  k = 0 sends nothing; k >= count
 * sends everything.  The sent values are AllReduced in ring order in fp32
 * (CCL_SUM, or CCL_AVG dividing once by N; CCL_AVG_PREMUL returns
 * CCL_ERR_UNSUPPORTED) and rounded once to dtype, written to every grads[r].
 * The threshold is found on the device by a radix select, with no host round
 * trip: a sample (one 256-element run in 16; in 32, 64 or 128 when the
 * sparser sample still expects 4096 keys at or above the k-th and the
 * standard deviation of its estimate of that key's rank, sqrt(k * 128) for
 * one run in 128, is at most count / 2048) places a window of one to four top-12-bit bins, one full pass
 * over g and e counts every key's top bits and the low 19 bits of the keys
 * in the window, and a second full pass runs only when the k-th key's top
 * bin fell outside the window.  One more pass then sends, keeps the
 * residuals and reduces.  work: device memory of ccl_plan_topk_work_bytes
 * bytes (about 10 MiB per rank), 16-byte aligned,
 * owned by the caller, not shared with a concurrent call; its contents need
 * no initialisation.  Up to 16 ranks and count < 2^32; grads, residuals and
 * work must not overlap (CCL_ERR_OVERLAP).  Launches: one to reset the work
 * buffer; when 0 < k < count the sample and its scan (large aligned inputs),
 * the full pass and its scan, the two fallback launches (which return at once
 * when the window held the bin), and the low histogram's two scans; and the
 * compressed pass (one launch, two with a partial last block of 128). */
ccl_status_t ccl_allreduce_topk(void *const *grads, float *const *residuals, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, size_t k, void *work, size_t work_bytes,
                                cudaStream_t stream);

/* Bytes of the work buffer ccl_allreduce_topk needs for nranks ranks. */
ccl_status_t ccl_plan_topk_work_bytes(int nranks, size_t *bytes);

/* The sample ccl_allreduce_topk takes for count elements per rank and this
 * k, when every gradient and residual is 16-byte aligned (others are never
 * sampled): *every = f when the sample reads one 256-element run in f (16,
 * 32, 64 or 128, by the rule in ccl_allreduce_topk's description), 0 when it
 * takes none -- k = 0, k >= count, or too few elements for the sample to
 * place a window (the select then counts the k-th key's top bin in a second
 * full pass).  Host only; CCL_ERR_INVALID_ARG for a null every or
 * count >= 2^32. */
ccl_status_t ccl_plan_topk_sample(size_t count, size_t k, uint32_t *every);

/* Bytes one rank would put on a link for Top-k with fp32 values and int32
 * indices: 8 * min(k, count), a ratio of 4 count / bytes = count / (2k) over
 * dense fp32 (Collective Communication, "Top-k sparsification": 500x, not
 * 1000x, for k = 0.001 count).  Host only. */
ccl_status_t ccl_plan_topk_bytes(size_t count, size_t k, size_t *bytes);

/* Step-by-step ReduceScatter that allocates nothing.  The pages have no
 * counterpart: this exists for callers that cannot let a library call
 * cudaMalloc -- a process whose framework has already reserved the GPU's
 * memory in its own caching pool (a raw cudaMalloc then fails or fragments
 * what is left), code that must not stall other streams on the device
 * synchronisation cudaMalloc/cudaFree can imply, or hosts that forbid driver
 * allocations after start-up.
 * Same arguments, result and error checks as ccl_reduce_scatter in
 * CCL_MODE_STEP (identical bits; the checks are the same code), but the
 * working copies of the N inputs live in one fixed array of
 * CCL_STATIC_SCRATCH_BYTES (32 MiB) in device memory, held by every GPU that
 * reserves it until the process exits.  nranks * round_up(count * element
 * size, 256) must not exceed CCL_STATIC_SCRATCH_BYTES: larger calls return
 * CCL_ERR_INVALID_ARG before anything is enqueued.  It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *   - Set-up, once per device: a call with count = 0 (valid nranks, dtype and
 *     op, non-NULL pointer arrays whose entries are not read) looks up the
 *     array's device address (cudaGetSymbolAddress, with that device current),
 *     loads every kernel this entry launches, caches the address and enqueues
 *     nothing; it returns CCL_ERR_CUDA if that fails.  Under CUDA's lazy module
 *     loading (the default since CUDA 12.2) this lookup is when the driver
 *     reserves the array, so make this call at start-up, before a caching
 *     pool takes the GPU's memory and before any stream capture.  A first
 *     call with count > 0 does the same set-up itself.
 *   - Every call on a device shares the array and leaves its contents behind.
 *     Each call overwrites every byte it later reads, so nothing needs
 *     clearing, but calls whose work overlaps on the GPU (other streams, other
 *     host threads) race on it: serialise them.
 *   - ccl_finalize forgets the cached address of the current device; call it
 *     after a cudaDeviceReset, before the next call on that device. */
ccl_status_t ccl_reduce_scatter_step_static(const void *const *send, void *const *recv, int nranks, size_t count,
                                            ccl_dtype_t dtype, ccl_op_t op, cudaStream_t stream);

/* Device working space that lets ccl_allreduce_host run at the host link's
 * speed: three stages of 64 MiB. */
#define CCL_HOST_WORK_BYTES_DEFAULT (192u * 1024u * 1024u)

/* AllReduce of rank buffers that live in HOST memory: the same result, bit for
 * bit, as ccl_allreduce on the same data (the ring fold of chunk c starting at
 * rank c of the count-element partition).  send[r], recv[r]: `count` elements
 * each, any memory the GPU can copy from and to (cudaMemcpyDefault); page-
 * locked host memory (cudaHostAlloc, cudaHostRegister) is what makes the
 * copies asynchronous and overlapped.  In place when send[r] == recv[r].
 * Two paths give the same bits:
 *   - in place over the host link, when CCL_HOST_PATH=direct (or
 *     ccl_set_host_path(CCL_HOST_PATH_DIRECT)) and every send[r] and recv[r]
 *     is page-locked host memory that the current device can address: one
 *     fused AllReduce launch on `stream` reads and writes them directly
 *     (both link directions busy at once, nothing staged; `work` is
 *     validated but not used);
 *   - staged, the default, and for any other memory:
 * the vector moves through `work` (DEVICE memory, caller-owned, 16-byte
 * aligned, work_bytes >= 3 * nranks * 256 * element size; larger is faster,
 * up to CCL_HOST_WORK_BYTES_DEFAULT) in slices: copies in and out run on two
 * library-owned streams so that both directions of the host link are busy at
 * once, and each slice is reduced on `stream` (the link is the bottleneck:
 * Collective Communication, Table 1, GPU<->CPU row; the overlap is the
 * pipelining of the section on NCCL).  Ordering: the call starts after the
 * work already enqueued on `stream`, and work enqueued on `stream` afterwards
 * sees every result in recv[].  Calls that share `work` must be ordered (one
 * stream, or events); the library orders its own stage reuse across calls.
 * Returns CCL_ERR_UNSUPPORTED while `stream` is being captured into a CUDA
 * graph, CCL_ERR_INVALID_ARG for a work buffer that is too small or
 * misaligned, and the common argument errors otherwise. */
ccl_status_t ccl_allreduce_host(const void *const *send, void *const *recv, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, void *work, size_t work_bytes,
                                cudaStream_t stream);

/* ------------------------------------------------------------------ */
/* Result checks and tracing                                           */
/* ------------------------------------------------------------------ */

/* Adds to *mismatches (a DEVICE counter the caller zeroes) the number of
 * elements, summed over ranks 1..nranks-1, whose bits differ from rank 0's.
 * After an AllReduce every rank must hold the same bits (Collective
 * Communication, Definition 1.1); the pages ask that results be checked
 * against silent corruption (section on pitfalls).  Never traps. */
ccl_status_t ccl_check_identical(const void *const *bufs, int nranks, size_t count, ccl_dtype_t dtype,
                                 unsigned long long *mismatches, cudaStream_t stream);

/* Automatic result checks, off unless CCL_CHECK is set (to anything but 0)
 * or enabled here.  While on, every AllReduce (fused or step, any order, the
 * compressed one), AllGather and Broadcast that succeeds also enqueues
 * ccl_check_identical over its outputs on the call's stream, adding to a
 * per-device counter the library owns (one cudaMalloc on the first checked
 * call on a device: make it before any stream capture).  Never traps. */
void ccl_set_check(int enabled);
/* Waits for the whole device, stores the current device's counter in
 * *mismatches (0 if nothing was checked yet) and, when reset != 0, sets the
 * counter back to 0. */
ccl_status_t ccl_check_read(unsigned long long *mismatches, int reset);

/* Debug builds (libccl_debug.so, compiled with CCL_DEBUG_BOUNDS) check every
 * global load and store of every kernel against the byte ranges of the
 * call's own buffers, library workspace included; an access outside them is
 * skipped, never performed, and counted.  Waits for the device and returns
 * the count and the first offending address.  Release builds return
 * CCL_ERR_UNSUPPORTED.  Calls whose work overlaps on the GPU share the range
 * table in debug builds: run them one at a time there. */
ccl_status_t ccl_debug_faults(unsigned long long *faults, unsigned long long *first_address);

/* One traced call: the collective, its shape, the kernels it enqueued, the
 * host time it took to validate, plan and enqueue, and its device time. */
typedef struct {
    char collective[24];
    int nranks;
    int dtype;
    int op;   /* -1 where the collective takes none */
    int mode; /* or the algorithm / compressor of the _algo / _compressed calls */
    int status;
    unsigned launches;
    unsigned long long count;
    unsigned long long host_ns;
    unsigned long long seq;
    /* Device time from the start to the end of the call's work on its stream
     * (two events recorded around it; Collective Communication, libraries
     * section: time a collective against a bare baseline with a profiler
     * before tuning it).  0 until that work has completed on the device --
     * ccl_trace_read fills it in once it has -- and 0 for calls not timed:
     * made while the stream was being captured into a CUDA graph, or in a
     * process without a device. */
    unsigned long long gpu_ns;
} ccl_trace_record_t;

/* Tracing is off unless CCL_TRACE is set (to anything but 0) or enabled here.
 * The last 4096 calls are kept. */
void ccl_set_trace(int enabled);
/* Copies up to max_records of the newest records, oldest first, into out
 * (out == NULL: returns how many are held). */
size_t ccl_trace_read(ccl_trace_record_t *out, size_t max_records);
void ccl_trace_clear(void);

/* ------------------------------------------------------------------ */
/* Settings (host only; no GPU needed)                                 */
/* ------------------------------------------------------------------ */

/* Library-wide settings, read from the environment once, on first use, and
 * replaced by the setters below (Collective Communication, libraries section:
 * NCCL is steered by environment variables such as NCCL_ALGO; bucket fusion
 * section: DDP's bucket_cap_mb, 25 MB by default).
 *   CCL_MODE=fused | step (any case): every call that takes a mode argument
 *     (AllReduce, ReduceScatter, AllGather, Broadcast, Reduce, Gather,
 *     Scatter, AllToAll(v), bucket AllReduce) runs in that mode whatever it
 *     passes, so that a whole program can be re-run with the ring executed
 *     step by step (same bits, slower) without changing its calls.  Unset or
 *     empty: each call's own argument.  A mode argument that is not a valid
 *     ccl_mode_t is still rejected.  Trace records show the mode that ran.
 *   CCL_BUCKET_MB=<MiB>, a positive decimal number (e.g. 25 or 0.5): the
 *     bucket size of ccl_bucket_allreduce and ccl_bucketer_create calls that
 *     pass bucket_bytes = 0; at least 4 bytes, at most 1 TiB.
 *   CCL_HOST_PATH=staged|direct: how ccl_allreduce_host moves its buffers.
 *     staged (the default): slices go through the caller's work buffer.
 *     direct: when every buffer is page-locked host memory that the device
 *     can address (cudaHostAlloc, cudaHostRegister), one fused launch reads
 *     and writes them in place over the host link; other memory is staged.
 *     ccl_set_host_path replaces it.
 *   CCL_TRACE, CCL_CHECK: ccl_set_trace, ccl_set_check.
 * A value that cannot be read is ignored (the default stays) with one line on
 * stderr.  The settings are process-wide and may be changed at any time; a
 * call uses the values current when it is made. */
typedef struct {
    int mode_override;           /* -1: none; else CCL_MODE_FUSED or CCL_MODE_STEP */
    int trace;                   /* 1 when call tracing is on */
    int check;                   /* 1 when automatic result checks are on */
    int host_path;               /* CCL_HOST_PATH_STAGED or CCL_HOST_PATH_DIRECT */
    size_t default_bucket_bytes; /* the bucket size that bucket_bytes = 0 selects */
} ccl_config_t;

/* The current settings (CCL_ERR_INVALID_ARG for a NULL out). */
ccl_status_t ccl_get_config(ccl_config_t *out);
/* mode: CCL_MODE_FUSED or CCL_MODE_STEP forces that mode; -1 removes the
 * override (CCL_MODE is then no longer consulted).  Anything else:
 * CCL_ERR_INVALID_ARG, nothing changed. */
ccl_status_t ccl_set_mode_override(int mode);
/* bytes >= 4 sets the default bucket size; 0 restores 25 MiB
 * (CCL_DEFAULT_BUCKET_BYTES); 1 to 3: CCL_ERR_INVALID_ARG, nothing changed. */
ccl_status_t ccl_set_default_bucket_bytes(size_t bytes);
/* ccl_allreduce_host's path: CCL_HOST_PATH_STAGED (through the work buffer)
 * or CCL_HOST_PATH_DIRECT (in place over the host link when every buffer
 * allows it, else staged).  Anything else: CCL_ERR_INVALID_ARG, nothing
 * changed. */
#define CCL_HOST_PATH_STAGED 0
#define CCL_HOST_PATH_DIRECT 1
ccl_status_t ccl_set_host_path(int path);

/* ------------------------------------------------------------------ */
/* Planner (host only; no GPU needed)                                  */
/* ------------------------------------------------------------------ */

/* Chunk partition of `count` elements over nranks: off[c], len[c] (HOST arrays
 * of nranks entries, written by the call). */
ccl_status_t ccl_plan_chunks(size_t count, int nranks, size_t *off, size_t *len);

/* Ring step table, HOST array of 2*(nranks-1)*nranks*3 int32 laid out
 * [phase][s][rank] = {send chunk, recv chunk, source rank}; phase 0 is the
 * ReduceScatter phase, phase 1 the AllGather phase. */
ccl_status_t ccl_plan_ring_schedule(int nranks, int32_t *table);

/* Bucket boundaries of the reversed tensor stream: writes min(nbuckets,
 * max_buckets)+1 stream offsets into starts (bucket b covers
 * [starts[b], starts[b+1])) and the bucket count into *nbuckets. */
ccl_status_t ccl_plan_buckets(const size_t *numels, int ntensors, size_t bucket_elems, size_t *starts,
                              size_t max_buckets, size_t *nbuckets);

/* AllToAllv displacements: sdispl[i*N+j] = elements before block j in
 * send[i]; rdispl[j*N+i] = elements before block i in recv[j]. */
ccl_status_t ccl_plan_alltoallv(int nranks, const size_t *counts, size_t *sdispl, size_t *rdispl);

/* Bytes one rank would put on a link for `count` elements under a
 * compressor: INT8 block: count + 4 * ceil(count / block) (codes plus fp32
 * scales, 4b/(b+4) times fewer than fp32: 3.88 at b = 128); THRESHOLD:
 * ceil(count / 8).  TOPK depends on k: ccl_plan_topk_bytes (CCL_ERR_INVALID_ARG
 * here). */
ccl_status_t ccl_plan_compressed_bytes(size_t count, ccl_compressor_t comp, int block, size_t *bytes);

/* Slices of ccl_allreduce_host for these arguments: writes up to max_slices
 * (off, len) pairs, in elements of every rank's buffer, and the total number
 * into *nslices (off/len may be NULL to ask for the number only).  The slices
 * tile [0, count) in order; each is at most the stage length
 * floor(work_bytes / (3 * nranks * element size)) rounded down to a multiple
 * of 256 elements, starts on a multiple of 256, and they grow from 1/16 of the
 * stage length at the start and shrink the same way at the end. */
ccl_status_t ccl_plan_host_slices(size_t count, int nranks, ccl_dtype_t dtype, size_t work_bytes, size_t *off,
                                  size_t *len, size_t max_slices, size_t *nslices);

/* Arena layout: per-rank stride (bytes_per_rank rounded up to `align`, a power
 * of two >= 256) and total bytes for nranks rank buffers in one allocation. */
ccl_status_t ccl_arena_layout(int nranks, size_t bytes_per_rank, size_t align, size_t *stride, size_t *total);

/* ------------------------------------------------------------------ */
/* Misc                                                                */
/* ------------------------------------------------------------------ */

const char *ccl_status_string(ccl_status_t status);
int ccl_version(void);

/* Number of kernels this library has enqueued since it was loaded (host-side
 * counter, for accounting; thread-safe). */
unsigned long long ccl_launch_count(void);

/* Per-rank traffic of the step-by-step mode (Lesson 3, reference solution:
 * every rank counts what it sends, and an AllReduce moves 2(N-1)K/N elements
 * per rank when N divides K).  sent[j] (HOST array of nranks entries) receives
 * the elements rank j has sent in the ring steps that this host thread's
 * step-mode calls launched since the last reset: the ReduceScatter and
 * AllGather steps of AllReduce, ReduceScatter, AllGather, Reduce and bucket
 * AllReduce, and ccl_reduce_scatter_step_static.  At ReduceScatter step s
 * rank j sends chunk (j - s) mod N, at the AllReduce's AllGather step s chunk
 * (j + 1 - s) mod N, and at the AllGather entry point's step s chunk
 * (j - s) mod N (the lengths of the call's chunk partition).  Copies outside
 * the ring (placing ReduceScatter's results, Broadcast's chain, the pairwise
 * AllToAll) are not counted, nor is anything in fused mode.  reset != 0 zeroes
 * the counters after reading.  Host only; CCL_ERR_INVALID_ARG for nranks
 * outside [1, CCL_MAX_RANKS] or a NULL sent. */
ccl_status_t ccl_step_sent(int nranks, unsigned long long *sent, int reset);

/* Frees the library's cached device workspace on the current device (used by
 * step-mode ReduceScatter, Reduce and bucket AllReduce) and forgets the cached
 * address of ccl_reduce_scatter_step_static's fixed array there (the array
 * itself stays).  Safe to call at any time when no call of this library is in
 * flight; call it after a cudaDeviceReset, before the next call on that
 * device, since the reset invalidates both. */
ccl_status_t ccl_finalize(void);

#ifdef __cplusplus
}
#endif

#endif /* CCL_H */
