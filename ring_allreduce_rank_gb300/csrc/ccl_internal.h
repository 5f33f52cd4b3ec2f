// ccl_internal.h -- host-side declarations shared by the library's translation
// units: kernel parameter blocks and launchers.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "../../include/ccl.h"
#include "ccl_device.cuh"
#include "fused.h"

namespace ccl {

// ------------------------------------------------------------------ argument checks
inline size_t elem_size(ccl_dtype_t dt) { return dt == CCL_BF16 ? 2 : 4; }
inline bool valid_dtype(ccl_dtype_t dt) { return dt == CCL_FP32 || dt == CCL_BF16; }
inline bool valid_op(ccl_op_t op)
{
    return op == CCL_SUM || op == CCL_AVG || op == CCL_MAX || op == CCL_PROD || op == CCL_MIN ||
           op == CCL_AVG_PREMUL;
}
// Operators that change a value even with one rank (x / 1 or x * 1 turns a
// NaN into the canonical NaN), so N = 1 in place is not a no-op for them.
inline bool scales(int op) { return op == CCL_AVG || op == CCL_AVG_PREMUL; }
// Step mode: a separate scaling launch after the ReduceScatter phase -- AVG's
// division, or the pre-multiplied AVG's scaling when N = 1 gives it no hop.
inline bool step_scale(int op, int nranks) { return op == CCL_AVG || (op == CCL_AVG_PREMUL && nranks == 1); }
inline bool valid_mode(ccl_mode_t m) { return m == CCL_MODE_FUSED || m == CCL_MODE_STEP; }
inline bool valid_ranks(int n) { return n >= 1 && n <= CCL_MAX_RANKS; }

inline bool mul_overflows(size_t a, size_t b) { return a != 0 && b > SIZE_MAX / a; }

inline ccl_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? CCL_OK : CCL_ERR_CUDA; }

// A byte range touched by a call: lo/hi, which rank, read or write.
struct Range {
    uintptr_t lo, hi;
    int rank;
};

// Writes must be pairwise disjoint; a read may overlap a write only in one of
// the call's in-place forms, decided by `allowed(read, write)`.
template <class Allowed>
inline ccl_status_t check_overlaps(std::vector<Range> writes, const std::vector<Range> &reads, Allowed allowed)
{
    writes.erase(std::remove_if(writes.begin(), writes.end(), [](const Range &r) { return r.lo == r.hi; }),
                 writes.end());
    std::sort(writes.begin(), writes.end(), [](const Range &a, const Range &b) { return a.lo < b.lo; });
    for (size_t i = 1; i < writes.size(); ++i)
        if (writes[i].lo < writes[i - 1].hi)
            return CCL_ERR_OVERLAP;
    for (const Range &r : reads) {
        if (r.lo == r.hi)
            continue;
        // first write whose end is past the read's start (ends are sorted too)
        auto it = std::upper_bound(writes.begin(), writes.end(), r.lo,
                                   [](uintptr_t v, const Range &w) { return v < w.hi; });
        for (; it != writes.end() && it->lo < r.hi; ++it)
            if (!allowed(r, *it))
                return CCL_ERR_OVERLAP;
    }
    return CCL_OK;
}

inline Range range_of(const void *p, size_t bytes, int rank)
{
    return Range{(uintptr_t)p, (uintptr_t)p + bytes, rank};
}

inline Partition make_partition(size_t count, int nranks)
{
    Partition p;
    p.q = count / (uint64_t)nranks;
    p.rem = (uint32_t)(count % (uint64_t)nranks);
    return p;
}

// ReduceScatter's argument checks (all but the mode), shared by
// ccl_reduce_scatter and ccl_reduce_scatter_step_static so that both answer
// every call alike: enums, NULL pointers (an empty chunk's output may be NULL),
// byte-count overflow, and overlaps (outputs pairwise disjoint; an output may
// sit inside its own rank's input only at that rank's chunk offset).  On
// CCL_OK, w and r hold the call's written and read ranges (empty for
// count = 0).
ccl_status_t check_reduce_scatter(const void *const *send, void *const *recv, int nranks, size_t count,
                                  ccl_dtype_t dtype, ccl_op_t op, std::vector<Range> &w, std::vector<Range> &r);


// ------------------------------------------------------------------ chained launches
// Kernels that run as a chain of programmatic dependent launches call this
// first: it waits until the kernel before it in the stream has completed and
// its writes are visible, then lets the next kernel's CTAs be scheduled, so
// that a launch and its ramp-up overlap the previous kernel's tail.  In a
// launch without the attribute the wait returns at once.
__device__ __forceinline__ void chain_entry()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// A launch in such a chain (programmatic stream serialisation).
template <class P>
inline cudaError_t launch_chained(void (*kernel)(P), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                  const P &p)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// ------------------------------------------------------------------ step mode
enum StepKind {
    STEP_RS = 0,     // rank i: chunk (i-1-s) += rank (i-1)'s copy
    STEP_AG = 1,     // rank i: chunk (i-s) = rank (i-1)'s copy (after the RS phase)
    STEP_AG_API = 2, // rank i: chunk (i-1-s) = rank (i-1)'s copy (AllGather from chunk i at rank i)
    STEP_SCALE = 3   // rank i: chunk (i+1) /= N (AVG, at the holder); pre-multiplied AVG: *= 1/N
};

template <int MAXR> struct StepParams {
    void *buf[MAXR];
    Partition part;
    int nranks;
    int s;
    int kind;
    int vec_aligned;
    uint32_t tiles;
    float n_f;
    float inv_n; // 1/nranks correctly rounded (pre-multiplied AVG)
};

cudaError_t launch_ring_step(int dt, int op, int kind, int s, void *const *bufs, int nranks, uint64_t count,
                             cudaStream_t stream);

// Loads every ring-step kernel into the current device's context (CUDA loads
// kernels lazily, at first launch, by default).
cudaError_t preload_ring_step_kernels();

// ------------------------------------------------------------------ copies
struct CopySeg {
    const char *src;
    char *dst;
    uint64_t nbytes;
    uint64_t tile_begin; // first tile index of this segment (prefix sum)
};

// Enqueue byte copies of the given segments (any alignment), split into as
// many launches as the parameter space requires.
cudaError_t launch_copy_segments(const CopySeg *segs, size_t nseg, cudaStream_t stream);

// Loads every segment-copy kernel into the current device's context.
cudaError_t preload_copy_kernels();

// AllGather / Broadcast fan-out: each source element is read once and written
// to every destination.  AllGather: src[c] is chunk c (partition of count over
// nchunks = ndst), destination offset off_c.  Broadcast: nchunks = 1.
cudaError_t launch_fanout(int dt, const void *const *src, int nchunks, void *const *dst, int ndst, uint64_t count,
                          cudaStream_t stream);

// ------------------------------------------------------------------ buckets
struct RedSeg {
    uint32_t tp;     // index of rank 0's pointer of this tensor in the pointer table
    uint32_t c;      // ring rotation start (chunk index within the bucket)
    uint64_t off;    // element offset inside the tensor
    uint64_t len;    // elements
    uint64_t tile_begin;
};

// max_ctas > 0 caps the grid (the CTAs then walk the tiles), so the
// reduction can run beside other kernels on part of the GPU.
cudaError_t launch_bucket_reduce(int dt, int op, void *const *tensor_ptrs /* [t*nranks + r] */, int ntensors,
                                 int nranks, const RedSeg *segs, size_t nseg, cudaStream_t stream, int max_ctas = 0);

// Bucket layout of a set of gradient tensors: the tensors laid end to end in
// reverse registration order, cut into buckets of B elements, and every
// (bucket, chunk) stream range cut at tensor boundaries into segments.
struct BucketPlan {
    size_t total = 0;                        // elements in the stream
    std::vector<size_t> pos;                 // stream position of tensor t
    std::vector<size_t> start;               // bucket b covers [start[b], start[b+1])
    std::vector<std::vector<RedSeg>> segs;   // per bucket
    std::vector<std::vector<int>> tensors;   // per bucket: the tensors it touches
};
void build_bucket_plan(const size_t *numels, int ntensors, int nranks, size_t bucket_elems, BucketPlan &plan);

// ------------------------------------------------------------------ other schedules' orders
enum Algo { ALGO_RING = 0, ALGO_HD = 1, ALGO_TREE = 2, ALGO_HIER = 3 };

// One-pass AllReduce under halving-doubling, binomial-tree or two-level
// hierarchical (group = ranks per group) summation order.
cudaError_t launch_order_allreduce(int dt, int op, int algo, int group, const void *const *send, void *const *recv,
                                   int nranks, uint64_t count, cudaStream_t stream);

// ------------------------------------------------------------------ compressed AllReduce
enum Compressor { COMP_INT8_BLOCK = 0, COMP_THRESHOLD = 1, COMP_TOPK = 2 };

// Error-feedback compression of every rank's gradient, ring-order fp32
// AllReduce of the transmitted values, one round to the gradients' type.
// COMP_TOPK reads each rank's threshold key from tau[rank] (device memory).
cudaError_t launch_compressed_allreduce(int dt, bool avg, int comp, int block, float threshold,
                                        void *const *grads, float *const *res, int nranks, uint64_t count,
                                        const uint32_t *tau, cudaStream_t stream);

// Top-k threshold per rank: the k-th largest key |u| (bits, sign cleared) of
// u = g + e, written to *tau_out[rank] in `work` (topk_work_bytes(nranks)).
constexpr int kTopkMaxRanks = 16;
size_t topk_work_bytes(int nranks);
// The sample's density for count elements and this k (one run of 256 in the
// returned number), or 0 when the select takes no sample; for buffers that
// are all 16-byte aligned (others are never sampled).
uint32_t topk_sample_every(uint64_t count, uint64_t k);
cudaError_t launch_topk_select(int dt, void *const *grads, float *const *res, int nranks, uint64_t count,
                               uint64_t k, void *work, const uint32_t **tau_out, cudaStream_t stream);

// ------------------------------------------------------------------ host-buffer AllReduce
constexpr int kHostStages = 3;            // device stages in flight: copy-in, reduce, copy-out
constexpr uint64_t kHostSliceUnit = 256;  // slice starts and stage lengths are multiples of this (elements)

struct HostSlice {
    uint64_t off, len; // elements of every rank's buffer
};

// Elements per rank in one stage of a work buffer of work_bytes (a multiple of
// kHostSliceUnit; 0 if the buffer is too small).
uint64_t host_stage_elems(int nranks, size_t elem_size, size_t work_bytes);
// Slices of [0, count): growing from stage_elems/16 to stage_elems, then
// shrinking again towards the end; every one at most stage_elems long.
void plan_host_slices(uint64_t count, uint64_t stage_elems, std::vector<HostSlice> &slices);
// Pipelined copy-in / reduce / copy-out through `work`; validated arguments.
cudaError_t run_host_allreduce(int dt, int op, const void *const *send, void *const *recv, int nranks,
                               uint64_t count, void *work, size_t work_bytes, cudaStream_t stream);

// ------------------------------------------------------------------ fixed working space
// Drops the cached device address of ccl_reduce_scatter_step_static's array on
// device `dev` (ccl_finalize), so that the next call resolves it again.
void forget_static_scratch(int dev);

// ------------------------------------------------------------------ bounds checks (debug builds)
// The byte ranges a call's kernels may touch.  Debug builds upload them on the
// call's stream before its kernels; release builds do nothing.
struct DbgRange {
    const void *lo;
    size_t bytes;
};
cudaError_t dbg_set_ranges(const std::vector<DbgRange> &ranges, cudaStream_t stream);

// ------------------------------------------------------------------ automatic result checks
// With checks on (CCL_CHECK or ccl_set_check), enqueue the bit comparison of
// nranks outputs of `count` elements on `stream`, adding to the device's
// counter; a no-op otherwise.
cudaError_t auto_check(const void *const *bufs, int nranks, uint64_t count, int elem_size, cudaStream_t stream);

// ------------------------------------------------------------------ settings
// The mode a call runs in: its own argument, or the one CCL_MODE /
// ccl_set_mode_override forces (invalid arguments are returned unchanged).
ccl_mode_t effective_mode(ccl_mode_t requested);
// Bucket size used when a call passes bucket_bytes = 0 (CCL_BUCKET_MB /
// ccl_set_default_bucket_bytes, else CCL_DEFAULT_BUCKET_BYTES).
size_t default_bucket_bytes();
// ccl_allreduce_host's path: CCL_HOST_PATH_STAGED or CCL_HOST_PATH_DIRECT
// (CCL_HOST_PATH / ccl_set_host_path).
int host_path();
// Whether automatic result checks and call tracing are on.
bool check_enabled();
bool trace_enabled();

// ------------------------------------------------------------------ bookkeeping
// (count_launches is declared in fused.h)
// kernels launched so far by the calling thread
unsigned long long thread_launch_count();

// Records one call in the trace ring buffer when tracing is on (CCL_TRACE or
// ccl_set_trace): construct at entry, pass the status through done().  The
// call's device time is taken with two events recorded on `stream` around it
// (not while the stream is being captured into a graph).
class TraceScope {
  public:
    TraceScope(const char *name, int nranks, uint64_t count, int dtype, int op, int mode, cudaStream_t stream);
    ccl_status_t done(ccl_status_t st)
    {
        finish((int)st);
        return st;
    }

  private:
    void finish(int status);
    bool active_;
    cudaStream_t stream_ = nullptr;
    cudaEvent_t ev0_ = nullptr, ev1_ = nullptr;
    ccl_trace_record_t rec_{};
    unsigned long long launches0_ = 0;
    long long t0_ = 0;
};

} // namespace ccl
