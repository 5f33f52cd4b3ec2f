// ccl_internal.h -- host-side declarations shared by the library's translation
// units: kernel parameter blocks and launchers.  Not part of the public ABI.
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/ccl.h"
#include "ccl_device.cuh"

namespace ccl {

constexpr int kSmallRanks = 16;
constexpr int kMaxRanks = 1024;

// ------------------------------------------------------------------ fused reduce
template <int MAXR> struct FusedParams {
    const void *send[MAXR];
    void *recv[MAXR];
    Partition part;
    int nranks;
    int write_mode;  // WRITE_CHUNK, WRITE_ALL or WRITE_ROOT
    int root;        // WRITE_ROOT: the one rank that receives the result
    int vec_aligned; // every pointer is 16-byte aligned
    uint32_t tiles;  // tiles per chunk (gridDim.x)
    float n_f;       // (float)nranks, the AVG divisor
};

enum WriteMode {
    WRITE_CHUNK = 0, // ReduceScatter: chunk c goes to recv[c], chunk-local
    WRITE_ALL = 1,   // AllReduce: every rank receives the whole result
    WRITE_ROOT = 2   // Reduce: only recv[root] receives the whole result
};

// Launch the one-pass ring-order reduction (AllReduce, ReduceScatter or Reduce).
cudaError_t launch_fused_reduce(int dt, int op, const void *const *send, void *const *recv, int nranks,
                                uint64_t count, int write_mode, int root, cudaStream_t stream);

// ------------------------------------------------------------------ step mode
enum StepKind {
    STEP_RS = 0,     // rank i: chunk (i-1-s) += rank (i-1)'s copy
    STEP_AG = 1,     // rank i: chunk (i-s) = rank (i-1)'s copy (after the RS phase)
    STEP_AG_API = 2, // rank i: chunk (i-1-s) = rank (i-1)'s copy (AllGather from chunk i at rank i)
    STEP_SCALE = 3   // rank i: chunk (i+1) /= N (AVG, at the holder)
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
};

cudaError_t launch_ring_step(int dt, int op, int kind, int s, void *const *bufs, int nranks, uint64_t count,
                             cudaStream_t stream);

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
enum Compressor { COMP_INT8_BLOCK = 0, COMP_THRESHOLD = 1 };

// Error-feedback compression of every rank's gradient, ring-order fp32
// AllReduce of the transmitted values, one round to the gradients' type.
cudaError_t launch_compressed_allreduce(int dt, bool avg, int comp, int block, float threshold,
                                        void *const *grads, float *const *res, int nranks, uint64_t count,
                                        cudaStream_t stream);

// ------------------------------------------------------------------ bookkeeping
void count_launches(unsigned long long n);

// Records one call in the trace ring buffer when tracing is on (CCL_TRACE or
// ccl_set_trace): construct at entry, pass the status through done().
class TraceScope {
  public:
    TraceScope(const char *name, int nranks, uint64_t count, int dtype, int op, int mode);
    ccl_status_t done(ccl_status_t st)
    {
        finish((int)st);
        return st;
    }

  private:
    void finish(int status);
    bool active_;
    ccl_trace_record_t rec_{};
    unsigned long long launches0_ = 0;
    long long t0_ = 0;
};

} // namespace ccl
