// bucketer.cu -- bucket-fused AllReduce that overlaps with the backward pass.
//
// DDP registers a hook per parameter; when the last gradient of a bucket is
// ready the bucket's AllReduce starts asynchronously while the backward pass
// goes on computing earlier layers (Collective Communication, "Layer-wise
// overlap" and "Bucket fusion": buckets are filled in reverse order of use in
// the forward pass, so the first bucket to fill holds the last layers).  Here
// the caller marks each gradient tensor ready with a CUDA event recorded on
// its compute stream; the communication stream is made to wait for it at once,
// and when every tensor a bucket touches is ready, the bucket's fused ring
// reduction is enqueued there.  The bits are those of ccl_bucket_allreduce: the same
// plan, the same segments, only launched bucket by bucket.
#include <algorithm>
#include <mutex>
#include <new>
#include <vector>

#include "../../include/ccl.h"
#include "ccl_internal.h"

struct ccl_bucketer {
    int T = 0, N = 0;
    int dt = 0, op = 0;
    std::vector<void *> tp;                 // [t][r]
    std::vector<ccl::DbgRange> ranges;      // every (tensor, rank) buffer, for debug builds
    ccl::BucketPlan plan;
    std::vector<std::vector<int>> buckets_of; // per tensor: the buckets it touches
    std::vector<int> remaining;             // per bucket: tensors not yet ready
    std::vector<char> ready;                // per tensor
    size_t launched = 0;
    int max_ctas = 0;                       // 0: one CTA per tile
    std::mutex mu;
};

using namespace ccl;

extern "C" {

ccl_status_t ccl_bucketer_create(void *const *ptrs, const size_t *numels, int ntensors, int nranks,
                                 size_t bucket_bytes, ccl_dtype_t dtype, ccl_op_t op, int max_ctas,
                                 ccl_bucketer_t **out)
{
    if (!out || max_ctas < 0 || nranks < 1 || nranks > CCL_MAX_RANKS || (dtype != CCL_FP32 && dtype != CCL_BF16) ||
        (op != CCL_SUM && op != CCL_AVG && op != CCL_MAX && op != CCL_PROD && op != CCL_MIN &&
         op != CCL_AVG_PREMUL) || ntensors < 1 ||
        !ptrs || !numels)
        return CCL_ERR_INVALID_ARG;
    *out = nullptr;
    const size_t es = dtype == CCL_BF16 ? 2 : 4;
    if (bucket_bytes == 0)
        bucket_bytes = default_bucket_bytes();
    const size_t B = bucket_bytes / es;
    if (B == 0)
        return CCL_ERR_INVALID_ARG;
    size_t total = 0;
    for (int t = 0; t < ntensors; ++t) {
        if (numels[t] > SIZE_MAX / es || total + numels[t] < total)
            return CCL_ERR_INVALID_ARG;
        total += numels[t];
    }
    // every (rank, tensor) buffer is written: all must be disjoint
    struct R { uintptr_t lo, hi; };
    std::vector<R> w;
    for (int r = 0; r < nranks; ++r)
        for (int t = 0; t < ntensors; ++t) {
            void *p = ptrs[(size_t)r * ntensors + t];
            if (numels[t] && !p)
                return CCL_ERR_INVALID_ARG;
            if (numels[t])
                w.push_back(R{(uintptr_t)p, (uintptr_t)p + numels[t] * es});
        }
    std::sort(w.begin(), w.end(), [](const R &a, const R &b) { return a.lo < b.lo; });
    for (size_t i = 1; i < w.size(); ++i)
        if (w[i].lo < w[i - 1].hi)
            return CCL_ERR_OVERLAP;

    auto *b = new (std::nothrow) ccl_bucketer;
    if (!b)
        return CCL_ERR_NO_MEMORY;
    b->T = ntensors;
    b->N = nranks;
    b->dt = (int)dtype;
    b->op = (int)op;
    b->max_ctas = max_ctas;
    b->tp.resize((size_t)ntensors * nranks);
    for (int r = 0; r < nranks; ++r)
        for (int t = 0; t < ntensors; ++t)
            b->tp[(size_t)t * nranks + r] = ptrs[(size_t)r * ntensors + t];
    for (int r = 0; r < nranks; ++r)
        for (int t = 0; t < ntensors; ++t)
            b->ranges.push_back(DbgRange{ptrs[(size_t)r * ntensors + t], numels[t] * es});
    build_bucket_plan(numels, ntensors, nranks, B, b->plan);
    const size_t nb = b->plan.segs.size();
    b->buckets_of.assign(ntensors, {});
    for (size_t k = 0; k < nb; ++k)
        for (int t : b->plan.tensors[k])
            b->buckets_of[t].push_back((int)k);
    b->remaining.resize(nb);
    for (size_t k = 0; k < nb; ++k)
        b->remaining[k] = (int)b->plan.tensors[k].size();
    b->ready.assign(ntensors, 0);
    *out = b;
    return CCL_OK;
}

ccl_status_t ccl_bucketer_mark_ready(ccl_bucketer_t *b, int tensor, cudaEvent_t ready, cudaStream_t comm_stream)
{
    if (!b || tensor < 0 || tensor >= b->T)
        return CCL_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(b->mu);
    if (b->ready[tensor])
        return CCL_ERR_INVALID_ARG; // marked twice in one step
    b->ready[tensor] = 1;
    // Everything enqueued on comm_stream from now on waits for this tensor.
    // Enqueued here rather than when its bucket fills, so the event only has
    // to live through this call; with tensors marked in the order they are
    // produced, an earlier wait never delays a later bucket.
    if (ready && cudaStreamWaitEvent(comm_stream, ready, 0) != cudaSuccess)
        return CCL_ERR_CUDA;
    for (int k : b->buckets_of[tensor]) {
        if (--b->remaining[k] != 0)
            continue;
        // the whole bucket is ready (its waits are already on comm_stream)
        const auto &segs = b->plan.segs[k];
        if (dbg_set_ranges(b->ranges, comm_stream) != cudaSuccess)
            return CCL_ERR_CUDA;
        if (launch_bucket_reduce(b->dt, b->op, b->tp.data(), b->T, b->N, segs.data(), segs.size(), comm_stream,
                                 b->max_ctas) != cudaSuccess)
            return CCL_ERR_CUDA;
        ++b->launched;
    }
    return CCL_OK;
}

ccl_status_t ccl_bucketer_reset(ccl_bucketer_t *b)
{
    if (!b)
        return CCL_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(b->mu);
    for (size_t k = 0; k < b->remaining.size(); ++k)
        b->remaining[k] = (int)b->plan.tensors[k].size();
    std::fill(b->ready.begin(), b->ready.end(), 0);
    b->launched = 0;
    return CCL_OK;
}

ccl_status_t ccl_bucketer_status(ccl_bucketer_t *b, size_t *nbuckets, size_t *launched)
{
    if (!b || !nbuckets || !launched)
        return CCL_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(b->mu);
    *nbuckets = b->plan.segs.size();
    *launched = b->launched;
    return CCL_OK;
}

ccl_status_t ccl_bucketer_destroy(ccl_bucketer_t *b)
{
    delete b;
    return CCL_OK;
}

} // extern "C"
