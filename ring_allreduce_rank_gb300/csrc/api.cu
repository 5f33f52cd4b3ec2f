// api.cu -- the exported C ABI (include/ccl.h): argument validation, planning
// (chunk partition, ring steps, bucket segments, all-to-all displacements) and
// dispatch to the kernels.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "../../include/ccl.h"
#include "ccl_internal.h"

namespace ccl {

static std::atomic<unsigned long long> g_launches{0};
// Every kernel of a call is launched from the calling thread, so a per-thread
// count gives a traced call its own launches even while other threads call in.
static thread_local unsigned long long t_launches = 0;

void count_launches(unsigned long long n)
{
    g_launches.fetch_add(n, std::memory_order_relaxed);
    t_launches += n;
}

unsigned long long thread_launch_count() { return t_launches; }

namespace {

// ------------------------------------------------------------------ workspace

struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mu;
std::unordered_map<int, Workspace> g_ws;

ccl_status_t get_workspace(size_t bytes, void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return CCL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace &w = g_ws[dev];
    if (w.bytes < bytes) {
        if (w.ptr)
            cudaFree(w.ptr);
        w.ptr = nullptr;
        w.bytes = 0;
        if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) {
            cudaGetLastError();
            w.ptr = nullptr;
            return CCL_ERR_NO_MEMORY;
        }
        w.bytes = bytes;
    }
    *out = w.ptr;
    return CCL_OK;
}

// ------------------------------------------------------------------ step-mode helpers

// The ring's two phases, step by step, in place on bufs (full K-element buffers).
ccl_status_t ring_steps_allreduce(int dt, int op, void *const *bufs, int nranks, size_t count, cudaStream_t st)
{
    for (int s = 0; s < nranks - 1; ++s)
        if (cudaError_t e = launch_ring_step(dt, op, STEP_RS, s, bufs, nranks, count, st))
            return from_cuda(e);
    if (step_scale(op, nranks))
        if (cudaError_t e = launch_ring_step(dt, op, STEP_SCALE, 0, bufs, nranks, count, st))
            return from_cuda(e);
    for (int s = 0; s < nranks - 1; ++s)
        if (cudaError_t e = launch_ring_step(dt, op, STEP_AG, s, bufs, nranks, count, st))
            return from_cuda(e);
    return CCL_OK;
}

ccl_status_t copy_ranks(const void *const *src, void *const *dst, int nranks, size_t bytes, cudaStream_t st)
{
    std::vector<CopySeg> segs;
    for (int r = 0; r < nranks; ++r)
        if (src[r] != dst[r])
            segs.push_back(CopySeg{static_cast<const char *>(src[r]), static_cast<char *>(dst[r]), bytes, 0});
    return from_cuda(launch_copy_segments(segs.data(), segs.size(), st));
}

#ifdef CCL_DEBUG_BOUNDS
// debug builds: upload the byte ranges this call's kernels may touch
ccl_status_t dbg_call(const std::vector<Range> &a, const std::vector<Range> &b, std::initializer_list<DbgRange> extra,
                      cudaStream_t st)
{
    std::vector<DbgRange> v;
    for (const Range &x : a)
        v.push_back(DbgRange{reinterpret_cast<const void *>(x.lo), (size_t)(x.hi - x.lo)});
    for (const Range &x : b)
        v.push_back(DbgRange{reinterpret_cast<const void *>(x.lo), (size_t)(x.hi - x.lo)});
    for (const DbgRange &x : extra)
        v.push_back(x);
    return from_cuda(dbg_set_ranges(v, st));
}
#define CCL_DBG(...)                                                                                                   \
    do {                                                                                                               \
        ccl_status_t s_ = dbg_call(__VA_ARGS__);                                                                       \
        if (s_ != CCL_OK)                                                                                              \
            return s_;                                                                                                 \
    } while (0)
#else
#define CCL_DBG(...)                                                                                                   \
    do {                                                                                                               \
    } while (0)
#endif

// The device's addresses of page-locked host buffers (cudaHostAlloc,
// cudaHostRegister) on the current device; false if any buffer is other
// memory (pageable, device, managed) or has no such address.
bool device_views(const void *const *send, void *const *recv, int nranks, const void **ds, void **dr)
{
    auto view = [](const void *p, void **out) {
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        *out = a.devicePointer;
        return a.type == cudaMemoryTypeHost && a.devicePointer != nullptr;
    };
    for (int i = 0; i < nranks; ++i) {
        void *v = nullptr;
        if (!view(send[i], &v))
            return false;
        ds[i] = v;
        if (!view(recv[i], &v))
            return false;
        dr[i] = v;
    }
    return true;
}

} // namespace

ccl_status_t check_reduce_scatter(const void *const *send, void *const *recv, int nranks, size_t count,
                                  ccl_dtype_t dtype, ccl_op_t op, std::vector<Range> &w, std::vector<Range> &r)
{
    w.clear();
    r.clear();
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_op(op) || !send || !recv)
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es) || mul_overflows(count, (size_t)nranks))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const Partition part = make_partition(count, nranks);
    for (int i = 0; i < nranks; ++i) {
        // an empty chunk's output may be NULL (K < N leaves chunks empty)
        if (!send[i] || (!recv[i] && part.len((uint32_t)i) > 0))
            return CCL_ERR_INVALID_ARG;
        w.push_back(range_of(recv[i], part.len((uint32_t)i) * es, i));
        r.push_back(range_of(send[i], count * es, i));
    }
    return check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return rd.rank == wr.rank && wr.lo == rd.lo + part.off((uint32_t)rd.rank) * es;
    });
}

} // namespace ccl

using namespace ccl;

// ====================================================================== C ABI

extern "C" {

const char *ccl_status_string(ccl_status_t s)
{
    switch (s) {
    case CCL_OK: return "ok";
    case CCL_ERR_INVALID_ARG: return "invalid argument";
    case CCL_ERR_UNSUPPORTED: return "unsupported";
    case CCL_ERR_OVERLAP: return "buffers overlap";
    case CCL_ERR_CUDA: return "CUDA error";
    case CCL_ERR_NO_MEMORY: return "out of device memory";
    case CCL_ERR_TIMEOUT: return "timeout";
    case CCL_ERR_CHECK_FAILED: return "result check failed";
    }
    return "unknown status";
}

int ccl_version(void) { return 10100; }

unsigned long long ccl_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

ccl_status_t ccl_finalize(void)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return CCL_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    auto it = g_ws.find(dev);
    if (it != g_ws.end()) {
        if (it->second.ptr)
            cudaFree(it->second.ptr);
        g_ws.erase(it);
    }
    forget_static_scratch(dev);
    return CCL_OK;
}

// ------------------------------------------------------------------ planner

ccl_status_t ccl_plan_chunks(size_t count, int nranks, size_t *off, size_t *len)
{
    if (!valid_ranks(nranks) || !off || !len)
        return CCL_ERR_INVALID_ARG;
    const Partition p = make_partition(count, nranks);
    for (int c = 0; c < nranks; ++c) {
        off[c] = (size_t)p.off((uint32_t)c);
        len[c] = (size_t)p.len((uint32_t)c);
    }
    return CCL_OK;
}

ccl_status_t ccl_plan_ring_schedule(int nranks, int32_t *table)
{
    if (!valid_ranks(nranks) || (!table && nranks > 1))
        return CCL_ERR_INVALID_ARG;
    const int steps = nranks - 1;
    for (int phase = 0; phase < 2; ++phase)
        for (int s = 0; s < steps; ++s)
            for (int i = 0; i < nranks; ++i) {
                int32_t *e = table + (((size_t)phase * steps + s) * nranks + i) * 3;
                // ReduceScatter: send (i-s), receive (i-1-s); AllGather: send (i+1-s), receive (i-s)
                e[0] = ring_mod(phase == 0 ? i - s : i + 1 - s, nranks);
                e[1] = ring_mod(phase == 0 ? i - 1 - s : i - s, nranks);
                e[2] = ring_mod(i - 1, nranks);
            }
    return CCL_OK;
}

ccl_status_t ccl_plan_buckets(const size_t *numels, int ntensors, size_t bucket_elems, size_t *starts,
                              size_t max_buckets, size_t *nbuckets)
{
    if (ntensors < 0 || (ntensors > 0 && !numels) || bucket_elems == 0 || !nbuckets)
        return CCL_ERR_INVALID_ARG;
    size_t total = 0;
    for (int t = 0; t < ntensors; ++t) {
        if (total + numels[t] < total)
            return CCL_ERR_INVALID_ARG;
        total += numels[t];
    }
    const size_t nb = (total + bucket_elems - 1) / bucket_elems;
    *nbuckets = nb;
    if (starts) {
        const size_t n = std::min(nb, max_buckets);
        for (size_t b = 0; b < n; ++b)
            starts[b] = b * bucket_elems;
        starts[n] = n == nb ? total : n * bucket_elems;
    }
    return CCL_OK;
}

ccl_status_t ccl_plan_alltoallv(int nranks, const size_t *counts, size_t *sdispl, size_t *rdispl)
{
    if (!valid_ranks(nranks) || !counts || !sdispl || !rdispl)
        return CCL_ERR_INVALID_ARG;
    const size_t N = (size_t)nranks;
    for (size_t i = 0; i < N; ++i) {
        size_t o = 0;
        for (size_t j = 0; j < N; ++j) {
            sdispl[i * N + j] = o;
            o += counts[i * N + j];
        }
    }
    for (size_t j = 0; j < N; ++j) {
        size_t o = 0;
        for (size_t i = 0; i < N; ++i) {
            rdispl[j * N + i] = o;
            o += counts[i * N + j];
        }
    }
    return CCL_OK;
}

ccl_status_t ccl_arena_layout(int nranks, size_t bytes_per_rank, size_t align, size_t *stride, size_t *total)
{
    if (!valid_ranks(nranks) || !stride || !total || align < 256 || (align & (align - 1)) != 0)
        return CCL_ERR_INVALID_ARG;
    if (bytes_per_rank > SIZE_MAX - align)
        return CCL_ERR_INVALID_ARG;
    const size_t s = (bytes_per_rank + align - 1) & ~(align - 1);
    if (mul_overflows(s, (size_t)nranks))
        return CCL_ERR_INVALID_ARG;
    *stride = s;
    *total = s * (size_t)nranks;
    return CCL_OK;
}

// ------------------------------------------------------------------ AllReduce

static ccl_status_t ccl_allreduce_impl(const void *const *send, void *const *recv, int nranks, size_t count, ccl_dtype_t dtype,
                           ccl_op_t op, ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_op(op) || !valid_mode(mode) || !send || !recv)
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const size_t bytes = count * es;
    std::vector<Range> w, r;
    bool in_place = true;
    for (int i = 0; i < nranks; ++i) {
        if (!send[i] || !recv[i])
            return CCL_ERR_INVALID_ARG;
        in_place = in_place && send[i] == recv[i];
        w.push_back(range_of(recv[i], bytes, i));
        r.push_back(range_of(send[i], bytes, i));
    }
    ccl_status_t st = check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return rd.rank == wr.rank && rd.lo == wr.lo;
    });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, r, {}, stream);
    if (nranks == 1 && in_place && !scales(op))
        return CCL_OK;
    if (mode == CCL_MODE_FUSED)
        return from_cuda(launch_fused_reduce((int)dtype, (int)op, send, recv, nranks, count, WRITE_ALL, 0, stream));
    if ((st = copy_ranks(send, recv, nranks, bytes, stream)) != CCL_OK)
        return st;
    return ring_steps_allreduce((int)dtype, (int)op, recv, nranks, count, stream);
}

// ------------------------------------------------------------------ ReduceScatter

static ccl_status_t ccl_reduce_scatter_impl(const void *const *send, void *const *recv, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_mode(mode))
        return CCL_ERR_INVALID_ARG;
    std::vector<Range> w, r;
    ccl_status_t st = check_reduce_scatter(send, recv, nranks, count, dtype, op, w, r);
    if (st != CCL_OK || count == 0)
        return st;
    const size_t es = elem_size(dtype);
    const Partition part = make_partition(count, nranks);
    CCL_DBG(w, r, {}, stream);
    if (mode == CCL_MODE_FUSED)
        return from_cuda(launch_fused_reduce((int)dtype, (int)op, send, recv, nranks, count, WRITE_CHUNK, 0, stream));
    // step mode: the ring's ReduceScatter phase on a workspace copy of the inputs
    void *ws = nullptr;
    if ((st = get_workspace(count * es * (size_t)nranks, &ws)) != CCL_OK)
        return st;
    CCL_DBG(w, r, {DbgRange{ws, count * es * (size_t)nranks}}, stream);
    std::vector<void *> bufs(nranks);
    for (int i = 0; i < nranks; ++i)
        bufs[i] = static_cast<char *>(ws) + (size_t)i * count * es;
    if ((st = copy_ranks(send, bufs.data(), nranks, count * es, stream)) != CCL_OK)
        return st;
    for (int s = 0; s < nranks - 1; ++s)
        if (cudaError_t e = launch_ring_step((int)dtype, (int)op, STEP_RS, s, bufs.data(), nranks, count, stream))
            return from_cuda(e);
    if (step_scale(op, nranks))
        if (cudaError_t e = launch_ring_step((int)dtype, (int)op, STEP_SCALE, 0, bufs.data(), nranks, count, stream))
            return from_cuda(e);
    // the phase leaves chunk c at rank c-1; hand it to rank c
    std::vector<CopySeg> segs;
    for (int c = 0; c < nranks; ++c)
        segs.push_back(CopySeg{static_cast<const char *>(bufs[ring_mod(c - 1, nranks)]) + part.off((uint32_t)c) * es,
                               static_cast<char *>(recv[c]), part.len((uint32_t)c) * es, 0});
    return from_cuda(launch_copy_segments(segs.data(), segs.size(), stream));
}

// ------------------------------------------------------------------ AllGather

static ccl_status_t ccl_allgather_impl(const void *const *send, void *const *recv, int nranks, size_t count, ccl_dtype_t dtype,
                           ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_mode(mode) || !send || !recv)
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const Partition part = make_partition(count, nranks);
    std::vector<Range> w, r;
    for (int i = 0; i < nranks; ++i) {
        // an empty chunk's input may be NULL (K < N leaves chunks empty)
        if (!recv[i] || (!send[i] && part.len((uint32_t)i) > 0))
            return CCL_ERR_INVALID_ARG;
        w.push_back(range_of(recv[i], count * es, i));
        r.push_back(range_of(send[i], part.len((uint32_t)i) * es, i));
    }
    ccl_status_t st = check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return rd.rank == wr.rank && rd.lo == wr.lo + part.off((uint32_t)rd.rank) * es;
    });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, r, {}, stream);
    if (mode == CCL_MODE_FUSED)
        return from_cuda(launch_fanout((int)dtype, send, nranks, recv, nranks, count, stream));
    // step mode: rank i starts with chunk i; ring steps forward the rest
    std::vector<CopySeg> segs;
    for (int i = 0; i < nranks; ++i)
        segs.push_back(CopySeg{static_cast<const char *>(send[i]),
                               static_cast<char *>(recv[i]) + part.off((uint32_t)i) * es,
                               part.len((uint32_t)i) * es, 0});
    if ((st = from_cuda(launch_copy_segments(segs.data(), segs.size(), stream))) != CCL_OK)
        return st;
    for (int s = 0; s < nranks - 1; ++s)
        if (cudaError_t e = launch_ring_step((int)dtype, CCL_SUM, STEP_AG_API, s, recv, nranks, count, stream))
            return from_cuda(e);
    return CCL_OK;
}

// ------------------------------------------------------------------ Broadcast

static ccl_status_t ccl_broadcast_impl(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                           ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_mode(mode) || !send || !recv || root < 0 ||
        root >= nranks || !send[root])
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const size_t bytes = count * es;
    std::vector<Range> w, r;
    for (int i = 0; i < nranks; ++i) {
        if (!recv[i])
            return CCL_ERR_INVALID_ARG;
        w.push_back(range_of(recv[i], bytes, i));
    }
    r.push_back(range_of(send[root], bytes, root));
    ccl_status_t st = check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return wr.rank == root && rd.lo == wr.lo;
    });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, r, {}, stream);
    if (mode == CCL_MODE_FUSED) {
        // in place, root already holds the data: write only the other ranks
        const void *src[1] = {send[root]};
        std::vector<void *> dst;
        for (int i = 0; i < nranks; ++i)
            if (recv[i] != send[root])
                dst.push_back(recv[i]);
        if (dst.empty())
            return CCL_OK;
        return from_cuda(launch_fanout((int)dtype, src, 1, dst.data(), (int)dst.size(), count, stream));
    }
    // step mode: a chain around the ring starting at root
    if (send[root] != recv[root]) {
        CopySeg s{static_cast<const char *>(send[root]), static_cast<char *>(recv[root]), bytes, 0};
        if ((st = from_cuda(launch_copy_segments(&s, 1, stream))) != CCL_OK)
            return st;
    }
    for (int s = 0; s < nranks - 1; ++s) {
        const int from = (root + s) % nranks, to = (root + s + 1) % nranks;
        CopySeg g{static_cast<const char *>(recv[from]), static_cast<char *>(recv[to]), bytes, 0};
        if ((st = from_cuda(launch_copy_segments(&g, 1, stream))) != CCL_OK)
            return st;
    }
    return CCL_OK;
}

// ------------------------------------------------------------------ AllToAll(v)

static ccl_status_t ccl_alltoallv_impl(const void *const *send, void *const *recv, int nranks, const size_t *counts,
                           ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_mode(mode) || !send || !recv || !counts)
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    const size_t N = (size_t)nranks;
    std::vector<size_t> sd(N * N), rd(N * N), stot(N, 0), rtot(N, 0);
    for (size_t i = 0; i < N; ++i)
        for (size_t j = 0; j < N; ++j) {
            const size_t c = counts[i * N + j];
            if (stot[i] + c < stot[i] || rtot[j] + c < rtot[j])
                return CCL_ERR_INVALID_ARG;
            stot[i] += c;
            rtot[j] += c;
        }
    for (size_t i = 0; i < N; ++i)
        if (mul_overflows(stot[i], es) || mul_overflows(rtot[i], es))
            return CCL_ERR_INVALID_ARG;
    ccl_plan_alltoallv(nranks, counts, sd.data(), rd.data());
    std::vector<Range> w, r;
    for (int i = 0; i < nranks; ++i) {
        if ((stot[i] && !send[i]) || (rtot[i] && !recv[i]))
            return CCL_ERR_INVALID_ARG;
        w.push_back(range_of(recv[i], rtot[i] * es, i));
        r.push_back(range_of(send[i], stot[i] * es, i));
    }
    ccl_status_t st = check_overlaps(w, r, [](const Range &, const Range &) { return false; });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, r, {}, stream);
    auto seg = [&](size_t i, size_t j) {
        return CopySeg{static_cast<const char *>(send[i]) + sd[i * N + j] * es,
                       static_cast<char *>(recv[j]) + rd[j * N + i] * es, counts[i * N + j] * es, 0};
    };
    std::vector<CopySeg> segs;
    if (mode == CCL_MODE_FUSED) {
        for (size_t i = 0; i < N; ++i)
            for (size_t j = 0; j < N; ++j)
                segs.push_back(seg(i, j));
        return from_cuda(launch_copy_segments(segs.data(), segs.size(), stream));
    }
    // pairwise schedule: step k, rank i sends its block for rank (i+k) mod N
    for (size_t k = 0; k < N; ++k) {
        segs.clear();
        for (size_t i = 0; i < N; ++i)
            segs.push_back(seg(i, (i + k) % N));
        if ((st = from_cuda(launch_copy_segments(segs.data(), segs.size(), stream))) != CCL_OK)
            return st;
    }
    return CCL_OK;
}

static ccl_status_t ccl_alltoall_impl(const void *const *send, void *const *recv, int nranks, size_t count, ccl_dtype_t dtype,
                          ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_ranks(nranks))
        return CCL_ERR_INVALID_ARG;
    if (mul_overflows(count, (size_t)nranks))
        return CCL_ERR_INVALID_ARG;
    std::vector<size_t> counts((size_t)nranks * nranks, count);
    return ccl_alltoallv_impl(send, recv, nranks, counts.data(), dtype, mode, stream);
}

// ------------------------------------------------------------------ bucket AllReduce

static ccl_status_t ccl_bucket_allreduce_impl(void *const *ptrs, const size_t *numels, int ntensors, int nranks,
                                  size_t bucket_bytes, ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode,
                                  cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_op(op) || !valid_mode(mode) || ntensors < 0 ||
        (ntensors > 0 && (!ptrs || !numels)))
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (bucket_bytes == 0)
        bucket_bytes = default_bucket_bytes();
    const size_t B = bucket_bytes / es;
    if (B == 0)
        return CCL_ERR_INVALID_ARG;
    const size_t T = (size_t)ntensors, N = (size_t)nranks;
    // stream layout: reverse registration order
    std::vector<size_t> pos(T);
    size_t total = 0;
    for (size_t k = T; k-- > 0;) {
        if (mul_overflows(numels[k], es) || total + numels[k] < total)
            return CCL_ERR_INVALID_ARG;
        pos[k] = total;
        total += numels[k];
    }
    if (total == 0)
        return CCL_OK;
    std::vector<Range> w;
    std::vector<void *> tp(T * N); // [t][r]
    for (size_t r = 0; r < N; ++r)
        for (size_t t = 0; t < T; ++t) {
            void *p = ptrs[r * T + t];
            if (numels[t] && !p)
                return CCL_ERR_INVALID_ARG;
            tp[t * N + r] = p;
            w.push_back(range_of(p, numels[t] * es, (int)r));
        }
    ccl_status_t st = check_overlaps(w, {}, [](const Range &, const Range &) { return false; });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, {}, {}, stream);
    // tensors in stream order
    std::vector<size_t> order;
    for (size_t k = T; k-- > 0;)
        if (numels[k])
            order.push_back(k);

    if (mode == CCL_MODE_FUSED) {
        // every (bucket, chunk) stream range cut at tensor boundaries, one launch
        BucketPlan plan;
        build_bucket_plan(numels, ntensors, nranks, B, plan);
        std::vector<RedSeg> segs;
        for (const auto &bs : plan.segs)
            segs.insert(segs.end(), bs.begin(), bs.end());
        return from_cuda(launch_bucket_reduce((int)dtype, (int)op, tp.data(), ntensors, nranks, segs.data(),
                                              segs.size(), stream));
    }
    // step mode: explicit pack -> ring steps -> unpack per bucket, through a workspace
    void *ws = nullptr;
    if ((st = get_workspace(std::min(B, total) * es * N, &ws)) != CCL_OK)
        return st;
    CCL_DBG(w, {}, {DbgRange{ws, std::min(B, total) * es * N}}, stream);
    std::vector<void *> bufs(N);
    for (size_t r = 0; r < N; ++r)
        bufs[r] = static_cast<char *>(ws) + r * std::min(B, total) * es;
    size_t oi = 0;
    for (size_t b0 = 0; b0 < total; b0 += B) {
        const size_t blen = std::min(B, total - b0);
        std::vector<CopySeg> pack, unpack;
        size_t lo = b0;
        size_t oj = oi;
        while (lo < b0 + blen) {
            while (pos[order[oj]] + numels[order[oj]] <= lo)
                ++oj;
            const size_t t = order[oj];
            const size_t e = std::min(b0 + blen, pos[t] + numels[t]);
            for (size_t r = 0; r < N; ++r) {
                char *tpr = static_cast<char *>(tp[t * N + r]) + (lo - pos[t]) * es;
                char *bpr = static_cast<char *>(bufs[r]) + (lo - b0) * es;
                pack.push_back(CopySeg{tpr, bpr, (e - lo) * es, 0});
                unpack.push_back(CopySeg{bpr, tpr, (e - lo) * es, 0});
            }
            lo = e;
        }
        oi = oj;
        if ((st = from_cuda(launch_copy_segments(pack.data(), pack.size(), stream))) != CCL_OK)
            return st;
        if ((st = ring_steps_allreduce((int)dtype, (int)op, bufs.data(), nranks, blen, stream)) != CCL_OK)
            return st;
        if ((st = from_cuda(launch_copy_segments(unpack.data(), unpack.size(), stream))) != CCL_OK)
            return st;
    }
    return CCL_OK;
}

// ------------------------------------------------------------------ Reduce / Gather / Scatter

static ccl_status_t ccl_reduce_impl(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                        ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_op(op) || !valid_mode(mode) || !send || !recv ||
        root < 0 || root >= nranks)
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es) || mul_overflows(count, (size_t)nranks))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const size_t bytes = count * es;
    if (!recv[root])
        return CCL_ERR_INVALID_ARG;
    std::vector<Range> w{range_of(recv[root], bytes, root)}, r;
    for (int i = 0; i < nranks; ++i) {
        if (!send[i])
            return CCL_ERR_INVALID_ARG;
        r.push_back(range_of(send[i], bytes, i));
    }
    ccl_status_t st = check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return rd.rank == wr.rank && rd.lo == wr.lo;
    });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, r, {}, stream);
    if (mode == CCL_MODE_FUSED)
        return from_cuda(launch_fused_reduce((int)dtype, (int)op, send, recv, nranks, count, WRITE_ROOT, root,
                                             stream));
    // step mode: the ring's ReduceScatter phase on a workspace copy, then every
    // finished chunk c is brought from rank c-1 to the root
    void *ws = nullptr;
    if ((st = get_workspace(bytes * (size_t)nranks, &ws)) != CCL_OK)
        return st;
    CCL_DBG(w, r, {DbgRange{ws, bytes * (size_t)nranks}}, stream);
    std::vector<void *> bufs(nranks);
    for (int i = 0; i < nranks; ++i)
        bufs[i] = static_cast<char *>(ws) + (size_t)i * bytes;
    if ((st = copy_ranks(send, bufs.data(), nranks, bytes, stream)) != CCL_OK)
        return st;
    for (int s = 0; s < nranks - 1; ++s)
        if (cudaError_t e = launch_ring_step((int)dtype, (int)op, STEP_RS, s, bufs.data(), nranks, count, stream))
            return from_cuda(e);
    if (step_scale(op, nranks))
        if (cudaError_t e = launch_ring_step((int)dtype, (int)op, STEP_SCALE, 0, bufs.data(), nranks, count, stream))
            return from_cuda(e);
    const Partition part = make_partition(count, nranks);
    std::vector<CopySeg> segs;
    for (int c = 0; c < nranks; ++c)
        segs.push_back(CopySeg{static_cast<const char *>(bufs[ring_mod(c - 1, nranks)]) + part.off((uint32_t)c) * es,
                               static_cast<char *>(recv[root]) + part.off((uint32_t)c) * es,
                               part.len((uint32_t)c) * es, 0});
    return from_cuda(launch_copy_segments(segs.data(), segs.size(), stream));
}

static ccl_status_t ccl_gather_impl(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                        ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_mode(mode) || !send || !recv || root < 0 ||
        root >= nranks || !recv[root])
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const Partition part = make_partition(count, nranks);
    std::vector<Range> w{range_of(recv[root], count * es, root)}, r;
    for (int i = 0; i < nranks; ++i) {
        if (!send[i] && part.len((uint32_t)i) > 0)
            return CCL_ERR_INVALID_ARG;
        r.push_back(range_of(send[i], part.len((uint32_t)i) * es, i));
    }
    ccl_status_t st = check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return rd.lo == wr.lo + part.off((uint32_t)rd.rank) * es;
    });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, r, {}, stream);
    if (mode == CCL_MODE_FUSED) {
        void *dst[1] = {recv[root]};
        return from_cuda(launch_fanout((int)dtype, send, nranks, dst, 1, count, stream));
    }
    // step mode: one rank's slice per launch, in rank order
    for (int i = 0; i < nranks; ++i) {
        CopySeg g{static_cast<const char *>(send[i]), static_cast<char *>(recv[root]) + part.off((uint32_t)i) * es,
                  part.len((uint32_t)i) * es, 0};
        if ((st = from_cuda(launch_copy_segments(&g, 1, stream))) != CCL_OK)
            return st;
    }
    return CCL_OK;
}

static ccl_status_t ccl_scatter_impl(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                         ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_mode(mode) || !send || !recv || root < 0 ||
        root >= nranks || !send[root])
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const Partition part = make_partition(count, nranks);
    std::vector<Range> w, r{range_of(send[root], count * es, root)};
    for (int i = 0; i < nranks; ++i) {
        if (!recv[i] && part.len((uint32_t)i) > 0)
            return CCL_ERR_INVALID_ARG;
        w.push_back(range_of(recv[i], part.len((uint32_t)i) * es, i));
    }
    ccl_status_t st = check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return wr.lo == rd.lo + part.off((uint32_t)wr.rank) * es;
    });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, r, {}, stream);
    std::vector<CopySeg> segs;
    for (int i = 0; i < nranks; ++i)
        segs.push_back(CopySeg{static_cast<const char *>(send[root]) + part.off((uint32_t)i) * es,
                               static_cast<char *>(recv[i]), part.len((uint32_t)i) * es, 0});
    if (mode == CCL_MODE_FUSED)
        return from_cuda(launch_copy_segments(segs.data(), segs.size(), stream));
    for (const CopySeg &g : segs)  // step mode: one destination per launch
        if ((st = from_cuda(launch_copy_segments(&g, 1, stream))) != CCL_OK)
            return st;
    return CCL_OK;
}

// ------------------------------------------------------------------ other schedules' orders

static ccl_status_t ccl_allreduce_algo_impl(const void *const *send, void *const *recv, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, ccl_algo_t algo, int group_size,
                                cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_op(op) || !send || !recv || algo < CCL_ALGO_RING ||
        algo > CCL_ALGO_HIERARCHICAL)
        return CCL_ERR_INVALID_ARG;
    if (algo == CCL_ALGO_HIERARCHICAL && (group_size < 1 || nranks % group_size != 0))
        return CCL_ERR_INVALID_ARG;
    if (op == CCL_AVG_PREMUL && algo != CCL_ALGO_RING)
        return CCL_ERR_UNSUPPORTED; // the other orders divide once, at the end
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const size_t bytes = count * es;
    std::vector<Range> w, r;
    for (int i = 0; i < nranks; ++i) {
        if (!send[i] || !recv[i])
            return CCL_ERR_INVALID_ARG;
        w.push_back(range_of(recv[i], bytes, i));
        r.push_back(range_of(send[i], bytes, i));
    }
    ccl_status_t st = check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return rd.rank == wr.rank && rd.lo == wr.lo;
    });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, r, {}, stream);
    if (algo == CCL_ALGO_RING)
        return from_cuda(launch_fused_reduce((int)dtype, (int)op, send, recv, nranks, count, WRITE_ALL, 0, stream));
    return from_cuda(launch_order_allreduce((int)dtype, (int)op, (int)algo, group_size, send, recv, nranks, count,
                                           stream));
}

// ------------------------------------------------------------------ compressed AllReduce

ccl_status_t ccl_plan_compressed_bytes(size_t count, ccl_compressor_t comp, int block, size_t *bytes)
{
    if (!bytes || (comp != CCL_COMP_INT8_BLOCK && comp != CCL_COMP_THRESHOLD) ||
        (comp == CCL_COMP_INT8_BLOCK && block < 1))
        return CCL_ERR_INVALID_ARG;
    if (comp == CCL_COMP_THRESHOLD)
        *bytes = (count + 7) / 8; // one bit per element
    else
        *bytes = count + 4 * ((count + (size_t)block - 1) / (size_t)block); // int8 codes + fp32 scales
    return CCL_OK;
}

static ccl_status_t ccl_allreduce_compressed_impl(void *const *grads, float *const *residuals, int nranks, size_t count,
                                      ccl_dtype_t dtype, ccl_op_t op, ccl_compressor_t comp, int block,
                                      float threshold, cudaStream_t stream)
{
    if (op == CCL_AVG_PREMUL)
        return CCL_ERR_UNSUPPORTED; // the compressed AllReduce divides once, at the end
    if (nranks < 1 || nranks > 16 || !valid_dtype(dtype) || (op != CCL_SUM && op != CCL_AVG) || !grads ||
        !residuals || (comp != CCL_COMP_INT8_BLOCK && comp != CCL_COMP_THRESHOLD) ||
        (comp == CCL_COMP_INT8_BLOCK && block != 64 && block != 128))
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, 4))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    std::vector<Range> w;
    for (int i = 0; i < nranks; ++i) {
        if (!grads[i] || !residuals[i])
            return CCL_ERR_INVALID_ARG;
        w.push_back(range_of(grads[i], count * es, i));
        w.push_back(range_of(residuals[i], count * 4, i));
    }
    ccl_status_t st = check_overlaps(w, {}, [](const Range &, const Range &) { return false; });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, {}, {}, stream);
    return from_cuda(launch_compressed_allreduce((int)dtype, op == CCL_AVG, (int)comp, block, threshold, grads,
                                                 residuals, nranks, count, nullptr, stream));
}

ccl_status_t ccl_plan_topk_bytes(size_t count, size_t k, size_t *bytes)
{
    if (!bytes)
        return CCL_ERR_INVALID_ARG;
    const size_t kept = k < count ? k : count;
    if (mul_overflows(kept, 8))
        return CCL_ERR_INVALID_ARG;
    *bytes = kept * 8; // an fp32 value and an int32 index per kept element
    return CCL_OK;
}

ccl_status_t ccl_plan_topk_work_bytes(int nranks, size_t *bytes)
{
    if (nranks < 1 || nranks > kTopkMaxRanks || !bytes)
        return CCL_ERR_INVALID_ARG;
    *bytes = topk_work_bytes(nranks);
    return CCL_OK;
}

ccl_status_t ccl_plan_topk_sample(size_t count, size_t k, uint32_t *every)
{
    if (!every || count >= ((size_t)1 << 32))
        return CCL_ERR_INVALID_ARG;
    *every = topk_sample_every(count, k);
    return CCL_OK;
}

static ccl_status_t ccl_allreduce_topk_impl(void *const *grads, float *const *residuals, int nranks, size_t count,
                                            ccl_dtype_t dtype, ccl_op_t op, size_t k, void *work, size_t work_bytes,
                                            cudaStream_t stream)
{
    if (op == CCL_AVG_PREMUL)
        return CCL_ERR_UNSUPPORTED; // the compressed AllReduce divides once, at the end
    if (nranks < 1 || nranks > kTopkMaxRanks || !valid_dtype(dtype) || (op != CCL_SUM && op != CCL_AVG) || !grads ||
        !residuals)
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, 4) || (uint64_t)count > 0xffffffffull) // 32-bit histogram bins
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    const size_t wb = topk_work_bytes(nranks);
    if (!work || work_bytes < wb || (uintptr_t)work % 16 != 0)
        return CCL_ERR_INVALID_ARG;
    std::vector<Range> w;
    for (int i = 0; i < nranks; ++i) {
        if (!grads[i] || !residuals[i])
            return CCL_ERR_INVALID_ARG;
        w.push_back(range_of(grads[i], count * es, i));
        w.push_back(range_of(residuals[i], count * 4, i));
    }
    w.push_back(range_of(work, wb, nranks));
    ccl_status_t st = check_overlaps(w, {}, [](const Range &, const Range &) { return false; });
    if (st != CCL_OK)
        return st;
    CCL_DBG(w, {}, {}, stream);
    const uint32_t *tau = nullptr;
    if (cudaError_t e = launch_topk_select((int)dtype, grads, residuals, nranks, count, k, work, &tau, stream))
        return from_cuda(e);
    return from_cuda(launch_compressed_allreduce((int)dtype, op == CCL_AVG, COMP_TOPK, 0, 0.0f, grads, residuals,
                                                 nranks, count, tau, stream));
}

// ------------------------------------------------------------------ host-buffer AllReduce

ccl_status_t ccl_plan_host_slices(size_t count, int nranks, ccl_dtype_t dtype, size_t work_bytes, size_t *off,
                                  size_t *len, size_t max_slices, size_t *nslices)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !nslices)
        return CCL_ERR_INVALID_ARG;
    const uint64_t L = host_stage_elems(nranks, elem_size(dtype), work_bytes);
    if (count > 0 && L == 0)
        return CCL_ERR_INVALID_ARG;
    std::vector<HostSlice> sl;
    plan_host_slices(count, L, sl);
    *nslices = sl.size();
    if (off && len)
        for (size_t k = 0; k < sl.size() && k < max_slices; ++k) {
            off[k] = sl[k].off;
            len[k] = sl[k].len;
        }
    return CCL_OK;
}

static ccl_status_t ccl_allreduce_host_impl(const void *const *send, void *const *recv, int nranks, size_t count,
                                            ccl_dtype_t dtype, ccl_op_t op, void *work, size_t work_bytes,
                                            cudaStream_t stream)
{
    if (!valid_ranks(nranks) || !valid_dtype(dtype) || !valid_op(op) || !send || !recv)
        return CCL_ERR_INVALID_ARG;
    const size_t es = elem_size(dtype);
    if (mul_overflows(count, es))
        return CCL_ERR_INVALID_ARG;
    if (count == 0)
        return CCL_OK;
    if (!work || (uintptr_t)work % 16 != 0 || host_stage_elems(nranks, es, work_bytes) == 0)
        return CCL_ERR_INVALID_ARG;
    const size_t bytes = count * es;
    std::vector<Range> w, r;
    bool in_place = true;
    for (int i = 0; i < nranks; ++i) {
        if (!send[i] || !recv[i])
            return CCL_ERR_INVALID_ARG;
        in_place = in_place && send[i] == recv[i];
        w.push_back(range_of(recv[i], bytes, i));
        r.push_back(range_of(send[i], bytes, i));
    }
    w.push_back(range_of(work, work_bytes, -1));
    ccl_status_t st = check_overlaps(w, r, [&](const Range &rd, const Range &wr) {
        return rd.rank == wr.rank && rd.lo == wr.lo;
    });
    if (st != CCL_OK)
        return st;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess)
        return CCL_ERR_CUDA;
    if (cap != cudaStreamCaptureStatusNone)
        return CCL_ERR_UNSUPPORTED;
    if (nranks == 1 && in_place && !scales(op))
        return CCL_OK;
    // On request, page-locked host buffers that the device can address: the
    // fused kernel reads and writes them in place over the host link, both
    // directions at once, with no staging memory.  Other memory is staged.
    std::vector<const void *> ds(nranks);
    std::vector<void *> dr(nranks);
    if (host_path() == CCL_HOST_PATH_DIRECT && device_views(send, recv, nranks, ds.data(), dr.data())) {
#ifdef CCL_DEBUG_BOUNDS
        std::vector<Range> dw, drd; // the kernel touches the device's addresses of the buffers
        for (int i = 0; i < nranks; ++i) {
            dw.push_back(range_of(dr[i], bytes, i));
            drd.push_back(range_of(ds[i], bytes, i));
        }
        CCL_DBG(dw, drd, {}, stream);
#endif
        return from_cuda(launch_fused_reduce((int)dtype, (int)op, ds.data(), dr.data(), nranks, count, WRITE_ALL, 0,
                                             stream));
    }
    CCL_DBG(w, r, {}, stream);
    return from_cuda(run_host_allreduce((int)dtype, (int)op, send, recv, nranks, count, work, work_bytes, stream));
}

// ------------------------------------------------------------------ traced entry points

// after a successful call whose outputs must be identical on every rank: the
// automatic result check (a no-op unless checks are on)
static ccl_status_t then_check(ccl_status_t st, const void *const *outs, int nranks, size_t count,
                               ccl_dtype_t dtype, cudaStream_t stream)
{
    if (st != CCL_OK)
        return st;
    return from_cuda(auto_check(outs, nranks, count, (int)elem_size(dtype), stream));
}

ccl_status_t ccl_allreduce(const void *const *send, void *const *recv, int nranks, size_t count, ccl_dtype_t dtype,
                           ccl_op_t op, ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("allreduce", nranks, count, (int)dtype, (int)op, (int)mode, stream);
    return tr.done(then_check(ccl_allreduce_impl(send, recv, nranks, count, dtype, op, mode, stream), recv, nranks,
                              count, dtype, stream));
}

ccl_status_t ccl_allreduce_host(const void *const *send, void *const *recv, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, void *work, size_t work_bytes,
                                cudaStream_t stream)
{
    TraceScope tr("allreduce_host", nranks, count, (int)dtype, (int)op, 0, stream);
    return tr.done(ccl_allreduce_host_impl(send, recv, nranks, count, dtype, op, work, work_bytes, stream));
}

ccl_status_t ccl_reduce_scatter(const void *const *send, void *const *recv, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("reduce_scatter", nranks, count, (int)dtype, (int)op, (int)mode, stream);
    return tr.done(ccl_reduce_scatter_impl(send, recv, nranks, count, dtype, op, mode, stream));
}

ccl_status_t ccl_allgather(const void *const *send, void *const *recv, int nranks, size_t count, ccl_dtype_t dtype,
                           ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("allgather", nranks, count, (int)dtype, -1, (int)mode, stream);
    return tr.done(then_check(ccl_allgather_impl(send, recv, nranks, count, dtype, mode, stream), recv, nranks, count,
                              dtype, stream));
}

ccl_status_t ccl_broadcast(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                           ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("broadcast", nranks, count, (int)dtype, -1, (int)mode, stream);
    return tr.done(then_check(ccl_broadcast_impl(send, recv, nranks, root, count, dtype, mode, stream), recv, nranks,
                              count, dtype, stream));
}

ccl_status_t ccl_alltoallv(const void *const *send, void *const *recv, int nranks, const size_t *counts,
                           ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("alltoallv", nranks, 0, (int)dtype, -1, (int)mode, stream);
    return tr.done(ccl_alltoallv_impl(send, recv, nranks, counts, dtype, mode, stream));
}

ccl_status_t ccl_alltoall(const void *const *send, void *const *recv, int nranks, size_t count, ccl_dtype_t dtype,
                          ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("alltoall", nranks, count, (int)dtype, -1, (int)mode, stream);
    return tr.done(ccl_alltoall_impl(send, recv, nranks, count, dtype, mode, stream));
}

ccl_status_t ccl_bucket_allreduce(void *const *ptrs, const size_t *numels, int ntensors, int nranks,
                                  size_t bucket_bytes, ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode,
                                  cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("bucket_allreduce", nranks, (size_t)ntensors, (int)dtype, (int)op, (int)mode, stream);
    return tr.done(ccl_bucket_allreduce_impl(ptrs, numels, ntensors, nranks, bucket_bytes, dtype, op, mode, stream));
}

ccl_status_t ccl_reduce(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                        ccl_dtype_t dtype, ccl_op_t op, ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("reduce", nranks, count, (int)dtype, (int)op, (int)mode, stream);
    return tr.done(ccl_reduce_impl(send, recv, nranks, root, count, dtype, op, mode, stream));
}

ccl_status_t ccl_gather(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                        ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("gather", nranks, count, (int)dtype, -1, (int)mode, stream);
    return tr.done(ccl_gather_impl(send, recv, nranks, root, count, dtype, mode, stream));
}

ccl_status_t ccl_scatter(const void *const *send, void *const *recv, int nranks, int root, size_t count,
                         ccl_dtype_t dtype, ccl_mode_t mode, cudaStream_t stream)
{
    mode = effective_mode(mode);
    TraceScope tr("scatter", nranks, count, (int)dtype, -1, (int)mode, stream);
    return tr.done(ccl_scatter_impl(send, recv, nranks, root, count, dtype, mode, stream));
}

ccl_status_t ccl_allreduce_algo(const void *const *send, void *const *recv, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, ccl_algo_t algo, int group_size,
                                cudaStream_t stream)
{
    TraceScope tr("allreduce_algo", nranks, count, (int)dtype, (int)op, (int)algo, stream);
    return tr.done(then_check(ccl_allreduce_algo_impl(send, recv, nranks, count, dtype, op, algo, group_size, stream),
                              recv, nranks, count, dtype, stream));
}

ccl_status_t ccl_allreduce_compressed(void *const *grads, float *const *residuals, int nranks, size_t count,
                                      ccl_dtype_t dtype, ccl_op_t op, ccl_compressor_t comp, int block,
                                      float threshold, cudaStream_t stream)
{
    TraceScope tr("allreduce_compressed", nranks, count, (int)dtype, (int)op, (int)comp, stream);
    return tr.done(then_check(ccl_allreduce_compressed_impl(grads, residuals, nranks, count, dtype, op, comp, block,
                                                            threshold, stream),
                              grads, nranks, count, dtype, stream));
}

ccl_status_t ccl_allreduce_topk(void *const *grads, float *const *residuals, int nranks, size_t count,
                                ccl_dtype_t dtype, ccl_op_t op, size_t k, void *work, size_t work_bytes,
                                cudaStream_t stream)
{
    TraceScope tr("allreduce_topk", nranks, count, (int)dtype, (int)op, (int)CCL_COMP_TOPK, stream);
    return tr.done(then_check(ccl_allreduce_topk_impl(grads, residuals, nranks, count, dtype, op, k, work,
                                                      work_bytes, stream),
                              grads, nranks, count, dtype, stream));
}

} // extern "C"
