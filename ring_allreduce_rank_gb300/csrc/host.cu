// host.cu -- AllReduce of rank buffers that live in host memory.
//
// With the ranks' buffers in host memory every call has to carry each input
// over the host link, reduce, and carry each result back.  The link is far
// slower than HBM (Collective Communication, Table 1: the GPU<->CPU row of
// the alpha-beta parameters), so the two copies set the time; issued one after
// the other they add up, while the link can carry both directions at once.
// The vector is therefore cut into slices that flow through a small ring of
// device stages: the copy-in of slice k+1 runs while slice k is reduced and
// slice k-1 is copied out -- the pipelining NCCL applies to its channels
// (Collective Communication, section on NCCL).  Slices start small, grow to
// the stage size and shrink again at the end, so the first copy-in and the
// last copy-out, which nothing overlaps, are short.
//
// Each slice is reduced with the chunk rotation of the whole vector: element
// e of chunk c (of the count-element partition) is folded starting at rank c,
// exactly as ccl_allreduce folds it, so the result has the same bits.
#include <mutex>
#include <unordered_map>
#include <vector>

#include "ccl_internal.h"

namespace ccl {

namespace {

struct HostPipe {
    size_t max_pitch = 0; // largest row pitch a 2D copy accepts on this device
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, h2d_end = nullptr, d2h_end = nullptr;
    cudaEvent_t in[kHostStages] = {}, red[kHostStages] = {}, out[kHostStages] = {};
};

std::mutex g_pipe_mu; // held for a whole call: the streams and events are shared
std::unordered_map<int, HostPipe> g_pipe;

// Releases whatever make_pipe created (null handles are skipped).
void destroy_pipe(HostPipe &p)
{
    for (cudaStream_t *st : {&p.h2d, &p.d2h})
        if (*st) {
            cudaStreamDestroy(*st);
            *st = nullptr;
        }
    cudaEvent_t *evs[] = {&p.start, &p.h2d_end, &p.d2h_end};
    for (cudaEvent_t *ev : evs)
        if (*ev) {
            cudaEventDestroy(*ev);
            *ev = nullptr;
        }
    for (int s = 0; s < kHostStages; ++s)
        for (cudaEvent_t *ev : {&p.in[s], &p.red[s], &p.out[s]})
            if (*ev) {
                cudaEventDestroy(*ev);
                *ev = nullptr;
            }
}

cudaError_t make_pipe(int dev, HostPipe &p)
{
    int pitch = 0;
    cudaError_t e = cudaDeviceGetAttribute(&pitch, cudaDevAttrMaxPitch, dev);
    p.max_pitch = pitch > 0 ? (size_t)pitch : 0;
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking);
    cudaEvent_t *evs[] = {&p.start, &p.h2d_end, &p.d2h_end};
    for (cudaEvent_t *ev : evs)
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    for (int s = 0; s < kHostStages && e == cudaSuccess; ++s) {
        e = cudaEventCreateWithFlags(&p.in[s], cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&p.red[s], cudaEventDisableTiming);
        if (e == cudaSuccess)
            e = cudaEventCreateWithFlags(&p.out[s], cudaEventDisableTiming);
    }
    return e;
}

// Byte stride between consecutive ranks' buffers when they are equally spaced
// rows that do not overlap (rank r at p[0] + r * stride, stride >= row_bytes,
// within the 2D copy's pitch limit); 0 otherwise.
size_t row_stride(const void *const *p, int nranks, size_t row_bytes, size_t max_pitch)
{
    if (nranks < 2)
        return row_bytes <= max_pitch ? row_bytes : 0;
    const uintptr_t b = (uintptr_t)p[0], d = (uintptr_t)p[1] - b;
    if ((uintptr_t)p[1] < b || d < row_bytes || d > max_pitch)
        return 0;
    for (int r = 2; r < nranks; ++r)
        if ((uintptr_t)p[r] != b + (uintptr_t)r * d)
            return 0;
    return (size_t)d;
}

// Segments of the slice [lo, lo + n) under the count-element partition: one
// per chunk the slice touches, offsets relative to the slice.
void slice_segments(const Partition &part, int nranks, uint64_t lo, uint64_t n, std::vector<RedSeg> &segs)
{
    segs.clear();
    const uint64_t hi = lo + n;
    const uint64_t big = (uint64_t)part.rem * (part.q + 1); // elements in the longer chunks
    uint32_t c = lo < big ? (uint32_t)(lo / (part.q + 1)) : part.rem + (uint32_t)((lo - big) / part.q);
    for (; c < (uint32_t)nranks; ++c) {
        const uint64_t a = part.off(c), b = a + part.len(c);
        if (a >= hi)
            break;
        const uint64_t s = a > lo ? a : lo, t = b < hi ? b : hi;
        if (t > s)
            segs.push_back(RedSeg{0u, c, s - lo, t - s, 0});
    }
}

} // namespace

uint64_t host_stage_elems(int nranks, size_t elem_size, size_t work_bytes)
{
    const uint64_t per = work_bytes / ((uint64_t)kHostStages * (uint64_t)nranks * elem_size);
    return per / kHostSliceUnit * kHostSliceUnit;
}

void plan_host_slices(uint64_t count, uint64_t stage_elems, std::vector<HostSlice> &slices)
{
    slices.clear();
    if (count == 0 || stage_elems == 0)
        return;
    uint64_t first = stage_elems / 16 / kHostSliceUnit * kHostSliceUnit;
    if (first < kHostSliceUnit)
        first = kHostSliceUnit;
    // Head slices grow from `first` to the stage size; tail slices mirror
    // them from the end.  Every slice starts on a multiple of the unit.
    std::vector<HostSlice> tail;
    uint64_t lo = 0, hi = count, L = first;
    while (lo < hi) {
        const uint64_t a = L < hi - lo ? L : hi - lo;
        slices.push_back(HostSlice{lo, a});
        lo += a;
        if (lo >= hi)
            break;
        // the tail slice ends at hi and starts on a unit boundary at most L before it
        uint64_t start = hi > L ? (hi - L + kHostSliceUnit - 1) / kHostSliceUnit * kHostSliceUnit : 0;
        if (start < lo)
            start = lo;
        tail.push_back(HostSlice{start, hi - start});
        hi = start;
        if (L < stage_elems)
            L = 2 * L < stage_elems ? 2 * L : stage_elems;
    }
    for (size_t k = tail.size(); k-- > 0;)
        if (tail[k].len)
            slices.push_back(tail[k]);
}

cudaError_t run_host_allreduce(int dt, int op, const void *const *send, void *const *recv, int nranks,
                               uint64_t count, void *work, size_t work_bytes, cudaStream_t stream)
{
    const size_t es = dt == DT_BF16 ? 2 : 4;
    const uint64_t L = host_stage_elems(nranks, es, work_bytes);
    std::vector<HostSlice> slices;
    plan_host_slices(count, L, slices);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_pipe_mu);
    auto it = g_pipe.find(dev);
    if (it == g_pipe.end()) {
        HostPipe p;
        if ((e = make_pipe(dev, p)) != cudaSuccess) {
            destroy_pipe(p); // nothing half-built is kept or leaked; the next call tries again
            return e;
        }
        it = g_pipe.emplace(dev, p).first;
    }
    HostPipe &P = it->second;
    Partition part;
    part.q = count / (uint64_t)nranks;
    part.rem = (uint32_t)(count % (uint64_t)nranks);
    // Rank buffers laid out as equally spaced rows of one allocation move with
    // one 2D copy per slice and direction instead of one copy per rank: each
    // copy costs microseconds to start, and a call has hundreds of them.
    // Equal spacing does not prove one allocation (separate allocations can
    // sit at equal distances), and a 2D copy cannot span two: the runtime then
    // refuses it when it is enqueued.  So the first refusal switches that
    // direction to per-rank copies for the rest of the call.
    const size_t stage_bytes = (size_t)L * es;
    const bool stage_ok = stage_bytes <= P.max_pitch;
    const size_t s_pitch = stage_ok ? row_stride(send, nranks, count * es, P.max_pitch) : 0;
    const size_t r_pitch = stage_ok ? row_stride(recv, nranks, count * es, P.max_pitch) : 0;
    bool rows_in = s_pitch != 0, rows_out = r_pitch != 0;

    // both copy streams start after the work already on `stream`
    if ((e = cudaEventRecord(P.start, stream)) != cudaSuccess)
        return e;
    if ((e = cudaStreamWaitEvent(P.h2d, P.start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(P.d2h, P.start, 0)) != cudaSuccess)
        return e;

    std::vector<void *> stage(nranks);
    std::vector<RedSeg> segs;
    for (size_t k = 0; k < slices.size() && e == cudaSuccess; ++k) {
        const int s = (int)(k % kHostStages);
        const uint64_t lo = slices[k].off, n = slices[k].len;
        const size_t bytes = n * es;
        for (int r = 0; r < nranks; ++r)
            stage[r] = static_cast<char *>(work) + ((size_t)s * nranks + r) * L * es;
        // the stage is free once its previous slice -- of this call or an
        // earlier one -- has been copied out (a never-recorded event is no wait)
        e = cudaStreamWaitEvent(P.h2d, P.out[s], 0);
        if (rows_in && e == cudaSuccess &&
            cudaMemcpy2DAsync(stage[0], stage_bytes, static_cast<const char *>(send[0]) + lo * es, s_pitch, bytes,
                              nranks, cudaMemcpyDefault, P.h2d) != cudaSuccess) {
            cudaGetLastError(); // refused at enqueue: nothing was queued
            rows_in = false;
        }
        for (int r = 0; r < nranks && !rows_in && e == cudaSuccess; ++r)
            e = cudaMemcpyAsync(stage[r], static_cast<const char *>(send[r]) + lo * es, bytes, cudaMemcpyDefault,
                                P.h2d);
        if (e == cudaSuccess)
            e = cudaEventRecord(P.in[s], P.h2d);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(stream, P.in[s], 0);
        if (e == cudaSuccess) {
            slice_segments(part, nranks, lo, n, segs);
            e = launch_bucket_reduce(dt, op, stage.data(), 1, nranks, segs.data(), segs.size(), stream);
        }
        if (e == cudaSuccess)
            e = cudaEventRecord(P.red[s], stream);
        if (e == cudaSuccess)
            e = cudaStreamWaitEvent(P.d2h, P.red[s], 0);
        if (rows_out && e == cudaSuccess &&
            cudaMemcpy2DAsync(static_cast<char *>(recv[0]) + lo * es, r_pitch, stage[0], stage_bytes, bytes, nranks,
                              cudaMemcpyDefault, P.d2h) != cudaSuccess) {
            cudaGetLastError();
            rows_out = false;
        }
        for (int r = 0; r < nranks && !rows_out && e == cudaSuccess; ++r)
            e = cudaMemcpyAsync(static_cast<char *>(recv[r]) + lo * es, stage[r], bytes, cudaMemcpyDefault, P.d2h);
        if (e == cudaSuccess)
            e = cudaEventRecord(P.out[s], P.d2h);
    }
    // join both copy streams back into `stream`, also after an error, so that
    // nothing the call enqueued outlives what the caller waits for
    cudaError_t j = cudaEventRecord(P.h2d_end, P.h2d);
    if (j == cudaSuccess)
        j = cudaEventRecord(P.d2h_end, P.d2h);
    if (j == cudaSuccess)
        j = cudaStreamWaitEvent(stream, P.h2d_end, 0);
    if (j == cudaSuccess)
        j = cudaStreamWaitEvent(stream, P.d2h_end, 0);
    return e != cudaSuccess ? e : j;
}

} // namespace ccl
