// check.cu -- result checks and call tracing.
//
// After an AllReduce every rank must hold the same bits (Collective
// Communication, Definition 1.1: gradient synchronisation leaves every replica
// identical; the section on pitfalls: silent corruption calls for checking
// results).  ccl_check_identical compares every rank's buffer with rank 0's,
// bit for bit, and adds the number of differing elements to a device counter;
// it never traps, so a corrupted result is reported, not fatal.
//
// Tracing keeps the last calls' descriptions (collective, ranks, count, type,
// op, mode, kernels launched, host time to enqueue, and device time from two
// events around the call's work on its stream) in a host ring buffer.
#include <atomic>
#include <chrono>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include <nvtx3/nvToolsExt.h>

#include "../../include/ccl.h"
#include "ccl_internal.h"

namespace ccl {

template <int MAXR> struct CheckParams {
    const void *buf[MAXR];
    uint64_t K;
    unsigned long long *mismatches;
    int nranks;
    int vec_aligned;
    int elem_size;
};

// one element (or 16-byte vector) per thread; differing lanes counted with a
// warp ballot and added once per warp
template <int MAXR>
__global__ void __launch_bounds__(kThreads) check_identical_kernel(const __grid_constant__ CheckParams<MAXR> p)
{
    const uint64_t i = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const int es = p.elem_size;
    const uint64_t per_vec = 16 / es;
    unsigned bad = 0;
    if (p.vec_aligned) {
        const uint64_t nv = p.K / per_vec;
        if (i < nv) {
            const uint4 a = ld16(static_cast<const char *>(p.buf[0]) + i * 16);
            for (int r = 1; r < p.nranks; ++r) {
                const uint4 b = ld16(static_cast<const char *>(p.buf[r]) + i * 16);
                const uint32_t x[4] = {a.x ^ b.x, a.y ^ b.y, a.z ^ b.z, a.w ^ b.w};
                for (int w = 0; w < 4; ++w) {
                    if (es == 4)
                        bad += x[w] != 0;
                    else
                        bad += ((x[w] & 0xffffu) != 0) + ((x[w] >> 16) != 0);
                }
            }
        }
        // the tail after the last whole vector, one element per thread of block 0
        if (blockIdx.x == 0)
            for (uint64_t e = nv * per_vec + threadIdx.x; e < p.K; e += kThreads)
                for (int r = 1; r < p.nranks; ++r)
                    bad += es == 4 ? ld_elem<DT_FP32>(p.buf[r], e) != ld_elem<DT_FP32>(p.buf[0], e)
                                   : ld_elem<DT_BF16>(p.buf[r], e) != ld_elem<DT_BF16>(p.buf[0], e);
    } else if (i < p.K) {
        for (int r = 1; r < p.nranks; ++r)
            bad += es == 4 ? ld_elem<DT_FP32>(p.buf[r], i) != ld_elem<DT_FP32>(p.buf[0], i)
                           : ld_elem<DT_BF16>(p.buf[r], i) != ld_elem<DT_BF16>(p.buf[0], i);
    }
    // warp total: lanes with nothing to add stay out of the atomic
    const unsigned any = __ballot_sync(0xffffffffu, bad != 0);
    unsigned total = bad;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        total += __shfl_xor_sync(0xffffffffu, total, o);
    if (any && (threadIdx.x & 31) == 0 && dbg_ok(p.mismatches, sizeof *p.mismatches))
        atomicAdd(p.mismatches, (unsigned long long)total);
}

template <int MAXR>
static cudaError_t launch_check_t(const void *const *bufs, int nranks, uint64_t count, int es,
                                  unsigned long long *mismatches, cudaStream_t stream)
{
    CheckParams<MAXR> p;
    bool aligned = true;
    for (int r = 0; r < MAXR; ++r) {
        p.buf[r] = r < nranks ? bufs[r] : nullptr;
        if (r < nranks)
            aligned = aligned && (uintptr_t)bufs[r] % 16 == 0;
    }
    p.K = count;
    p.mismatches = mismatches;
    p.nranks = nranks;
    p.vec_aligned = aligned ? 1 : 0;
    p.elem_size = es;
    const uint64_t work = aligned ? count / (16 / es) : count;
    uint64_t blocks = (work + kThreads - 1) / kThreads;
    if (blocks == 0)
        blocks = 1;
    if (blocks > 0x7fffffffull)
        return cudaErrorInvalidValue;
    check_identical_kernel<MAXR><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ bounds checks (debug builds)

#ifdef CCL_DEBUG_BOUNDS
__device__ unsigned g_dbg_n = 0;
__device__ unsigned long long g_dbg_r[kDbgMaxRanges][2];
__device__ unsigned g_dbg_faults = 0;
__device__ unsigned long long g_dbg_first_fault = 0;
#endif

cudaError_t dbg_set_ranges(const std::vector<DbgRange> &ranges, cudaStream_t stream)
{
#ifdef CCL_DEBUG_BOUNDS
    // CCL_DEBUG_SHRINK (tests of the checker only): register the first half
    // of every range, so that the second half's accesses are counted and
    // skipped -- nothing outside the buffers is touched either way
    static const bool shrink = [] {
        const char *e = std::getenv("CCL_DEBUG_SHRINK");
        return e && e[0] && std::strcmp(e, "0") != 0;
    }();
    std::vector<unsigned long long> r;
    r.reserve(ranges.size() * 2);
    for (const DbgRange &g : ranges) {
        if (r.size() / 2 == (size_t)kDbgMaxRanges || !g.lo || !g.bytes)
            continue;
        const unsigned long long lo = (unsigned long long)(uintptr_t)g.lo;
        r.push_back(lo);
        r.push_back(lo + (shrink ? g.bytes / 2 : g.bytes));
    }
    const unsigned n = (unsigned)(r.size() / 2);
    cudaError_t e = cudaSuccess;
    if (n)
        e = cudaMemcpyToSymbolAsync(g_dbg_r, r.data(), r.size() * sizeof(unsigned long long), 0,
                                    cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbolAsync(g_dbg_n, &n, sizeof n, 0, cudaMemcpyHostToDevice, stream);
    return e;
#else
    (void)ranges;
    (void)stream;
    return cudaSuccess;
#endif
}

// ------------------------------------------------------------------ automatic checks

namespace {
std::atomic<int> g_check_on{-1}; // -1: read CCL_CHECK on first use
std::mutex g_chk_mu;
std::unordered_map<int, unsigned long long *> g_chk_ctr; // per device
} // namespace

bool check_enabled()
{
    int v = g_check_on.load(std::memory_order_relaxed);
    if (v < 0) {
        const char *env = std::getenv("CCL_CHECK");
        v = (env && env[0] && std::strcmp(env, "0") != 0) ? 1 : 0;
        g_check_on.store(v, std::memory_order_relaxed);
    }
    return v > 0;
}

cudaError_t auto_check(const void *const *bufs, int nranks, uint64_t count, int elem_size, cudaStream_t stream)
{
    if (!check_enabled() || nranks < 2 || count == 0)
        return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    unsigned long long *ctr = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_chk_mu);
        auto it = g_chk_ctr.find(dev);
        if (it == g_chk_ctr.end()) {
            if ((e = cudaMalloc(&ctr, sizeof *ctr)) != cudaSuccess || (e = cudaMemset(ctr, 0, sizeof *ctr)) != cudaSuccess)
                return e;
            g_chk_ctr[dev] = ctr;
        } else {
            ctr = it->second;
        }
    }
    std::vector<DbgRange> rg; // debug builds: the outputs and the counter
    for (int r = 0; r < nranks; ++r)
        rg.push_back(DbgRange{bufs[r], (size_t)count * (size_t)elem_size});
    rg.push_back(DbgRange{ctr, sizeof *ctr});
    if ((e = dbg_set_ranges(rg, stream)) != cudaSuccess)
        return e;
    return nranks <= kSmallRanks ? launch_check_t<kSmallRanks>(bufs, nranks, count, elem_size, ctr, stream)
                                 : launch_check_t<kMaxRanks>(bufs, nranks, count, elem_size, ctr, stream);
}

// ------------------------------------------------------------------ tracing

namespace {
constexpr size_t kTraceCap = 4096;
std::mutex g_trace_mu;
ccl_trace_record_t g_trace[kTraceCap];
// the events around each held call, until its device time has been read
struct EventPair {
    cudaEvent_t start, end;
};
EventPair g_trace_ev[kTraceCap];
size_t g_trace_next = 0, g_trace_count = 0;

void release(EventPair &p)
{
    // an event still pending is released by the runtime once it completes
    if (p.start)
        cudaEventDestroy(p.start);
    if (p.end)
        cudaEventDestroy(p.end);
    p.start = p.end = nullptr;
}

// Fills in the device time of a held call whose events have completed.
void resolve(size_t slot)
{
    EventPair &p = g_trace_ev[slot];
    if (!p.end || cudaEventQuery(p.end) != cudaSuccess)
        return;
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, p.start, p.end) == cudaSuccess && ms >= 0.0f)
        g_trace[slot].gpu_ns = (unsigned long long)((double)ms * 1e6 + 0.5);
    release(p);
}
std::atomic<int> g_trace_on{-1}; // -1: read CCL_TRACE on first use
} // namespace

bool trace_enabled()
{
    int v = g_trace_on.load(std::memory_order_relaxed);
    if (v < 0) {
        const char *env = std::getenv("CCL_TRACE");
        v = (env && env[0] && std::strcmp(env, "0") != 0) ? 1 : 0;
        g_trace_on.store(v, std::memory_order_relaxed);
    }
    return v > 0;
}

TraceScope::TraceScope(const char *name, int nranks, uint64_t count, int dtype, int op, int mode,
                       cudaStream_t stream)
    : active_(trace_enabled()), stream_(stream)
{
    // an NVTX range per call, so that profiler timelines name the collective
    // (no cost beyond a check when no tool is attached)
    nvtxRangePushA(name);
    if (!active_)
        return;
    std::memset(&rec_, 0, sizeof rec_);
    std::strncpy(rec_.collective, name, sizeof rec_.collective - 1);
    rec_.nranks = nranks;
    rec_.count = count;
    rec_.dtype = dtype;
    rec_.op = op;
    rec_.mode = mode;
    launches0_ = thread_launch_count();
    t0_ = std::chrono::steady_clock::now().time_since_epoch().count();
    // device time: an event before the call's work on its stream (none while
    // the stream is being captured, where events would become graph nodes)
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return;
    }
    if (cudaEventCreate(&ev0_) != cudaSuccess || cudaEventCreate(&ev1_) != cudaSuccess ||
        cudaEventRecord(ev0_, stream) != cudaSuccess) {
        cudaGetLastError();
        EventPair p{ev0_, ev1_};
        release(p);
        ev0_ = ev1_ = nullptr;
    }
}

void TraceScope::finish(int status)
{
    nvtxRangePop();
    if (!active_)
        return;
    active_ = false;
    const long long t1 = std::chrono::steady_clock::now().time_since_epoch().count();
    rec_.status = status;
    rec_.launches = (unsigned)(thread_launch_count() - launches0_);
    rec_.host_ns = (unsigned long long)(t1 - t0_);
    rec_.gpu_ns = 0;
    EventPair ev{ev0_, ev1_};
    if (ev.end && cudaEventRecord(ev.end, stream_) != cudaSuccess) {
        cudaGetLastError();
        release(ev);
    }
    std::lock_guard<std::mutex> lk(g_trace_mu);
    rec_.seq = g_trace_count;
    release(g_trace_ev[g_trace_next]); // the overwritten call's events, if unread
    g_trace[g_trace_next] = rec_;
    g_trace_ev[g_trace_next] = ev;
    g_trace_next = (g_trace_next + 1) % kTraceCap;
    ++g_trace_count;
}

} // namespace ccl

using namespace ccl;

extern "C" {

ccl_status_t ccl_check_identical(const void *const *bufs, int nranks, size_t count, ccl_dtype_t dtype,
                                 unsigned long long *mismatches, cudaStream_t stream)
{
    if (nranks < 1 || nranks > CCL_MAX_RANKS || (dtype != CCL_FP32 && dtype != CCL_BF16) || !bufs || !mismatches)
        return CCL_ERR_INVALID_ARG;
    for (int r = 0; r < nranks; ++r)
        if (!bufs[r] && count)
            return CCL_ERR_INVALID_ARG;
    if (count == 0 || nranks == 1)
        return CCL_OK;
    const int es = dtype == CCL_BF16 ? 2 : 4;
    std::vector<DbgRange> rg; // debug builds: the buffers and the counter
    for (int r = 0; r < nranks; ++r)
        rg.push_back(DbgRange{bufs[r], count * (size_t)es});
    rg.push_back(DbgRange{mismatches, sizeof *mismatches});
    if (dbg_set_ranges(rg, stream) != cudaSuccess)
        return CCL_ERR_CUDA;
    const cudaError_t e = nranks <= kSmallRanks ? launch_check_t<kSmallRanks>(bufs, nranks, count, es, mismatches, stream)
                                                : launch_check_t<kMaxRanks>(bufs, nranks, count, es, mismatches, stream);
    return e == cudaSuccess ? CCL_OK : CCL_ERR_CUDA;
}

void ccl_set_trace(int enabled) { g_trace_on.store(enabled ? 1 : 0, std::memory_order_relaxed); }

void ccl_set_check(int enabled) { g_check_on.store(enabled ? 1 : 0, std::memory_order_relaxed); }

ccl_status_t ccl_debug_faults(unsigned long long *faults, unsigned long long *first_address)
{
#ifdef CCL_DEBUG_BOUNDS
    if (!faults || !first_address)
        return CCL_ERR_INVALID_ARG;
    unsigned n = 0;
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpyFromSymbol(&n, g_dbg_faults, sizeof n) != cudaSuccess ||
        cudaMemcpyFromSymbol(first_address, g_dbg_first_fault, sizeof *first_address) != cudaSuccess)
        return CCL_ERR_CUDA;
    *faults = n;
    return CCL_OK;
#else
    (void)faults;
    (void)first_address;
    return CCL_ERR_UNSUPPORTED;
#endif
}

ccl_status_t ccl_check_read(unsigned long long *mismatches, int reset)
{
    if (!mismatches)
        return CCL_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return CCL_ERR_CUDA;
    unsigned long long *ctr = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_chk_mu);
        auto it = g_chk_ctr.find(dev);
        if (it != g_chk_ctr.end())
            ctr = it->second;
    }
    *mismatches = 0;
    if (!ctr)
        return CCL_OK; // nothing checked on this device yet
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(mismatches, ctr, sizeof *ctr, cudaMemcpyDeviceToHost) != cudaSuccess)
        return CCL_ERR_CUDA;
    if (reset && cudaMemset(ctr, 0, sizeof *ctr) != cudaSuccess)
        return CCL_ERR_CUDA;
    return CCL_OK;
}

size_t ccl_trace_read(ccl_trace_record_t *out, size_t max_records)
{
    std::lock_guard<std::mutex> lk(g_trace_mu);
    const size_t have = g_trace_count < kTraceCap ? g_trace_count : kTraceCap;
    const size_t n = out ? (max_records < have ? max_records : have) : have;
    if (out)
        for (size_t k = 0; k < n; ++k) { // oldest first, the newest n records
            const size_t slot = (g_trace_next + kTraceCap - n + k) % kTraceCap;
            resolve(slot);
            out[k] = g_trace[slot];
        }
    return n;
}

void ccl_trace_clear(void)
{
    std::lock_guard<std::mutex> lk(g_trace_mu);
    for (size_t k = 0; k < kTraceCap; ++k)
        release(g_trace_ev[k]);
    g_trace_next = 0;
    g_trace_count = 0;
}

} // extern "C"
