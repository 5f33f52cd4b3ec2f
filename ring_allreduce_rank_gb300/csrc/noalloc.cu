// noalloc.cu -- step-by-step ReduceScatter that never allocates device memory.
//
// The regular step-mode ReduceScatter (ccl_reduce_scatter with CCL_MODE_STEP)
// needs N*count elements of working space, which the library gets with
// cudaMalloc the first time and keeps.  Some callers cannot let a library do
// that: a process whose framework has already reserved the GPU's memory in its
// own caching pool (a raw cudaMalloc then fails or fragments what is left),
// code that must not stall other streams on the implicit device
// synchronisation that cudaMalloc/cudaFree can cause, or hosts that forbid
// driver allocations outside start-up.  This variant runs the same ring steps
// with its working space in one fixed array in device memory.
//
// When that array is reserved depends on how CUDA loads this library's device
// code.  Under lazy loading (the default since CUDA 12.2) it is reserved the
// first time a device resolves its address, not when the library is loaded.
// A call with count = 0 does exactly that set-up on the current device: it
// resolves the address (reserving the array) and loads every kernel the entry
// launches, so that later calls need no device memory at all.
#include <mutex>
#include <unordered_map>
#include <vector>

#include "../../include/ccl.h"
#include "ccl_internal.h"

namespace {

// The working space, CCL_STATIC_SCRATCH_BYTES per device.  Every GPU that
// reserves it keeps it until the process exits.  All calls on a device share
// it, so two calls whose work overlaps on that GPU (different streams, or
// different host threads) race on it.
static __device__ __align__(256) unsigned char ccl_static_scratch[CCL_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
std::unordered_map<int, void *> g_scratch_addr; // device -> device address of ccl_static_scratch

// Host code only sees a host-side stand-in for ccl_static_scratch; the device
// address comes from cudaGetSymbolAddress, once per device, with that device
// current.  The first lookup on a device also loads the kernels this entry
// launches.
ccl_status_t scratch_address(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return CCL_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    auto it = g_scratch_addr.find(dev);
    if (it == g_scratch_addr.end()) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, ccl_static_scratch) != cudaSuccess || p == nullptr ||
            ccl::preload_ring_step_kernels() != cudaSuccess || ccl::preload_copy_kernels() != cudaSuccess) {
            cudaGetLastError();
            return CCL_ERR_CUDA;
        }
        it = g_scratch_addr.emplace(dev, p).first;
    }
    *out = it->second;
    return CCL_OK;
}

} // namespace

void ccl::forget_static_scratch(int dev)
{
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    g_scratch_addr.erase(dev);
}

using namespace ccl;

extern "C" ccl_status_t ccl_reduce_scatter_step_static(const void *const *send, void *const *recv, int nranks,
                                                       size_t count, ccl_dtype_t dtype, ccl_op_t op,
                                                       cudaStream_t stream)
{
    // the same checks, in the same order, as ccl_reduce_scatter
    std::vector<Range> w, r;
    ccl_status_t st = check_reduce_scatter(send, recv, nranks, count, dtype, op, w, r);
    if (st != CCL_OK)
        return st;
    const size_t es = elem_size(dtype);
    // each rank's working copy starts on a 256-byte boundary
    const size_t stride = (count * es + 255) & ~(size_t)255;
    if (stride < count * es || stride > CCL_STATIC_SCRATCH_BYTES / (size_t)nranks)
        return CCL_ERR_INVALID_ARG; // more than the fixed working space holds
    void *base = nullptr;
    if ((st = scratch_address(&base)) != CCL_OK)
        return st;
    if (count == 0)
        return CCL_OK; // the set-up call: array reserved, kernels loaded, nothing enqueued
    const Partition part = make_partition(count, nranks);
    std::vector<void *> bufs(nranks);
    for (int i = 0; i < nranks; ++i)
        bufs[i] = static_cast<char *>(base) + (size_t)i * stride;
    {   // debug builds: the scratch rows and the call's buffers
        std::vector<DbgRange> rg;
        for (int i = 0; i < nranks; ++i) {
            rg.push_back(DbgRange{send[i], count * es});
            rg.push_back(DbgRange{bufs[i], count * es});
            rg.push_back(DbgRange{recv[i], part.len((uint32_t)i) * es});
        }
        if (dbg_set_ranges(rg, stream) != cudaSuccess)
            return CCL_ERR_CUDA;
    }
    // Every scratch byte the ring reads below is first written by this copy, so
    // whatever an earlier call left in the array never reaches the result.
    std::vector<CopySeg> segs;
    for (int i = 0; i < nranks; ++i)
        segs.push_back(CopySeg{static_cast<const char *>(send[i]), static_cast<char *>(bufs[i]), count * es, 0});
    if (launch_copy_segments(segs.data(), segs.size(), stream) != cudaSuccess)
        return CCL_ERR_CUDA;
    for (int s = 0; s < nranks - 1; ++s)
        if (launch_ring_step((int)dtype, (int)op, STEP_RS, s, bufs.data(), nranks, count, stream) != cudaSuccess)
            return CCL_ERR_CUDA;
    // AVG divides once at the end; the pre-multiplied AVG scales inside the
    // steps, and needs this launch only when N = 1 gives it no step
    if (step_scale((int)op, nranks) &&
        launch_ring_step((int)dtype, (int)op, STEP_SCALE, 0, bufs.data(), nranks, count, stream) != cudaSuccess)
        return CCL_ERR_CUDA;
    // the ReduceScatter phase leaves chunk c finished at rank c-1; hand it to rank c
    segs.clear();
    for (int c = 0; c < nranks; ++c)
        segs.push_back(CopySeg{static_cast<const char *>(bufs[ring_mod(c - 1, nranks)]) +
                                   part.off((uint32_t)c) * es,
                               static_cast<char *>(recv[c]), part.len((uint32_t)c) * es, 0});
    if (launch_copy_segments(segs.data(), segs.size(), stream) != cudaSuccess)
        return CCL_ERR_CUDA;
    return CCL_OK;
}
