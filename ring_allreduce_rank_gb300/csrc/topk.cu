// topk.cu -- the threshold of Top-k sparsification, found on the device.
//
// Top-k ("Top-k sparsification", Collective Communication) sends, per rank,
// the values of u = g + e whose magnitude reaches the k-th largest magnitude
// |u|_(k), every tie included, and keeps the rest as residual.  Magnitudes are
// ordered as the bit patterns of |u| (the sign bit cleared): for numbers that
// is the order of |u|, and a NaN lands above every number.  The k-th largest
// 31-bit key tau is found by a radix select on the top 12 key bits (bits
// 30..19, a 4096-bin histogram) and then the low 19 bits of the keys in the
// top bin that holds the k-th key (a 2^19-bin histogram, 2 MB per rank,
// resident in L2).  Both histograms come out of ONE full pass over g and e:
//   1. a sample (one run of 256 elements in every 16, 32, 64 or 128)
//      histograms its top bits, and a scan picks a window of top bins that
//      holds the k-th key with high probability: the bins between the
//      sample's order statistics k f -+ m (f the sampled fraction, m five
//      standard deviations of the count), at most kWindowMax of them;
//   2. the full pass counts every key's top bits exactly (shared-memory
//      atomics per CTA, merged into a 64-bit histogram per rank) and the low
//      bits of the keys inside the window (global atomics);
//   3. a scan of the exact top histogram fixes the top bin of the k-th key;
//      if the window missed it, a second full pass counts that bin's low bits
//      (its launches return at once when the window held the bin);
//   4. block sums and a last scan of the low histogram give the exact key.
// The sample only decides how much work the select does, never its result.
// The compressed AllReduce kernel then sends u where key(u) >= tau, in the
// same pass that writes the residuals and folds the sent values in ring order.
//
// Everything stays on the device and in the caller's work buffer, so a call
// never waits for the host and can be captured in a CUDA graph.
#include <cmath>

#include "ccl_internal.h"

namespace ccl {

// A top digit (8 exponent bits, 4 mantissa bits) is 1/16 of a binade: the
// window's digits hold few keys (one low-histogram increment each), and each
// digit's low histogram is 2 MB per rank.
constexpr int kTopBins = 4096;          // key bits 30..19
constexpr int kLowBits = 19;            // key bits 18..0
constexpr uint32_t kLowBins = 1u << kLowBits;
constexpr int kLowBlocks = 256;         // a low histogram in blocks of 2048 bins
constexpr int kLowPerBlock = (int)(kLowBins / kLowBlocks);
// The window covers the top digits between the sample's two bounds, at most
// this many (a quarter of a binade): narrow when the sample pins the k-th key
// down, as wide as it needs to be otherwise.
constexpr int kWindowMax = 4;
constexpr int kRegions = kWindowMax + 1; // low histograms per rank: the window's, then the fallback's
constexpr int kRun = 32;                // groups of 8 elements in a sampled run (one group per lane)
// The sample takes one run in every 16; for large inputs one in every 32, 64
// or 128, which reads less of g and e, as long as its window stays as narrow:
// see sample_every.
constexpr uint32_t kSampleMin = 16, kSampleMax = 128;
constexpr uint64_t kSampleTarget = 4096;
constexpr int kInitCtas = 64;           // CTAs per rank that clear low histograms
constexpr uint32_t kNoWindow = 0xffffffffu;

struct TopkState {
    uint32_t prefix;        // top digit of the k-th key, once fixed
    uint32_t tau;           // the k-th largest key, once found
    unsigned long long kr;  // rank (1-based) of the k-th key among the keys with that top digit
    uint32_t wlo;           // first top digit of the window, or kNoWindow
    uint32_t region;        // low histogram that counts the k-th key's top bin
    uint32_t hit;           // the window held that bin: no second pass
    uint32_t nwin;          // top digits in the window (0: none)
};

// Work buffer, for n ranks: top[n][kTopBins] (u64), stop[n][kTopBins] (u32,
// the sample's), low[n][kRegions][kLowBins] (u32), blk[n][kLowBlocks] (u64),
// state[n], tau[n].
struct TopkParams {
    const void *grads[kTopkMaxRanks];
    const float *res[kTopkMaxRanks];
    unsigned long long *top;
    uint32_t *stop;
    uint32_t *low;
    unsigned long long *blk;
    TopkState *state;
    uint32_t *tau; // read by the compressed kernel
    uint64_t K;
    unsigned long long k;
    unsigned long long qa, qb; // the sample's order statistics that bound the window (qa < qb)
    uint32_t every;            // the sample takes run q when q % every == 0
    int nranks;
    int vec_ok; // every gradient and residual 16-byte aligned
};

__device__ __forceinline__ uint32_t topk_key(float g, float e) { return __float_as_uint(__fadd_rn(g, e)) & 0x7fffffffu; }

// g and e stream through L2 once: streaming loads (evict first) leave the
// low histograms, which the window's keys count into, resident in L2.
template <class T> __device__ __forceinline__ T gload_stream(const T *p)
{
    T v{};
    if (dbg_ok(p, sizeof(T)))
        v = __ldcs(p);
    return v;
}

// u = g + e for the 8 elements of group gi (16-byte loads; vec_ok buffers).
template <int DT, class F> __device__ __forceinline__ void group_keys(const void *g, const float *e, uint64_t gi, F &&f)
{
    float gv[8];
    if (DT == DT_BF16) {
        const uint4 w = gload_stream(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(g) + gi * 8));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            gv[2 * j] = __uint_as_float(ws[j] << 16);
            gv[2 * j + 1] = __uint_as_float(ws[j] & 0xffff0000u);
        }
    } else {
        const float4 a = gload_stream(reinterpret_cast<const float4 *>(static_cast<const float *>(g) + gi * 8));
        const float4 b = gload_stream(reinterpret_cast<const float4 *>(static_cast<const float *>(g) + gi * 8 + 4));
        gv[0] = a.x; gv[1] = a.y; gv[2] = a.z; gv[3] = a.w;
        gv[4] = b.x; gv[5] = b.y; gv[6] = b.z; gv[7] = b.w;
    }
    const float4 ea = gload_stream(reinterpret_cast<const float4 *>(e + gi * 8)),
                 eb = gload_stream(reinterpret_cast<const float4 *>(e + gi * 8 + 4));
    const float ev[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
#pragma unroll
    for (int j = 0; j < 8; ++j)
        f(topk_key(gv[j], ev[j]));
}

// Calls f(key) for every element of rank r that this CTA covers: groups of 8
// elements with 16-byte loads, the rest (all of it when a buffer is
// unaligned) one element at a time.
template <int DT, class F> __device__ __forceinline__ void for_each_key(const TopkParams &p, int r, F &&f)
{
    const void *g = p.grads[r];
    const float *e = p.res[r];
    const uint64_t K = p.K;
    const uint64_t ng = p.vec_ok ? K / 8 : 0;
    const uint64_t stride = (uint64_t)gridDim.x * kThreads;
    for (uint64_t gi = (uint64_t)blockIdx.x * kThreads + threadIdx.x; gi < ng; gi += stride)
        group_keys<DT>(g, e, gi, f);
    for (uint64_t i = ng * 8 + (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < K; i += stride) {
        const uint32_t b = ld_elem<DT>(g, i);
        f(topk_key(__uint_as_float(DT == DT_BF16 ? b << 16 : b), gload<float>(e + i)));
    }
}

// Exclusive prefix sum of one value per thread, in thread order.  Every
// thread of the CTA calls it; ws holds kThreads / 32 values of shared memory.
__device__ __forceinline__ unsigned long long cta_exclusive_scan(unsigned long long s, unsigned long long *ws)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned long long incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    __syncthreads(); // ws may still be read by an earlier call
    if (lane == 31)
        ws[warp] = incl;
    __syncthreads();
    unsigned long long base = 0;
    for (int w = 0; w < warp; ++w)
        base += ws[w];
    return base + incl - s;
}

// Merge a CTA's shared-memory histogram into a global one.
template <class T> __device__ __forceinline__ void merge_hist(const uint32_t *h, T *gh)
{
    for (int i = threadIdx.x; i < kTopBins; i += kThreads)
        if (h[i] && dbg_ok(gh + i, sizeof(T)))
            atomicAdd(gh + i, (T)h[i]);
}

__device__ __forceinline__ uint32_t *low_region(const TopkParams &p, int r, uint32_t region)
{
    return p.low + ((size_t)r * kRegions + region) * kLowBins;
}

// The select's kernels, and the compressed pass after them, run as a chain of
// programmatic dependent launches (chain_entry, launch_chained).
__global__ void __launch_bounds__(kThreads) topk_init_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    const int r = blockIdx.y;
    if (p.k > 0 && p.k < p.K) { // the window's low histograms, only when a select follows
        uint4 *low = reinterpret_cast<uint4 *>(low_region(p, r, 0));
        for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < kWindowMax * kLowBins / 4; i += gridDim.x * kThreads)
            gstore<uint4>(low + i, make_uint4(0, 0, 0, 0));
    }
    if (blockIdx.x != 0)
        return;
    for (int i = threadIdx.x; i < kTopBins; i += kThreads) {
        gstore<unsigned long long>(p.top + (size_t)r * kTopBins + i, 0ull);
        gstore<uint32_t>(p.stop + (size_t)r * kTopBins + i, 0u);
    }
    if (threadIdx.x == 0) {
        TopkState s;
        s.prefix = 0;
        s.kr = p.k;
        // k = 0: no key reaches tau, nothing is sent; k >= K: every key does
        s.tau = p.k == 0 ? 0xffffffffu : 0u;
        s.wlo = kNoWindow;
        s.region = kWindowMax;
        s.hit = 0;
        s.nwin = 0;
        gstore<TopkState>(p.state + r, s);
        gstore<uint32_t>(p.tau + r, s.tau);
    }
}

// 1. The sample: run q of 32 groups (one per lane of a warp) for q = 0, f,
// 2f, ... (f = p.every): whole 512-byte (bf16) or 1 KB (fp32, residuals)
// spans, so the sample reads about 1/f of the bytes.
template <int DT>
__global__ void __launch_bounds__(kThreads) topk_sample_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    __shared__ uint32_t h[kTopBins];
    for (int i = threadIdx.x; i < kTopBins; i += kThreads)
        h[i] = 0u;
    __syncthreads();
    const int r = blockIdx.y, lane = threadIdx.x & 31;
    const uint64_t ng = p.K / 8, nruns = (ng + kRun - 1) / kRun;
    const uint64_t nsampled = (nruns + p.every - 1) / p.every;
    const uint64_t warps = (uint64_t)gridDim.x * (kThreads / 32);
    for (uint64_t w = (uint64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); w < nsampled; w += warps) {
        const uint64_t gi = w * p.every * kRun + (uint64_t)lane;
        if (gi < ng)
            group_keys<DT>(p.grads[r], p.res[r], gi, [&](uint32_t key) { atomicAdd(&h[key >> kLowBits], 1u); });
    }
    __syncthreads();
    merge_hist<uint32_t>(h, p.stop + (size_t)r * kTopBins);
}

// The window: the top digits dB..dA of the sample's qb-th and qa-th largest
// keys, when there are at most kWindowMax of them.
__global__ void __launch_bounds__(kThreads) topk_window_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    constexpr int kPer = kTopBins / kThreads;
    __shared__ unsigned long long ws[kThreads / 32];
    __shared__ int dA, dB;
    const int r = blockIdx.x, t = threadIdx.x;
    if (t == 0)
        dA = dB = -1;
    const uint32_t *gh = p.stop + (size_t)r * kTopBins;
    unsigned long long c[kPer], s = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        c[j] = gload<uint32_t>(gh + (kTopBins - 1 - (t * kPer + j)));
        s += c[j];
    }
    const unsigned long long excl = cta_exclusive_scan(s, ws); // its barriers order dA, dB's reset
    unsigned long long acc = excl;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int d = kTopBins - 1 - (t * kPer + j);
        if (acc < p.qa && p.qa <= acc + c[j])
            dA = d;
        if (acc < p.qb && p.qb <= acc + c[j])
            dB = d;
        acc += c[j];
    }
    __syncthreads();
    if (t == 0 && dA >= 0 && dB >= 0 && dA - dB < kWindowMax) {
        TopkState st = gload<TopkState>(p.state + r);
        st.wlo = (uint32_t)dB;
        st.nwin = (uint32_t)(dA - dB + 1);
        gstore<TopkState>(p.state + r, st);
    }
}

// A CTA's cache of window bins in shared memory: a slot holds one bin (its
// index into the window's low histograms) and that bin's count so far.  When
// the window's keys fall on few bins -- residuals of bf16-valued numbers leave
// only a few low bits free -- counting them here spares L2 a stream of
// reductions into the same few addresses; keys whose slot another bin holds go
// to L2 directly.  Each slot is flushed once, when the CTA ends.
constexpr int kBinCache = 256;
constexpr uint32_t kEmptySlot = 0xffffffffu;

// 2. The full pass: exact top histogram, and the low bits of the keys whose
// top bin lies in the window.
template <int DT>
__global__ void __launch_bounds__(kThreads) topk_main_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    __shared__ uint32_t h[kTopBins];
    __shared__ uint32_t cache_bin[kBinCache], cache_cnt[kBinCache];
    for (int i = threadIdx.x; i < kTopBins; i += kThreads)
        h[i] = 0u;
    for (int i = threadIdx.x; i < kBinCache; i += kThreads) {
        cache_bin[i] = kEmptySlot;
        cache_cnt[i] = 0u;
    }
    __syncthreads();
    const int r = blockIdx.y;
    const TopkState st = gload<TopkState>(p.state + r);
    const uint32_t wlo = st.wlo, nwin = st.nwin;
    uint32_t *low = low_region(p, r, 0);
    for_each_key<DT>(p, r, [&](uint32_t key) {
        const uint32_t d = key >> kLowBits;
        atomicAdd(&h[d], 1u);
        const uint32_t w = d - wlo; // wraps past nwin below the window
        if (w < nwin) {
            const uint32_t bin = w * kLowBins + (key & (kLowBins - 1u)); // < kWindowMax * kLowBins
            const uint32_t slot = (bin * 2654435761u) >> 24;            // Fibonacci hash, 256 slots
            const uint32_t held = atomicCAS(&cache_bin[slot], kEmptySlot, bin);
            if (held == kEmptySlot || held == bin) {
                atomicAdd(&cache_cnt[slot], 1u);
            } else {
                uint32_t *b = low + bin;
                if (dbg_ok(b, sizeof(uint32_t)))
                    atomicAdd(b, 1u);
            }
        }
    });
    __syncthreads();
    merge_hist<unsigned long long>(h, p.top + (size_t)r * kTopBins);
    for (int i = threadIdx.x; i < kBinCache; i += kThreads) {
        const uint32_t bin = cache_bin[i], n = cache_cnt[i];
        if (bin != kEmptySlot && n) {
            uint32_t *b = low + bin;
            if (dbg_ok(b, sizeof(uint32_t)))
                atomicAdd(b, n);
        }
    }
}

// 3. One CTA per rank: the top bin of the k-th key, walking from the top;
// whether the window counted its low bits.
__global__ void __launch_bounds__(kThreads) topk_top_scan_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    constexpr int kPer = kTopBins / kThreads;
    __shared__ unsigned long long ws[kThreads / 32];
    const int r = blockIdx.x, t = threadIdx.x;
    const unsigned long long *gh = p.top + (size_t)r * kTopBins;
    const TopkState st = gload<TopkState>(p.state + r); // read before the one write below
    unsigned long long c[kPer], s = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) { // thread t: bins kTopBins-1-t*kPer downwards
        c[j] = gload<unsigned long long>(gh + (kTopBins - 1 - (t * kPer + j)));
        s += c[j];
    }
    unsigned long long acc = cta_exclusive_scan(s, ws);
    if (acc < st.kr && st.kr <= acc + s) {
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (acc + c[j] >= st.kr) {
                TopkState n = st;
                n.prefix = (uint32_t)(kTopBins - 1 - (t * kPer + j));
                n.kr = st.kr - acc;
                const uint32_t w = n.prefix - st.wlo;
                n.hit = w < st.nwin ? 1u : 0u;
                n.region = n.hit ? w : (uint32_t)kWindowMax;
                gstore<TopkState>(p.state + r, n);
                break;
            }
            acc += c[j];
        }
    }
}

// The fallback when the window missed: clear the fallback histogram, then a
// second full pass counts the low bits of the chosen top bin into it.
__global__ void __launch_bounds__(kThreads) topk_fallback_clear_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    const int r = blockIdx.y;
    if (gload<TopkState>(p.state + r).hit)
        return;
    uint4 *low = reinterpret_cast<uint4 *>(low_region(p, r, kWindowMax));
    for (uint32_t i = blockIdx.x * kThreads + threadIdx.x; i < kLowBins / 4; i += gridDim.x * kThreads)
        gstore<uint4>(low + i, make_uint4(0, 0, 0, 0));
}

template <int DT>
__global__ void __launch_bounds__(kThreads) topk_fallback_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    const int r = blockIdx.y;
    const TopkState st = gload<TopkState>(p.state + r);
    if (st.hit)
        return;
    uint32_t *low = low_region(p, r, kWindowMax);
    for_each_key<DT>(p, r, [&](uint32_t key) {
        if ((key >> kLowBits) == st.prefix) {
            uint32_t *b = low + (key & (kLowBins - 1u));
            if (dbg_ok(b, sizeof(uint32_t)))
                atomicAdd(b, 1u);
        }
    });
}

// 4. Sum of each 2048-bin block of the low histogram that holds the k-th key.
__global__ void __launch_bounds__(kThreads) topk_low_sum_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    __shared__ unsigned long long ws[kThreads / 32];
    const int r = blockIdx.y, b = blockIdx.x;
    const uint32_t region = gload<TopkState>(p.state + r).region;
    const uint4 *q = reinterpret_cast<const uint4 *>(low_region(p, r, region) + (size_t)b * kLowPerBlock);
    unsigned long long s = 0;
    for (int i = threadIdx.x; i < kLowPerBlock / 4; i += kThreads) {
        const uint4 v = gload<uint4>(q + i);
        s += (unsigned long long)v.x + v.y + v.z + v.w;
    }
    const unsigned long long before = cta_exclusive_scan(s, ws);
    if (threadIdx.x == kThreads - 1)
        gstore<unsigned long long>(p.blk + (size_t)r * kLowBlocks + b, before + s);
}

// One CTA per rank: the block, then the bin within it, that holds the k-th
// key among the keys of the chosen top bin; tau = top digit : low bits.
__global__ void __launch_bounds__(kThreads) topk_low_scan_kernel(const __grid_constant__ TopkParams p)
{
    chain_entry();
    static_assert(kLowBlocks == kThreads, "one block sum per thread");
    constexpr int kPer = kLowPerBlock / kThreads;
    __shared__ unsigned long long ws[kThreads / 32];
    __shared__ int sel_block;
    __shared__ unsigned long long sel_kr;
    const int r = blockIdx.x, t = threadIdx.x;
    const TopkState st = gload<TopkState>(p.state + r);
    if (t == 0) {
        sel_block = -1;
        sel_kr = 0;
    }
    // blocks from the top: thread t takes block kLowBlocks-1-t
    const unsigned long long bs = gload<unsigned long long>(p.blk + (size_t)r * kLowBlocks + (kLowBlocks - 1 - t));
    const unsigned long long before = cta_exclusive_scan(bs, ws); // its barriers also order the stores above
    if (before < st.kr && st.kr <= before + bs) {
        sel_block = kLowBlocks - 1 - t;
        sel_kr = st.kr - before;
    }
    __syncthreads();
    const int B = sel_block;
    if (B < 0)
        return; // cannot happen when the histograms are consistent; tau keeps its initial value
    const uint32_t *low = low_region(p, r, st.region) + (size_t)B * kLowPerBlock;
    unsigned long long c[kPer], s = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        c[j] = gload<uint32_t>(low + (kLowPerBlock - 1 - (t * kPer + j)));
        s += c[j];
    }
    const unsigned long long kr = sel_kr;
    unsigned long long acc = cta_exclusive_scan(s, ws);
    if (acc < kr && kr <= acc + s) {
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (acc + c[j] >= kr) {
                const uint32_t bin = (uint32_t)B * kLowPerBlock + (uint32_t)(kLowPerBlock - 1 - (t * kPer + j));
                TopkState n = st;
                n.tau = (st.prefix << kLowBits) | bin;
                n.kr = kr - acc;
                gstore<TopkState>(p.state + r, n);
                gstore<uint32_t>(p.tau + r, n.tau);
                break;
            }
            acc += c[j];
        }
    }
}

size_t topk_work_bytes(int nranks)
{
    const size_t n = (size_t)nranks;
    return n * (kTopBins * sizeof(unsigned long long) + kTopBins * sizeof(uint32_t) +
                (size_t)kRegions * kLowBins * sizeof(uint32_t) + kLowBlocks * sizeof(unsigned long long) +
                sizeof(TopkState) + sizeof(uint32_t));
}

// The sample's density, one run in `every`: 16, or the sparsest of 32, 64 and
// 128 under which (a) the sample still expects kSampleTarget keys at or above
// the k-th, and (b) the sample's estimate of the k-th key's rank among all
// count keys, whose standard deviation is about sqrt(k every), stays within
// count / 2048.  (a) bounds the window's relative width in ranks; (b) keeps
// it narrow in values where k is a large share of the keys (near the median a
// band of ranks spans far more of a binade than in the tail).
static uint32_t sample_every(uint64_t count, uint64_t k)
{
    const uint64_t band = count / 2048; // count < 2^32: band^2 < 2^42
    uint32_t every = kSampleMin;
    while (every < kSampleMax && k / (2 * every) >= kSampleTarget && k * (2 * every) <= band * band)
        every *= 2;
    return every;
}

// The sample's size, and the order statistics that bound the window: the
// number of sampled keys at or above the k-th key is about k f (f the
// sampled fraction), with a standard deviation below sqrt(k f); five of them
// on each side.  false when the sample is too small to place a window.
static bool sample_bounds(uint64_t count, uint64_t k, uint32_t every, unsigned long long *qa, unsigned long long *qb)
{
    const uint64_t ng = count / 8, nruns = (ng + kRun - 1) / kRun;
    uint64_t groups = 0;
    for (uint64_t q = 0; q < nruns; q += every)
        groups += ng - q * kRun < (uint64_t)kRun ? ng - q * kRun : (uint64_t)kRun;
    const double nsamp = 8.0 * (double)groups;
    const double mean = (double)k * nsamp / (double)count;
    const double m = 5.0 * sqrt(mean) + 2.0;
    if (mean - m < 1.0 || mean + m > nsamp)
        return false;
    *qa = (unsigned long long)(mean - m);
    *qb = (unsigned long long)ceil(mean + m);
    return true;
}

uint32_t topk_sample_every(uint64_t count, uint64_t k)
{
    if (k == 0 || k >= count)
        return 0; // tau is final after the first launch
    const uint32_t every = sample_every(count, k);
    unsigned long long qa = 0, qb = 0;
    return sample_bounds(count, k, every, &qa, &qb) ? every : 0;
}

cudaError_t launch_topk_select(int dt, void *const *grads, float *const *res, int nranks, uint64_t count,
                               uint64_t k, void *work, const uint32_t **tau_out, cudaStream_t stream)
{
    if (nranks < 1 || nranks > kTopkMaxRanks)
        return cudaErrorInvalidValue;
    TopkParams p;
    bool vec = true;
    for (int r = 0; r < kTopkMaxRanks; ++r) {
        p.grads[r] = r < nranks ? grads[r] : nullptr;
        p.res[r] = r < nranks ? res[r] : nullptr;
        if (r < nranks)
            vec = vec && (uintptr_t)grads[r] % 16 == 0 && (uintptr_t)res[r] % 16 == 0;
    }
    const size_t n = (size_t)nranks;
    char *w = static_cast<char *>(work);
    p.top = reinterpret_cast<unsigned long long *>(w);
    w += n * kTopBins * sizeof(unsigned long long);
    p.stop = reinterpret_cast<uint32_t *>(w);
    w += n * kTopBins * sizeof(uint32_t);
    p.low = reinterpret_cast<uint32_t *>(w);
    w += n * kRegions * kLowBins * sizeof(uint32_t);
    p.blk = reinterpret_cast<unsigned long long *>(w);
    w += n * kLowBlocks * sizeof(unsigned long long);
    p.state = reinterpret_cast<TopkState *>(w);
    w += n * sizeof(TopkState);
    p.tau = reinterpret_cast<uint32_t *>(w);
    p.K = count;
    p.k = k;
    p.qa = p.qb = 0;
    p.every = sample_every(count, k);
    p.nranks = nranks;
    p.vec_ok = vec ? 1 : 0;
    *tau_out = p.tau;
    const bool select = k > 0 && k < count;
    topk_init_kernel<<<dim3(select ? kInitCtas : 1, (unsigned)nranks), kThreads, 0, stream>>>(p);
    count_launches(1);
    if (cudaError_t e = cudaGetLastError())
        return e;
    if (!select)
        return cudaSuccess; // tau is already final
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    // about eight resident CTAs per SM over all ranks, no more than the elements need
    const uint64_t items = (count / (vec ? 8 : 1) + kThreads - 1) / kThreads;
    uint64_t per_rank = (uint64_t)sms * 8 / (uint64_t)nranks;
    if (per_rank < 1)
        per_rank = 1;
    if (per_rank > items)
        per_rank = items > 0 ? items : 1;
    const dim3 grid((unsigned)per_rank, (unsigned)nranks);
    unsigned long long launches = 0;
    if (vec && sample_bounds(count, k, p.every, &p.qa, &p.qb)) {
        const uint64_t nruns = (count / 8 + kRun - 1) / kRun;
        const uint64_t swarps = (nruns + p.every - 1) / p.every;
        uint64_t sctas = (swarps + kThreads / 32 - 1) / (kThreads / 32);
        if (sctas > per_rank)
            sctas = per_rank;
        const dim3 sgrid((unsigned)sctas, (unsigned)nranks), block(kThreads), one((unsigned)nranks);
        cudaError_t e2 = launch_chained<TopkParams>(
            dt == DT_FP32 ? topk_sample_kernel<DT_FP32> : topk_sample_kernel<DT_BF16>, sgrid, block, 0, stream, p);
        if (e2 == cudaSuccess)
            e2 = launch_chained<TopkParams>(topk_window_kernel, one, block, 0, stream, p);
        if (e2 != cudaSuccess)
            return e2;
        launches += 2;
    }
    const bool f32 = dt == DT_FP32;
    const dim3 block(kThreads), one((unsigned)nranks);
    using K = void (*)(TopkParams);
    const K chain[] = {f32 ? topk_main_kernel<DT_FP32> : topk_main_kernel<DT_BF16>, topk_top_scan_kernel,
                       topk_fallback_clear_kernel, f32 ? topk_fallback_kernel<DT_FP32> : topk_fallback_kernel<DT_BF16>,
                       topk_low_sum_kernel, topk_low_scan_kernel};
    const dim3 grids[] = {grid, one, dim3(kInitCtas, (unsigned)nranks), grid, dim3(kLowBlocks, (unsigned)nranks), one};
    for (int i = 0; i < 6; ++i)
        if (cudaError_t e2 = launch_chained<TopkParams>(chain[i], grids[i], block, 0, stream, p))
            return e2;
    count_launches(launches + 6);
    return cudaGetLastError();
}

} // namespace ccl
