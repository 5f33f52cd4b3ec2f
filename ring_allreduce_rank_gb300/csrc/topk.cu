// topk.cu -- the threshold of Top-k sparsification, found on the device.
//
// Top-k ("Top-k sparsification", Collective Communication) sends, per rank,
// the values of u = g + e whose magnitude reaches the k-th largest magnitude
// |u|_(k), every tie included, and keeps the rest as residual.  Magnitudes are
// ordered as the bit patterns of |u| (the sign bit cleared): for numbers that
// is the order of |u|, and a NaN lands above every number.  The k-th largest
// 31-bit key tau is found by a radix select in three digit passes (11, 11 and
// 9 bits, most significant first).  Each pass re-forms u from g and e, counts
// the keys that agree with the digits fixed so far in a 2048-bin histogram
// (shared-memory atomics per CTA, merged into a 64-bit histogram per rank),
// and a one-CTA-per-rank scan walks the bins from the top to the bin holding
// the k-th key, fixing the next digit and the rank of the key within it.
// After the third pass tau is exact.  The compressed AllReduce kernel then
// sends u where key(u) >= tau, in the same pass that writes the residuals and
// folds the sent values in ring order.
//
// Everything stays on the device and in the caller's work buffer, so a call
// never waits for the host and can be captured in a CUDA graph.
#include "ccl_internal.h"

namespace ccl {

constexpr int kTopkBins = 2048;

struct TopkState {
    uint32_t prefix;        // digits fixed so far
    uint32_t tau;           // the k-th largest key, once all digits are fixed
    unsigned long long kr;  // rank (1-based) of the k-th key among keys that match prefix
};

struct TopkParams {
    const void *grads[kTopkMaxRanks];
    const float *res[kTopkMaxRanks];
    unsigned long long *hist; // [nranks][kTopkBins]
    TopkState *state;         // [nranks]
    uint32_t *tau;            // [nranks], read by the compressed kernel
    uint64_t K;
    unsigned long long k;
    int nranks;
    int pass;   // 0, 1, 2
    int vec_ok; // every gradient and residual 16-byte aligned
};

// Digit layout of the 31-bit key: pass 0 takes bits 30..20, pass 1 bits
// 19..9, pass 2 bits 8..0.  Keys enter a pass's histogram only when the bits
// above its digit equal the prefix fixed by the earlier passes.
__host__ __device__ __forceinline__ int topk_shift(int pass) { return pass == 0 ? 20 : (pass == 1 ? 9 : 0); }
__host__ __device__ __forceinline__ int topk_bits(int pass) { return pass == 2 ? 9 : 11; }

__device__ __forceinline__ uint32_t topk_key(float g, float e) { return __float_as_uint(__fadd_rn(g, e)) & 0x7fffffffu; }

__device__ __forceinline__ void topk_count(uint32_t *h, uint32_t key, int pass, uint32_t prefix)
{
    const int sh = topk_shift(pass);
    const uint32_t above = pass == 0 ? 0u : key >> (sh + topk_bits(pass));
    if (above == prefix)
        atomicAdd(&h[(key >> sh) & ((1u << topk_bits(pass)) - 1u)], 1u);
}

__global__ void __launch_bounds__(kThreads) topk_init_kernel(const __grid_constant__ TopkParams p)
{
    const int r = blockIdx.x;
    for (int i = threadIdx.x; i < kTopkBins; i += kThreads)
        gstore<unsigned long long>(p.hist + (size_t)r * kTopkBins + i, 0ull);
    if (threadIdx.x == 0) {
        TopkState s;
        s.prefix = 0;
        s.kr = p.k;
        // k = 0: no key reaches tau, nothing is sent; k >= K: every key does
        s.tau = p.k == 0 ? 0xffffffffu : 0u;
        gstore<TopkState>(p.state + r, s);
        gstore<uint32_t>(p.tau + r, s.tau);
    }
}

template <int DT>
__global__ void __launch_bounds__(kThreads) topk_hist_kernel(const __grid_constant__ TopkParams p)
{
    __shared__ uint32_t h[kTopkBins];
    for (int i = threadIdx.x; i < kTopkBins; i += kThreads)
        h[i] = 0u;
    __syncthreads();
    const int r = blockIdx.y, pass = p.pass;
    const uint32_t prefix = pass == 0 ? 0u : gload<TopkState>(p.state + r).prefix;
    const void *g = p.grads[r];
    const float *e = p.res[r];
    const uint64_t K = p.K;
    const uint64_t ng = p.vec_ok ? K / 8 : 0; // whole groups of 8 elements
    for (uint64_t gi = (uint64_t)blockIdx.x * kThreads + threadIdx.x; gi < ng; gi += (uint64_t)gridDim.x * kThreads) {
        float gv[8];
        if (DT == DT_BF16) {
            const uint4 w = gload<uint4>(static_cast<const uint16_t *>(g) + gi * 8);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                gv[2 * j] = __uint_as_float(ws[j] << 16);
                gv[2 * j + 1] = __uint_as_float(ws[j] & 0xffff0000u);
            }
        } else {
            const float4 a = gload<float4>(static_cast<const float *>(g) + gi * 8);
            const float4 b = gload<float4>(static_cast<const float *>(g) + gi * 8 + 4);
            gv[0] = a.x; gv[1] = a.y; gv[2] = a.z; gv[3] = a.w;
            gv[4] = b.x; gv[5] = b.y; gv[6] = b.z; gv[7] = b.w;
        }
        const float4 ea = gload<float4>(e + gi * 8), eb = gload<float4>(e + gi * 8 + 4);
        const float ev[8] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
#pragma unroll
        for (int j = 0; j < 8; ++j)
            topk_count(h, topk_key(gv[j], ev[j]), pass, prefix);
    }
    // the elements no whole group covers (all of them when a buffer is unaligned)
    for (uint64_t i = ng * 8 + (uint64_t)blockIdx.x * kThreads + threadIdx.x; i < K; i += (uint64_t)gridDim.x * kThreads) {
        const uint32_t b = ld_elem<DT>(g, i);
        topk_count(h, topk_key(__uint_as_float(DT == DT_BF16 ? b << 16 : b), gload<float>(e + i)), pass, prefix);
    }
    __syncthreads();
    unsigned long long *gh = p.hist + (size_t)r * kTopkBins;
    for (int i = threadIdx.x; i < kTopkBins; i += kThreads)
        if (h[i] && dbg_ok(gh + i, sizeof(unsigned long long)))
            atomicAdd(gh + i, (unsigned long long)h[i]);
}

// One CTA per rank: walk this pass's bins from the largest digit down to the
// one where the running count reaches kr; fix that digit, take the counts
// above it off kr, and clear the histogram for the next pass.
__global__ void __launch_bounds__(kThreads) topk_scan_kernel(const __grid_constant__ TopkParams p)
{
    constexpr int kPer = kTopkBins / kThreads; // bins per thread (pass 2 uses the first quarter of them)
    __shared__ unsigned long long warp_sum[kThreads / 32];
    const int r = blockIdx.x, pass = p.pass, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int nb = 1 << topk_bits(pass), per = nb / kThreads;
    unsigned long long *gh = p.hist + (size_t)r * kTopkBins;
    // read before the barriers below: one thread rewrites it after them
    const TopkState st = gload<TopkState>(p.state + r);
    // thread t holds bins nb-1-t*per ... nb-per-t*per (descending)
    unsigned long long c[kPer];
    unsigned long long s = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        c[j] = j < per ? gload<unsigned long long>(gh + (nb - 1 - (t * per + j))) : 0ull;
        s += c[j];
    }
    __syncthreads(); // every count is read before any is cleared
#pragma unroll
    for (int j = 0; j < kPer; ++j)
        if (j < per)
            gstore<unsigned long long>(gh + (nb - 1 - (t * per + j)), 0ull);
    // exclusive scan of s in thread order (descending bins)
    unsigned long long incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        warp_sum[warp] = incl;
    __syncthreads();
    unsigned long long base = 0;
    for (int w = 0; w < warp; ++w)
        base += warp_sum[w];
    const unsigned long long excl = base + incl - s;
    if (excl < st.kr && st.kr <= excl + s) {
        unsigned long long acc = excl;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            if (j < per && acc + c[j] >= st.kr) {
                const uint32_t digit = (uint32_t)(nb - 1 - (t * per + j));
                TopkState n;
                n.prefix = (st.prefix << topk_bits(pass)) | digit;
                n.kr = st.kr - acc;
                n.tau = pass == 2 ? n.prefix : st.tau;
                gstore<TopkState>(p.state + r, n);
                if (pass == 2)
                    gstore<uint32_t>(p.tau + r, n.prefix);
                break;
            }
            acc += c[j];
        }
    }
}

size_t topk_work_bytes(int nranks)
{
    const size_t n = (size_t)nranks;
    return n * kTopkBins * sizeof(unsigned long long) + n * sizeof(TopkState) + n * sizeof(uint32_t);
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
    char *w = static_cast<char *>(work);
    p.hist = reinterpret_cast<unsigned long long *>(w);
    p.state = reinterpret_cast<TopkState *>(w + (size_t)nranks * kTopkBins * sizeof(unsigned long long));
    p.tau = reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(p.state) + (size_t)nranks * sizeof(TopkState));
    p.K = count;
    p.k = k;
    p.nranks = nranks;
    p.pass = 0;
    p.vec_ok = vec ? 1 : 0;
    *tau_out = p.tau;
    topk_init_kernel<<<(unsigned)nranks, kThreads, 0, stream>>>(p);
    count_launches(1);
    if (cudaError_t e = cudaGetLastError())
        return e;
    if (k == 0 || k >= count)
        return cudaSuccess; // tau is already final
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
        return e;
    // about eight resident CTAs per SM over all ranks, no more than the elements need
    const uint64_t groups = (count / (vec ? 8 : 1) + kThreads - 1) / kThreads;
    uint64_t per_rank = (uint64_t)sms * 8 / (uint64_t)nranks;
    if (per_rank < 1)
        per_rank = 1;
    if (per_rank > groups)
        per_rank = groups > 0 ? groups : 1;
    for (int pass = 0; pass < 3; ++pass) {
        p.pass = pass;
        if (dt == DT_FP32)
            topk_hist_kernel<DT_FP32><<<dim3((unsigned)per_rank, (unsigned)nranks), kThreads, 0, stream>>>(p);
        else
            topk_hist_kernel<DT_BF16><<<dim3((unsigned)per_rank, (unsigned)nranks), kThreads, 0, stream>>>(p);
        topk_scan_kernel<<<(unsigned)nranks, kThreads, 0, stream>>>(p);
        count_launches(2);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

} // namespace ccl
