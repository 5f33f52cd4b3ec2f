// bucket.cu -- bucket-fused gradient AllReduce without a staging buffer.
//
// DDP-style bucket fusion (Collective Communication, "Bucket fusion") lays the
// gradient tensors end to end in reverse registration order, cuts the stream
// into fixed-size buckets and AllReduces each bucket as one message, with the
// bucket's own N-chunk partition.  Instead of copying tensors into a bucket,
// reducing, and copying back (three passes), the planner cuts every (bucket,
// chunk) range at tensor boundaries into segments {tensor, rotation start c,
// offset, length}, and this kernel folds each segment in place where the
// tensors live: one read of every contribution and one write per rank, the
// same bytes as a single AllReduce of the whole stream.
#include <algorithm>
#include <unordered_map>
#include <vector>

#include "ccl_internal.h"

namespace ccl {

constexpr int kBucketPtrs = 1024; // tensor pointers per launch (8 KB)
constexpr int kBucketSegs = 700;  // segments per launch (22.4 KB)
constexpr uint32_t kSegVecFlag = 0x80000000u;

struct BucketParams {
    void *tp[kBucketPtrs]; // [local tensor][rank]
    RedSeg seg[kBucketSegs];
    uint64_t ntiles;
    uint32_t nseg;
    int nranks;
    float n_f;
    float inv_n; // 1/nranks correctly rounded (pre-multiplied AVG)
};

// One tile of one segment: fold its positions over the ranks in ring order
// (rotation start c) and write the result to every rank, in place.
template <int DT, int OP, int NR>
__device__ __forceinline__ void bucket_tile(const BucketParams &p, uint64_t tile)
{
    constexpr int VEC = DType<DT>::kVec;
    constexpr uint64_t TV = kThreads;
    uint32_t lo = 0, hi = p.nseg - 1;
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].tile_begin <= tile)
            lo = mid;
        else
            hi = mid - 1;
    }
    const RedSeg s = p.seg[lo];
    const uint64_t t = tile - s.tile_begin;
    const int N = NR > 0 ? NR : p.nranks;
    const int c = (int)(s.c & ~kSegVecFlag);
    const bool vec = (s.c & kSegVecFlag) != 0;
    const void *const *ptrs = p.tp + s.tp;
    const uint64_t off = s.off, end = s.off + s.len;

    auto do_elem = [&](uint64_t e) {
        uint32_t acc = ring_fold_elem<DT, OP>(ptrs, N, c, e, p.inv_n);
        if (OP == OP_AVG)
            acc = avg_elem<DT>(acc, p.n_f);
        for (int q = 0; q < N; ++q)
            st_elem<DT>(p.tp[s.tp + q], e, acc);
    };

    if (!vec) {
        const uint64_t e0 = off + t * TV * VEC;
        for (int k = 0; k < VEC; ++k) {
            const uint64_t e = e0 + (uint64_t)k * kThreads + threadIdx.x;
            if (e < end)
                do_elem(e);
        }
        return;
    }
    const uint64_t vb = (off + VEC - 1) / VEC, ve = end / VEC;
    if (t == 0) {
        const uint64_t hb = vb < ve ? vb * VEC : end;
        for (uint64_t e = off + threadIdx.x; e < hb; e += kThreads)
            do_elem(e);
        if (vb < ve)
            for (uint64_t e = ve * VEC + threadIdx.x; e < end; e += kThreads)
                do_elem(e);
    }
    const uint64_t v = vb + t * TV + threadIdx.x;
    if (v >= ve)
        return;
    uint4 acc = ring_fold_vec<DT, OP, NR>(ptrs, N, c, v * 16, p.inv_n);
    if (OP == OP_AVG)
        acc = avg_vec<DT>(acc, p.n_f);
    if (NR > 0) {
#pragma unroll
        for (int q = 0; q < NR; ++q)
            st16(static_cast<char *>(p.tp[s.tp + q]) + v * 16, acc);
    } else {
        for (int q = 0; q < N; ++q)
            st16(static_cast<char *>(p.tp[s.tp + q]) + v * 16, acc);
    }
}

// One CTA per tile, or -- with a capped grid, so that the reduction shares the
// GPU with other kernels instead of claiming every SM -- a grid-stride walk.
template <int DT, int OP, int NR>
__global__ void __launch_bounds__(kThreads) bucket_reduce_kernel(const __grid_constant__ BucketParams p)
{
    for (uint64_t tile = blockIdx.x; tile < p.ntiles; tile += gridDim.x)
        bucket_tile<DT, OP, NR>(p, tile);
}

template <int DT> static uint64_t seg_tiles(const RedSeg &s)
{
    constexpr int VEC = DType<DT>::kVec;
    if (s.c & kSegVecFlag) {
        const uint64_t vb = (s.off + VEC - 1) / VEC, ve = (s.off + s.len) / VEC;
        const uint64_t nv = ve > vb ? ve - vb : 0;
        const uint64_t t = (nv + kThreads - 1) / kThreads;
        return t ? t : 1;
    }
    const uint64_t te = (uint64_t)kThreads * VEC;
    const uint64_t t = (s.len + te - 1) / te;
    return t ? t : 1;
}

template <int DT, int OP>
static cudaError_t launch_batch(BucketParams &p, uint64_t tiles, int max_ctas, cudaStream_t stream)
{
    p.ntiles = tiles;
    if (max_ctas > 0 && tiles > (uint64_t)max_ctas)
        tiles = (uint64_t)max_ctas;
    if (tiles > 0x7fffffffull)
        return cudaErrorInvalidValue;
    if (p.nranks == 8)
        bucket_reduce_kernel<DT, OP, 8><<<(unsigned)tiles, kThreads, 0, stream>>>(p);
    else if (p.nranks == 4)
        bucket_reduce_kernel<DT, OP, 4><<<(unsigned)tiles, kThreads, 0, stream>>>(p);
    else
        bucket_reduce_kernel<DT, OP, 0><<<(unsigned)tiles, kThreads, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

template <int DT, int OP>
static cudaError_t launch_bucket_t(void *const *tensor_ptrs, int ntensors, int nranks, const RedSeg *segs,
                                   size_t nseg, int max_ctas, cudaStream_t stream)
{
    (void)ntensors;
    std::vector<char> storage(sizeof(BucketParams));
    BucketParams &p = *reinterpret_cast<BucketParams *>(storage.data());
    std::unordered_map<uint32_t, uint32_t> local; // global tensor -> local pointer base
    auto reset = [&]() {
        local.clear();
        p.nseg = 0;
        p.nranks = nranks;
        p.n_f = (float)nranks;
        p.inv_n = 1.0f / (float)nranks;
    };
    reset();
    uint32_t nptr = 0;
    uint64_t tiles = 0;
    for (size_t i = 0; i < nseg; ++i) {
        const RedSeg &g = segs[i];
        if (g.len == 0)
            continue;
        bool have = local.count(g.tp) != 0;
        if (p.nseg == (uint32_t)kBucketSegs || (!have && nptr + (uint32_t)nranks > (uint32_t)kBucketPtrs)) {
            cudaError_t e = launch_batch<DT, OP>(p, tiles, max_ctas, stream);
            if (e != cudaSuccess)
                return e;
            reset();
            nptr = 0;
            tiles = 0;
            have = false;
        }
        uint32_t base;
        if (!have) {
            base = nptr;
            for (int r = 0; r < nranks; ++r)
                p.tp[nptr + r] = tensor_ptrs[(size_t)g.tp * nranks + r];
            local[g.tp] = base;
            nptr += (uint32_t)nranks;
        } else {
            base = local[g.tp];
        }
        bool aligned = true;
        for (int r = 0; r < nranks; ++r)
            aligned = aligned && ((uintptr_t)p.tp[base + r] % 16 == 0);
        RedSeg sg = g;
        sg.tp = base;
        sg.c = g.c | (aligned ? kSegVecFlag : 0u);
        sg.tile_begin = tiles;
        tiles += seg_tiles<DT>(sg);
        p.seg[p.nseg++] = sg;
    }
    if (p.nseg)
        return launch_batch<DT, OP>(p, tiles, max_ctas, stream);
    return cudaSuccess;
}

template <int DT>
static cudaError_t launch_bucket_dt(int op, void *const *tp, int nt, int nr, const RedSeg *s, size_t ns, int mc,
                                    cudaStream_t st)
{
    switch (op) {
    case OP_SUM: return launch_bucket_t<DT, OP_SUM>(tp, nt, nr, s, ns, mc, st);
    case OP_AVG: return launch_bucket_t<DT, OP_AVG>(tp, nt, nr, s, ns, mc, st);
    case OP_MAX: return launch_bucket_t<DT, OP_MAX>(tp, nt, nr, s, ns, mc, st);
    case OP_PROD: return launch_bucket_t<DT, OP_PROD>(tp, nt, nr, s, ns, mc, st);
    case OP_MIN: return launch_bucket_t<DT, OP_MIN>(tp, nt, nr, s, ns, mc, st);
    case OP_AVGP: return launch_bucket_t<DT, OP_AVGP>(tp, nt, nr, s, ns, mc, st);
    }
    return cudaErrorInvalidValue;
}

void build_bucket_plan(const size_t *numels, int ntensors, int nranks, size_t B, BucketPlan &plan)
{
    const size_t T = (size_t)ntensors;
    plan.pos.assign(T, 0);
    plan.total = 0;
    for (size_t k = T; k-- > 0;) { // reverse registration order
        plan.pos[k] = plan.total;
        plan.total += numels[k];
    }
    std::vector<size_t> order; // non-empty tensors in stream order
    for (size_t k = T; k-- > 0;)
        if (numels[k])
            order.push_back(k);
    plan.start.clear();
    plan.segs.clear();
    plan.tensors.clear();
    size_t oi = 0;
    for (size_t b0 = 0; b0 < plan.total; b0 += B) {
        const size_t blen = std::min(B, plan.total - b0);
        Partition part;
        part.q = blen / (uint64_t)nranks;
        part.rem = (uint32_t)(blen % (uint64_t)nranks);
        std::vector<RedSeg> segs;
        std::vector<int> ts;
        for (int c = 0; c < nranks; ++c) {
            size_t lo = b0 + part.off((uint32_t)c);
            const size_t hi = lo + part.len((uint32_t)c);
            while (lo < hi) {
                while (plan.pos[order[oi]] + numels[order[oi]] <= lo)
                    ++oi;
                const size_t t = order[oi];
                const size_t e = std::min(hi, plan.pos[t] + numels[t]);
                segs.push_back(RedSeg{(uint32_t)t, (uint32_t)c, lo - plan.pos[t], e - lo, 0});
                if (ts.empty() || ts.back() != (int)t)
                    if (std::find(ts.begin(), ts.end(), (int)t) == ts.end())
                        ts.push_back((int)t);
                lo = e;
            }
        }
        plan.start.push_back(b0);
        plan.segs.push_back(std::move(segs));
        plan.tensors.push_back(std::move(ts));
    }
    plan.start.push_back(plan.total);
}

cudaError_t launch_bucket_reduce(int dt, int op, void *const *tensor_ptrs, int ntensors, int nranks,
                                 const RedSeg *segs, size_t nseg, cudaStream_t stream, int max_ctas)
{
    if (nranks > kBucketPtrs)
        return cudaErrorInvalidValue;
    if (dt == DT_FP32)
        return launch_bucket_dt<DT_FP32>(op, tensor_ptrs, ntensors, nranks, segs, nseg, max_ctas, stream);
    return launch_bucket_dt<DT_BF16>(op, tensor_ptrs, ntensors, nranks, segs, nseg, max_ctas, stream);
}

} // namespace ccl
