// orders.cu -- AllReduce under the pages' other schedules, computed in one
// pass: each schedule fixes a different summation order, so each gives its
// own bits, and this kernel reproduces them exactly.
//
//   halving-doubling (Collective Communication, "Recursive halving-doubling
//     (butterfly)"; Distributed LLM collectives, "Recursive Halving-Doubling"):
//     round k pairs i with i XOR 2^k, k = 0, 1, ...  For p not a power of two,
//     the first 2r ranks (r = p - 2^floor(log2 p)) are first added pairwise,
//     (2v, 2v+1).  Per element this is a balanced binary tree over the
//     "virtual" leaves, adjacent leaves first.
//   binomial tree (Collective Communication, "Tree AllReduce"): level k adds
//     rank i + 2^k into rank i; per element a binomial tree over the ranks in
//     order, the root's subtrees joined smallest first.
//   two-level hierarchical (AllReduce survey, two-level table): ring
//     ReduceScatter inside groups of L consecutive ranks, ring AllReduce among
//     the G = N/L group representatives, ring AllGather inside the groups.
//     Per element: a ring fold over groups, starting at group d, of ring folds
//     inside each group starting at local rank c (c: the element's intra
//     chunk, d: its sub-chunk inside chunk c).
//
// The trees are evaluated with a binary counter of partial sums: after leaf
// number n, level j holds a partial iff bit j of n is set; a new leaf carries
// through the set bits.  The counter's slots are fully unrolled, so they live
// in registers.  N a power of two (where both trees coincide) has a
// compile-time version for N in {2, 4, 8, 16}.
#include "ccl_internal.h"

namespace ccl {

constexpr int kLevels = 11; // 2^10 = 1024 ranks

template <int MAXR> struct OrderParams {
    const void *send[MAXR];
    void *recv[MAXR];
    uint64_t K;
    int nranks;
    int algo;     // ALGO_HD, ALGO_TREE, ALGO_HIER
    int L, G;     // hierarchical: ranks per group, groups
    int vec_aligned;
    float n_f;
};

// ------------------------------------------------------------------ value-generic helpers

template <int DT, int OP> struct VecOps {
    using V = uint4;
    static __device__ __forceinline__ V load(const void *base, uint64_t i) { return ld16(static_cast<const char *>(base) + i * 16); }
    static __device__ __forceinline__ void store(void *base, uint64_t i, const V &v) { st16(static_cast<char *>(base) + i * 16, v); }
    static __device__ __forceinline__ V hop(const V &a, const V &b) { return hop_vec<DT, OP>(a, b); }
    static __device__ __forceinline__ V avg(const V &v, float n) { return avg_vec<DT>(v, n); }
};

template <int DT, int OP> struct ElemOps {
    using V = uint32_t;
    static __device__ __forceinline__ V load(const void *base, uint64_t i) { return ld_elem<DT>(base, i); }
    static __device__ __forceinline__ void store(void *base, uint64_t i, V v) { st_elem<DT>(base, i, v); }
    static __device__ __forceinline__ V hop(V a, V b) { return hop_elem<DT, OP>(a, b); }
    static __device__ __forceinline__ V avg(V v, float n) { return avg_elem<DT>(v, n); }
};

// Binary counter of partial sums.
template <class O> struct Counter {
    typename O::V slot[kLevels];
    uint32_t n = 0;
    __device__ __forceinline__ void push(typename O::V carry)
    {
        bool open = true;
#pragma unroll
        for (int j = 0; j < kLevels; ++j) {
            if (open) {
                if (n & (1u << j)) {
                    carry = O::hop(slot[j], carry); // earlier partial on the left
                } else {
                    slot[j] = carry;
                    open = false;
                }
            }
        }
        ++n;
    }
    // join what is left, smallest level first (the binomial tree's order)
    __device__ __forceinline__ typename O::V finish()
    {
        typename O::V acc{};
        bool have = false;
#pragma unroll
        for (int j = 0; j < kLevels; ++j) {
            if (n & (1u << j)) {
                acc = have ? O::hop(slot[j], acc) : slot[j];
                have = true;
            }
        }
        return acc;
    }
};

// Balanced tree over x[lo, lo + n), n a power of two, adjacent leaves first.
template <class O, int N, int LO> struct Balanced {
    static __device__ __forceinline__ typename O::V eval(const typename O::V *x)
    {
        return O::hop(Balanced<O, N / 2, LO>::eval(x), Balanced<O, N / 2, LO + N / 2>::eval(x));
    }
};
template <class O, int LO> struct Balanced<O, 1, LO> {
    static __device__ __forceinline__ typename O::V eval(const typename O::V *x) { return x[LO]; }
};

// ------------------------------------------------------------------ one position, any value type

template <class O, int NR, int MAXR>
__device__ __forceinline__ typename O::V fold_tree(const OrderParams<MAXR> &p, uint64_t i)
{
    using V = typename O::V;
    if constexpr (NR > 0) {
        // N a power of two: halving-doubling and the binomial tree coincide
        V x[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r)
            x[r] = O::load(p.send[r], i);
        return Balanced<O, NR, 0>::eval(x);
    } else {
        const int N = p.nranks;
        Counter<O> ctr;
        if (p.algo == ALGO_HD) {
            int pw = 1;
            while (pw * 2 <= N)
                pw *= 2;
            const int r = N - pw;
            for (int v = 0; v < pw; ++v) {
                V leaf;
                if (v < r)
                    leaf = O::hop(O::load(p.send[2 * v + 1], i), O::load(p.send[2 * v], i));
                else
                    leaf = O::load(p.send[v + r], i);
                ctr.push(leaf);
            }
        } else {
            V next = O::load(p.send[0], i);
            for (int r = 0; r < N; ++r) {
                const V cur = next;
                if (r + 1 < N)
                    next = O::load(p.send[r + 1], i); // next leaf in flight while this one is folded
                ctr.push(cur);
            }
        }
        return ctr.finish();
    }
}

template <class O, int NL, int MAXR>
__device__ __forceinline__ typename O::V fold_hier(const OrderParams<MAXR> &p, uint64_t i, int c, int d)
{
    using V = typename O::V;
    const int L = NL > 0 ? NL : p.L, G = p.G;
    V acc{};
    for (int k = 0; k < G; ++k) {
        const int g = (d + k) % G;
        const void *const *grp = p.send + g * L;
        V part;
        if constexpr (NL > 0) {
            V x[NL > 0 ? NL : 1];
            int r = c;
#pragma unroll
            for (int j = 0; j < NL; ++j) {
                x[j] = O::load(grp[r], i);
                r = (r + 1 == NL) ? 0 : r + 1;
            }
            part = x[0];
#pragma unroll
            for (int j = 1; j < NL; ++j)
                part = O::hop(x[j], part);
        } else {
            int r = c;
            part = O::load(grp[r], i);
            for (int j = 1; j < L; ++j) {
                r = (r + 1 == L) ? 0 : r + 1;
                part = O::hop(O::load(grp[r], i), part);
            }
        }
        acc = k == 0 ? part : O::hop(part, acc);
    }
    return acc;
}

template <class O, int NR, int MAXR>
__device__ __forceinline__ void finish_store(const OrderParams<MAXR> &p, uint64_t i, typename O::V acc, int op)
{
    const int N = NR > 0 ? NR : p.nranks;
    if (op == OP_AVG)
        acc = O::avg(acc, p.n_f);
    for (int q = 0; q < N; ++q)
        O::store(p.recv[q], i, acc);
}

// ------------------------------------------------------------------ kernels

// halving-doubling / binomial tree: the order does not depend on the position
template <int DT, int OP, int NR, int MAXR>
__global__ void __launch_bounds__(kThreads) tree_order_kernel(const __grid_constant__ OrderParams<MAXR> p)
{
    constexpr int VEC = DType<DT>::kVec;
    const uint64_t nv = p.vec_aligned ? p.K / VEC : 0;
    const uint64_t v = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    if (v < nv)
        finish_store<VecOps<DT, OP>, NR>(p, v, fold_tree<VecOps<DT, OP>, NR>(p, v), OP);
    // elements not covered by whole vectors: the tail, or everything when unaligned
    const uint64_t e0 = nv * VEC;
    const uint64_t per_block = (uint64_t)kThreads * VEC;
    for (uint64_t e = e0 + (uint64_t)blockIdx.x * per_block + threadIdx.x;
         e < p.K && e < e0 + ((uint64_t)blockIdx.x + 1) * per_block; e += kThreads)
        finish_store<ElemOps<DT, OP>, NR>(p, e, fold_tree<ElemOps<DT, OP>, NR>(p, e), OP);
}

// hierarchical: blockIdx.y = segment (c, d); the segment's positions share c, d
template <int DT, int OP, int NL, int MAXR>
__global__ void __launch_bounds__(kThreads) hier_order_kernel(const __grid_constant__ OrderParams<MAXR> p)
{
    constexpr int VEC = DType<DT>::kVec;
    const int L = NL > 0 ? NL : p.L, G = p.G;
    const int c = blockIdx.y / G, d = blockIdx.y % G;
    Partition outer{p.K / (uint64_t)L, (uint32_t)(p.K % (uint64_t)L)};
    const uint64_t lc = outer.len(c);
    Partition inner{lc / (uint64_t)G, (uint32_t)(lc % (uint64_t)G)};
    const uint64_t off = outer.off(c) + inner.off(d), end = off + inner.len(d);
    const uint64_t t = blockIdx.x;
    using VO = VecOps<DT, OP>;
    using EO = ElemOps<DT, OP>;
    if (!p.vec_aligned) {
        for (int k = 0; k < VEC; ++k) {
            const uint64_t e = off + t * kThreads * VEC + (uint64_t)k * kThreads + threadIdx.x;
            if (e < end)
                finish_store<EO, 0>(p, e, fold_hier<EO, NL>(p, e, c, d), OP);
        }
        return;
    }
    const uint64_t vb = (off + VEC - 1) / VEC, ve = end / VEC;
    if (t == 0) {
        const uint64_t hb = vb < ve ? vb * VEC : end;
        for (uint64_t e = off + threadIdx.x; e < hb; e += kThreads)
            finish_store<EO, 0>(p, e, fold_hier<EO, NL>(p, e, c, d), OP);
        if (vb < ve)
            for (uint64_t e = ve * VEC + threadIdx.x; e < end; e += kThreads)
                finish_store<EO, 0>(p, e, fold_hier<EO, NL>(p, e, c, d), OP);
    }
    const uint64_t v = vb + t * kThreads + threadIdx.x;
    if (v < ve)
        finish_store<VO, 0>(p, v, fold_hier<VO, NL>(p, v, c, d), OP);
}

// ------------------------------------------------------------------ launch

template <int DT, int OP, int MAXR>
static cudaError_t launch_order_t(int algo, int L, const void *const *send, void *const *recv, int nranks,
                                  uint64_t count, cudaStream_t stream)
{
    constexpr int VEC = DType<DT>::kVec;
    OrderParams<MAXR> p;
    bool aligned = true;
    for (int r = 0; r < MAXR; ++r) {
        p.send[r] = r < nranks ? send[r] : nullptr;
        p.recv[r] = r < nranks ? recv[r] : nullptr;
        if (r < nranks)
            aligned = aligned && (uintptr_t)send[r] % 16 == 0 && (uintptr_t)recv[r] % 16 == 0;
    }
    p.K = count;
    p.nranks = nranks;
    p.algo = algo;
    p.L = algo == ALGO_HIER ? L : 1;
    p.G = algo == ALGO_HIER ? nranks / L : 1;
    p.vec_aligned = aligned ? 1 : 0;
    p.n_f = (float)nranks;
    if (algo == ALGO_HIER) {
        const uint64_t seg = count / (uint64_t)nranks + 2; // longest segment
        const uint64_t tiles = aligned ? (seg / VEC + 2 + kThreads - 1) / kThreads
                                       : (seg + (uint64_t)kThreads * VEC - 1) / ((uint64_t)kThreads * VEC);
        if (tiles > 0x7fffffffull)
            return cudaErrorInvalidValue;
        const dim3 grid((unsigned)(tiles ? tiles : 1), (unsigned)nranks);
        switch (L) {
        case 2: hier_order_kernel<DT, OP, 2, MAXR><<<grid, kThreads, 0, stream>>>(p); break;
        case 4: hier_order_kernel<DT, OP, 4, MAXR><<<grid, kThreads, 0, stream>>>(p); break;
        case 8: hier_order_kernel<DT, OP, 8, MAXR><<<grid, kThreads, 0, stream>>>(p); break;
        default: hier_order_kernel<DT, OP, 0, MAXR><<<grid, kThreads, 0, stream>>>(p); break;
        }
    } else {
        // one thread per vector, and each CTA also takes its share of the tail
        const uint64_t nv = aligned ? count / VEC : 0;
        const uint64_t rest = count - nv * VEC;
        uint64_t blocks = (nv + kThreads - 1) / kThreads;
        const uint64_t tail_blocks = (rest + (uint64_t)kThreads * VEC - 1) / ((uint64_t)kThreads * VEC);
        if (tail_blocks > blocks)
            blocks = tail_blocks;
        if (blocks == 0)
            blocks = 1;
        if (blocks > 0x7fffffffull)
            return cudaErrorInvalidValue;
        const bool pow2 = (nranks & (nranks - 1)) == 0;
        switch (pow2 ? nranks : 0) {
        case 2: tree_order_kernel<DT, OP, 2, MAXR><<<(unsigned)blocks, kThreads, 0, stream>>>(p); break;
        case 4: tree_order_kernel<DT, OP, 4, MAXR><<<(unsigned)blocks, kThreads, 0, stream>>>(p); break;
        case 8: tree_order_kernel<DT, OP, 8, MAXR><<<(unsigned)blocks, kThreads, 0, stream>>>(p); break;
        case 16: tree_order_kernel<DT, OP, 16, MAXR><<<(unsigned)blocks, kThreads, 0, stream>>>(p); break;
        default: tree_order_kernel<DT, OP, 0, MAXR><<<(unsigned)blocks, kThreads, 0, stream>>>(p); break;
        }
    }
    count_launches(1);
    return cudaGetLastError();
}

template <int DT, int OP>
static cudaError_t launch_order_op(int algo, int L, const void *const *s, void *const *r, int n, uint64_t k,
                                   cudaStream_t st)
{
    if (n <= kSmallRanks)
        return launch_order_t<DT, OP, kSmallRanks>(algo, L, s, r, n, k, st);
    return launch_order_t<DT, OP, kMaxRanks>(algo, L, s, r, n, k, st);
}

template <int DT>
static cudaError_t launch_order_dt(int op, int algo, int L, const void *const *s, void *const *r, int n, uint64_t k,
                                   cudaStream_t st)
{
    switch (op) {
    case OP_SUM: return launch_order_op<DT, OP_SUM>(algo, L, s, r, n, k, st);
    case OP_AVG: return launch_order_op<DT, OP_AVG>(algo, L, s, r, n, k, st);
    case OP_MAX: return launch_order_op<DT, OP_MAX>(algo, L, s, r, n, k, st);
    case OP_PROD: return launch_order_op<DT, OP_PROD>(algo, L, s, r, n, k, st);
    case OP_MIN: return launch_order_op<DT, OP_MIN>(algo, L, s, r, n, k, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_order_allreduce(int dt, int op, int algo, int group, const void *const *send, void *const *recv,
                                   int nranks, uint64_t count, cudaStream_t stream)
{
    if (dt == DT_FP32)
        return launch_order_dt<DT_FP32>(op, algo, group, send, recv, nranks, count, stream);
    return launch_order_dt<DT_BF16>(op, algo, group, send, recv, nranks, count, stream);
}

} // namespace ccl
