// step.cu -- step-faithful ring: one launch per ring step, for validating the
// schedule against the fused kernels.
//
// ReduceScatter phase, step s (Collectives and sharded matmul, "ring
// ReduceScatter"; Lesson 3 reference solution): rank i adds the chunk
// (i-1-s) mod N that rank i-1 sends into its own copy of that chunk.
// AllGather phase, step s: rank i stores chunk (i-s) mod N from rank i-1.
// Within one step the chunk a rank receives is never the chunk its right
// neighbour reads from it, so a step can run in place with no snapshot; the
// stream order between launches is the step barrier.
//
// Pre-multiplied AVG: rank i adds into chunk (i-1-s) only at step s, so its
// own copy is still the unscaled input then and is scaled as it is read; what
// arrives was scaled by its sender, except at step 0, where rank i-1 sends an
// untouched input chunk.  That scales every contribution exactly once without
// a separate pass over the buffers (N = 1, which has no steps, scales with
// one STEP_SCALE launch).

#include "ccl_internal.h"

namespace ccl {

// Incoming operand of a ReduceScatter hop: only at step 0 is it an input.
template <int DT, int OP> __device__ __forceinline__ uint32_t incoming_elem(uint32_t v, int s, float inv)
{
    return (OP == OP_AVGP && s == 0) ? pre_elem<DT, OP>(v, inv) : v;
}

template <int DT, int OP> __device__ __forceinline__ uint4 incoming_vec(const uint4 &v, int s, float inv)
{
    return (OP == OP_AVGP && s == 0) ? pre_vec<DT, OP>(v, inv) : v;
}

template <int DT, int OP, int MAXR>
__device__ __forceinline__ void step_elem(const StepParams<MAXR> &p, int kind, int i, int left, uint64_t e)
{
    if (kind == STEP_RS) {
        const uint32_t incoming = incoming_elem<DT, OP>(ld_elem<DT>(p.buf[left], e), p.s, p.inv_n);
        st_elem<DT>(p.buf[i], e, hop_elem<DT, OP>(pre_elem<DT, OP>(ld_elem<DT>(p.buf[i], e), p.inv_n), incoming));
    } else if (kind == STEP_SCALE) {
        const uint32_t v = ld_elem<DT>(p.buf[i], e);
        st_elem<DT>(p.buf[i], e, OP == OP_AVGP ? pre_elem<DT, OP>(v, p.inv_n) : avg_elem<DT>(v, p.n_f));
    } else {
        st_elem<DT>(p.buf[i], e, ld_elem<DT>(p.buf[left], e));
    }
}

template <int DT, int OP, int MAXR>
__global__ void __launch_bounds__(kThreads) ring_step_kernel(const __grid_constant__ StepParams<MAXR> p)
{
    chain_entry(); // every step after a phase's first is chained to the step before
    constexpr int VEC = DType<DT>::kVec;
    constexpr int U = 2;
    constexpr uint64_t TV = (uint64_t)kThreads * U;
    const int N = p.nranks;
    const int i = blockIdx.y;
    const int left = ring_mod(i - 1, N);
    const int kind = p.kind;
    int c;
    if (kind == STEP_RS || kind == STEP_AG_API)
        c = ring_mod(i - 1 - p.s, N);
    else if (kind == STEP_AG)
        c = ring_mod(i - p.s, N);
    else
        c = ring_mod(i + 1, N);
    const uint64_t off = p.part.off(c), end = off + p.part.len(c);
    const uint32_t t = blockIdx.x;

    if (!p.vec_aligned) {
        const uint64_t e0 = off + (uint64_t)t * TV * VEC;
        for (int k = 0; k < U * VEC; ++k) {
            const uint64_t e = e0 + (uint64_t)k * kThreads + threadIdx.x;
            if (e < end)
                step_elem<DT, OP, MAXR>(p, kind, i, left, e);
        }
        return;
    }
    const uint64_t vb = (off + VEC - 1) / VEC, ve = end / VEC;
    if (t == 0) {
        const uint64_t hb = vb < ve ? vb * VEC : end;
        for (uint64_t e = off + threadIdx.x; e < hb; e += kThreads)
            step_elem<DT, OP, MAXR>(p, kind, i, left, e);
        if (vb < ve)
            for (uint64_t e = ve * VEC + threadIdx.x; e < end; e += kThreads)
                step_elem<DT, OP, MAXR>(p, kind, i, left, e);
    }
    // all of this thread's loads first, then the hops and stores (the volatile
    // loads and stores keep program order, so they are batched by hand)
    uint4 mine[U], theirs[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint64_t v = vb + (uint64_t)t * TV + (uint64_t)u * kThreads + threadIdx.x;
        if (v < ve) {
            if (kind == STEP_RS || kind == STEP_SCALE)
                mine[u] = ld16(static_cast<const char *>(p.buf[i]) + v * 16);
            if (kind != STEP_SCALE)
                theirs[u] = ld16(static_cast<const char *>(p.buf[left]) + v * 16);
        }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint64_t v = vb + (uint64_t)t * TV + (uint64_t)u * kThreads + threadIdx.x;
        if (v < ve) {
            uint4 out;
            if (kind == STEP_RS)
                out = hop_vec<DT, OP>(pre_vec<DT, OP>(mine[u], p.inv_n), incoming_vec<DT, OP>(theirs[u], p.s, p.inv_n));
            else if (kind == STEP_SCALE)
                out = OP == OP_AVGP ? pre_vec<DT, OP>(mine[u], p.inv_n) : avg_vec<DT>(mine[u], p.n_f);
            else
                out = theirs[u];
            st16(static_cast<char *>(p.buf[i]) + v * 16, out);
        }
    }
}

template <int DT, int OP, int MAXR>
static cudaError_t launch_step_t(int kind, int s, void *const *bufs, int nranks, uint64_t count, cudaStream_t stream)
{
    constexpr int VEC = DType<DT>::kVec;
    StepParams<MAXR> p;
    bool aligned = true;
    for (int r = 0; r < nranks; ++r) {
        p.buf[r] = bufs[r];
        aligned = aligned && ((uintptr_t)bufs[r] % 16 == 0);
    }
    for (int r = nranks; r < MAXR; ++r)
        p.buf[r] = nullptr;
    p.part.q = count / (uint64_t)nranks;
    p.part.rem = (uint32_t)(count % (uint64_t)nranks);
    p.nranks = nranks;
    p.s = s;
    p.kind = kind;
    p.vec_aligned = aligned ? 1 : 0;
    p.n_f = (float)nranks;
    p.inv_n = 1.0f / (float)nranks;
    const uint64_t te = (uint64_t)kThreads * 2 * VEC;
    const uint64_t tiles = (p.part.q + 1 + te - 1) / te;
    if (tiles > 0x7fffffffull)
        return cudaErrorInvalidValue;
    p.tiles = (uint32_t)tiles;
    // A ring step depends on the step before it; every step but a phase's
    // first (which follows whatever the stream held) is a chained launch.  With
    // one rank there is no step before the scaling launch.
    const bool first = ((kind == STEP_RS || kind == STEP_AG_API) && s == 0) || nranks == 1;
    if (first) {
        ring_step_kernel<DT, OP, MAXR><<<dim3((unsigned)tiles, (unsigned)nranks), kThreads, 0, stream>>>(p);
    } else if (cudaError_t e = launch_chained<StepParams<MAXR>>(ring_step_kernel<DT, OP, MAXR>,
                                                                dim3((unsigned)tiles, (unsigned)nranks), dim3(kThreads),
                                                                0, stream, p)) {
        return e;
    }
    count_launches(1);
    return cudaGetLastError();
}

template <int DT, int OP>
static cudaError_t launch_step_op(int kind, int s, void *const *bufs, int nranks, uint64_t count,
                                  cudaStream_t stream)
{
    if (nranks <= kSmallRanks)
        return launch_step_t<DT, OP, kSmallRanks>(kind, s, bufs, nranks, count, stream);
    return launch_step_t<DT, OP, kMaxRanks>(kind, s, bufs, nranks, count, stream);
}

template <int DT>
static cudaError_t launch_step_dt(int op, int kind, int s, void *const *bufs, int nranks, uint64_t count,
                                  cudaStream_t stream)
{
    switch (op) {
    case OP_SUM: return launch_step_op<DT, OP_SUM>(kind, s, bufs, nranks, count, stream);
    case OP_AVG: return launch_step_op<DT, OP_AVG>(kind, s, bufs, nranks, count, stream);
    case OP_MAX: return launch_step_op<DT, OP_MAX>(kind, s, bufs, nranks, count, stream);
    case OP_PROD: return launch_step_op<DT, OP_PROD>(kind, s, bufs, nranks, count, stream);
    case OP_MIN: return launch_step_op<DT, OP_MIN>(kind, s, bufs, nranks, count, stream);
    case OP_AVGP: return launch_step_op<DT, OP_AVGP>(kind, s, bufs, nranks, count, stream);
    }
    return cudaErrorInvalidValue;
}

// Loads every ring-step kernel into the current device's context now rather
// than at its first launch (CUDA's default lazy loading), so that a later
// launch needs no device memory for code.
template <int DT, int OP> static cudaError_t preload_step_op()
{
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, ring_step_kernel<DT, OP, kSmallRanks>);
    return e != cudaSuccess ? e : cudaFuncGetAttributes(&a, ring_step_kernel<DT, OP, kMaxRanks>);
}

template <int DT> static cudaError_t preload_step_dt()
{
    const cudaError_t e[] = {preload_step_op<DT, OP_SUM>(), preload_step_op<DT, OP_AVG>(),
                             preload_step_op<DT, OP_MAX>(), preload_step_op<DT, OP_PROD>(),
                             preload_step_op<DT, OP_MIN>(), preload_step_op<DT, OP_AVGP>()};
    for (cudaError_t x : e)
        if (x != cudaSuccess)
            return x;
    return cudaSuccess;
}

cudaError_t preload_ring_step_kernels()
{
    const cudaError_t e = preload_step_dt<DT_FP32>();
    return e != cudaSuccess ? e : preload_step_dt<DT_BF16>();
}

// Elements each rank has sent in ring steps launched by this thread (Lesson 3's
// per-rank traffic counter): at ReduceScatter step s rank j sends chunk
// (j - s) mod N, at AllGather step s chunk (j + 1 - s) mod N, and in the
// AllGather entry point's steps (which start from chunk j at rank j) chunk
// (j - s) mod N.
static thread_local std::vector<unsigned long long> t_sent;

static void count_sent(int kind, int s, int nranks, uint64_t count)
{
    if (kind == STEP_SCALE)
        return;
    if (t_sent.size() < (size_t)nranks)
        t_sent.resize((size_t)nranks, 0ull);
    const uint64_t q = count / (uint64_t)nranks, rem = count % (uint64_t)nranks;
    const int shift = kind == STEP_AG ? 1 - s : -s;
    for (int j = 0; j < nranks; ++j) {
        const int c = ((j + shift) % nranks + nranks) % nranks;
        t_sent[(size_t)j] += q + ((uint64_t)c < rem ? 1 : 0);
    }
}

cudaError_t launch_ring_step(int dt, int op, int kind, int s, void *const *bufs, int nranks, uint64_t count,
                             cudaStream_t stream)
{
    // copies do not depend on the op: share one instantiation
    if (kind == STEP_AG || kind == STEP_AG_API)
        op = OP_SUM;
    const cudaError_t e = dt == DT_FP32 ? launch_step_dt<DT_FP32>(op, kind, s, bufs, nranks, count, stream)
                                        : launch_step_dt<DT_BF16>(op, kind, s, bufs, nranks, count, stream);
    if (e == cudaSuccess)
        count_sent(kind, s, nranks, count);
    return e;
}

} // namespace ccl

extern "C" ccl_status_t ccl_step_sent(int nranks, unsigned long long *sent, int reset)
{
    using ccl::t_sent;
    if (nranks < 1 || nranks > CCL_MAX_RANKS || !sent)
        return CCL_ERR_INVALID_ARG;
    for (int j = 0; j < nranks; ++j)
        sent[j] = (size_t)j < t_sent.size() ? t_sent[(size_t)j] : 0ull;
    if (reset)
        t_sent.assign(t_sent.size(), 0ull);
    return CCL_OK;
}
