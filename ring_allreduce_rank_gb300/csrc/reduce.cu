// reduce.cu -- the fused ring-order reduction: AllReduce and ReduceScatter in
// one pass over memory.
//
// The ring (Collectives and sharded matmul, "ring ReduceScatter": at step s
// rank i sends chunk (i-s) mod N right and the receiver adds it into its own
// copy) carries chunk c from rank c through c+1, ..., c-1, adding one
// contribution per hop.  Its end state is, per element of chunk c, the fold
//     R = x_{c-1} (+) ( ... (x_{c+1} (+) x_c))
// rounded to the buffer type after every hop, AVG dividing once by N (the
// pre-multiplied AVG instead scales every x_r by 1/N as it is loaded), and the
// AllGather phase (AllReduce survey, phase 2) copying R to every rank.  This
// kernel computes that end state directly: each element's N contributions are
// read once, folded in ring order in registers, and written once per rank --
// N*M bytes read and N*M written for AllReduce, the least any implementation
// can move, instead of the ~5(N-1)M bytes the step-by-step schedule moves.
//
// Work decomposition: grid (tiles, N); blockIdx.y is the chunk c, so the ring
// rotation start is uniform per CTA.  Inside a chunk, threads take 16-byte
// vectors (4 fp32 / 8 bf16) aligned to the buffers; the unaligned head and tail
// of each chunk are done element by element by the chunk's first CTA.  When a
// chunk's output cannot be vector-aligned (unaligned pointers, or a
// ReduceScatter chunk whose offset is not a multiple of the vector) the CTA
// walks its tile element by element instead.  The same kernel serves Reduce:
// the root receives the AllReduce's result and no other rank is written.
#include "fused.h"

namespace ccl {

// vectors per thread: enough 16-byte loads in flight per thread without
// spilling (N=8 with two vectors measured 0.6 % faster than one)
template <int NR> struct Unroll { static constexpr int kU = NR == 2 ? 4 : (NR <= 8 ? 2 : 1); };

// Element path: one element at a time, all ranks, ring order.
template <int DT, int OP, int MAXR>
__device__ __forceinline__ void reduce_elem(const FusedParams<MAXR> &p, int N, uint32_t c, uint64_t e,
                                            uint64_t out_base)
{
    int r = (int)c;
    uint32_t acc = pre_elem<DT, OP>(ld_elem<DT>(p.send[r], e), p.inv_n);
    for (int k = 1; k < N; ++k) {
        if (++r == N)
            r = 0;
        acc = hop_elem<DT, OP>(pre_elem<DT, OP>(ld_elem<DT>(p.send[r], e), p.inv_n), acc);
    }
    if (OP == OP_AVG)
        acc = avg_elem<DT>(acc, p.n_f);
    if (p.write_mode == WRITE_ALL) {
        for (int q = 0; q < N; ++q)
            st_elem<DT>(p.recv[q], e, acc);
    } else if (p.write_mode == WRITE_ROOT) {
        st_elem<DT>(p.recv[p.root], e, acc);
    } else {
        st_elem<DT>(p.recv[c], e - out_base, acc);
    }
}

// ReduceScatter chunk whose offset is not a whole vector: fold aligned input
// vectors, then build each (aligned) output vector from two neighbouring
// lanes' results.  A warp folds 32 input vectors and stores 31 output vectors.
template <int DT, int OP, int NR, int MAXR>
__device__ __forceinline__ void reduce_scatter_shifted(const FusedParams<MAXR> &p, int N, uint32_t c, uint64_t off,
                                                       uint64_t len, uint32_t t)
{
    constexpr int VEC = DType<DT>::kVec;
    constexpr int WARPS = kThreads / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t nout = len / VEC;            // whole output vectors
    const int d = (int)(off % VEC);             // misalignment in elements
    const uint64_t a0 = off / VEC;              // input vector holding the chunk's first element
    const uint64_t K = (uint64_t)p.part.q * (uint64_t)N + p.part.rem;
    const uint64_t j0 = ((uint64_t)t * WARPS + warp) * 31; // this warp's first output vector
    if (t == 0)  // the last, partial output vector
        for (uint64_t e = off + nout * VEC + threadIdx.x; e < off + len; e += kThreads)
            reduce_elem<DT, OP, MAXR>(p, N, c, e, off);
    if (j0 >= nout)
        return; // whole warp
    const uint64_t a = a0 + j0 + lane;
    uint4 r = make_uint4(0, 0, 0, 0);
    if ((a + 1) * VEC <= K) {
        r = ring_fold_vec<DT, OP, NR>(p.send, N, (int)c, a * 16, p.inv_n);
        if (OP == OP_AVG)
            r = avg_vec<DT>(r, p.n_f);
    } else {
        // the buffer's last, partial vector: elements past K stay zero (never stored)
        uint32_t h[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) {
            const uint64_t e = a * VEC + k;
            uint32_t v = 0;
            if (e < K) {
                v = ring_fold_elem<DT, OP>(p.send, N, (int)c, e, p.inv_n);
                if (OP == OP_AVG)
                    v = avg_elem<DT>(v, p.n_f);
            }
            h[k] = v;
        }
        if (DT == DT_FP32)
            r = make_uint4(h[0], h[1], h[2], h[3]);
        else
            r = make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
    }
    uint4 nx;
    nx.x = __shfl_down_sync(0xffffffffu, r.x, 1);
    nx.y = __shfl_down_sync(0xffffffffu, r.y, 1);
    nx.z = __shfl_down_sync(0xffffffffu, r.z, 1);
    nx.w = __shfl_down_sync(0xffffffffu, r.w, 1);
    const uint64_t j = j0 + lane;
    if (lane < 31 && j < nout)
        st16(static_cast<char *>(p.recv[c]) + j * 16, shift_window<DT>(r, nx, d));
}

// Many ranks, short chunks.  The paths below walk the ranks in groups, one
// round trip to memory per group, so a call's time grows with N even for a
// few elements per chunk.  Here one CTA per chunk first loads every rank's
// copy of its chunk into shared memory -- all N x len loads in flight at once --
// then folds each element from shared memory in ring order (the same hops,
// the same bits) and writes the results with independent stores.
constexpr uint64_t kSmallChunkMax = 64;           // elements per chunk
constexpr size_t kSmallChunkSmem = 48 * 1024;     // the default dynamic shared-memory limit

template <int DT, int OP, int MAXR>
__global__ void __launch_bounds__(kThreads) small_chunk_kernel(const __grid_constant__ FusedParams<MAXR> p)
{
    extern __shared__ uint32_t sx[]; // [N][L] input bits, then [L] results
    const int N = p.nranks;
    const uint32_t c = blockIdx.x;
    const uint64_t off = p.part.off(c);
    const int L = (int)p.part.len(c);
    if (L == 0)
        return;
    for (int i = threadIdx.x; i < N * L; i += kThreads) {
        const int r = i / L;
        sx[i] = pre_elem<DT, OP>(ld_elem<DT>(p.send[r], off + (uint64_t)(i - r * L)), p.inv_n);
    }
    __syncthreads();
    uint32_t *res = sx + (size_t)N * L;
    for (int e = threadIdx.x; e < L; e += kThreads) {
        // the ring order c, c+1, ..., N-1, 0, ..., c-1 as two linear runs, so
        // that unrolled reads of shared memory run ahead of the dependent hops
        uint32_t acc = sx[(int)c * L + e];
#pragma unroll 8
        for (int r = (int)c + 1; r < N; ++r)
            acc = hop_elem<DT, OP>(sx[r * L + e], acc);
#pragma unroll 8
        for (int r = 0; r < (int)c; ++r)
            acc = hop_elem<DT, OP>(sx[r * L + e], acc);
        if (OP == OP_AVG)
            acc = avg_elem<DT>(acc, p.n_f);
        res[e] = acc;
    }
    __syncthreads();
    if (p.write_mode == WRITE_ALL) {
        for (int i = threadIdx.x; i < N * L; i += kThreads) {
            const int r = i / L, e = i - r * L;
            st_elem<DT>(p.recv[r], off + (uint64_t)e, res[e]);
        }
    } else {
        for (int e = threadIdx.x; e < L; e += kThreads) {
            if (p.write_mode == WRITE_ROOT)
                st_elem<DT>(p.recv[p.root], off + (uint64_t)e, res[e]);
            else
                st_elem<DT>(p.recv[c], (uint64_t)e, res[e]);
        }
    }
}

template <int DT, int OP, int NR, int MAXR>
__global__ void __launch_bounds__(kThreads) fused_reduce_kernel(const __grid_constant__ FusedParams<MAXR> p)
{
    constexpr int VEC = DType<DT>::kVec;
    constexpr int ES = DType<DT>::kSize;
    constexpr int U = NR > 0 ? Unroll<NR>::kU : 1;
    constexpr uint64_t TV = (uint64_t)kThreads * U; // vectors per tile
    const int N = NR > 0 ? NR : p.nranks;
    const uint32_t c = blockIdx.y;
    const uint32_t t = blockIdx.x;
    const uint64_t off = p.part.off(c), len = p.part.len(c), end = off + len;
    const uint64_t out_base = p.write_mode == WRITE_CHUNK ? off : 0;
    const bool vec_ok = p.vec_aligned && (p.write_mode != WRITE_CHUNK || (off % VEC) == 0);

    if (p.vec_aligned && p.write_mode == WRITE_CHUNK && (off % VEC) != 0) {
        reduce_scatter_shifted<DT, OP, NR, MAXR>(p, N, c, off, len, t);
        return;
    }
    if (!vec_ok) {
        // element path over tile t of the chunk
        const uint64_t e0 = off + (uint64_t)t * TV * VEC;
#pragma unroll 4
        for (int i = 0; i < U * VEC; ++i) {
            const uint64_t e = e0 + (uint64_t)i * kThreads + threadIdx.x;
            if (e < end)
                reduce_elem<DT, OP, MAXR>(p, N, c, e, out_base);
        }
        return;
    }

    const uint64_t vb = (off + VEC - 1) / VEC, ve = end / VEC;
    if (t == 0) {
        // unaligned head and tail of the chunk (or all of a chunk shorter than a vector span)
        const uint64_t hb = vb < ve ? vb * VEC : end;
        for (uint64_t e = off + threadIdx.x; e < hb; e += kThreads)
            reduce_elem<DT, OP, MAXR>(p, N, c, e, out_base);
        if (vb < ve)
            for (uint64_t e = ve * VEC + threadIdx.x; e < end; e += kThreads)
                reduce_elem<DT, OP, MAXR>(p, N, c, e, out_base);
    }
    if (vb >= ve)
        return;
    const uint64_t v0 = vb + (uint64_t)t * TV + threadIdx.x;
    if (v0 >= ve)
        return;

    if (NR > 0) {
        // Exact rank count: every load of every rank for U vectors is issued
        // before the first hop, so a thread has U*N 16-byte loads in flight.
        uint4 x[U][NR > 0 ? NR : 1];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = v0 + (uint64_t)u * kThreads;
            if (v < ve) {
                int r = (int)c;
#pragma unroll
                for (int k = 0; k < NR; ++k) {
                    x[u][k] = ld16(static_cast<const char *>(p.send[r]) + v * 16);
                    r = (r + 1 == NR) ? 0 : r + 1;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint64_t v = v0 + (uint64_t)u * kThreads;
            if (v < ve) {
                uint4 acc = pre_vec<DT, OP>(x[u][0], p.inv_n);
#pragma unroll
                for (int k = 1; k < NR; ++k)
                    acc = hop_vec<DT, OP>(pre_vec<DT, OP>(x[u][k], p.inv_n), acc);
                if (OP == OP_AVG)
                    acc = avg_vec<DT>(acc, p.n_f);
                if (p.write_mode == WRITE_ALL) {
#pragma unroll
                    for (int q = 0; q < NR; ++q)
                        st16(static_cast<char *>(p.recv[q]) + v * 16, acc);
                } else if (p.write_mode == WRITE_ROOT) {
                    st16(static_cast<char *>(p.recv[p.root]) + v * 16, acc);
                } else {
                    st16(static_cast<char *>(p.recv[c]) + (v * VEC - out_base) * ES, acc);
                }
            }
        }
    } else {
        // Any rank count: ranks in groups of 8, the next group's loads issued
        // before the current group is folded.
        const uint64_t v = v0;
        uint4 acc = make_uint4(0, 0, 0, 0);
        uint4 cur[8], nxt[8];
        int r = (int)c;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            if (j < N) {
                cur[j] = ld16(static_cast<const char *>(p.send[r]) + v * 16);
                r = (r + 1 == N) ? 0 : r + 1;
            }
        }
        for (int g = 0; g < N; g += 8) {
            const int gn = g + 8;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (gn + j < N) {
                    nxt[j] = ld16(static_cast<const char *>(p.send[r]) + v * 16);
                    r = (r + 1 == N) ? 0 : r + 1;
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (g + j < N)
                    acc = (g + j == 0) ? pre_vec<DT, OP>(cur[0], p.inv_n)
                                       : hop_vec<DT, OP>(pre_vec<DT, OP>(cur[j], p.inv_n), acc);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j)
                cur[j] = nxt[j];
        }
        if (OP == OP_AVG)
            acc = avg_vec<DT>(acc, p.n_f);
        if (p.write_mode == WRITE_ALL) {
            for (int q = 0; q < N; ++q)
                st16(static_cast<char *>(p.recv[q]) + v * 16, acc);
        } else if (p.write_mode == WRITE_ROOT) {
            st16(static_cast<char *>(p.recv[p.root]) + v * 16, acc);
        } else {
            st16(static_cast<char *>(p.recv[c]) + (v * VEC - out_base) * ES, acc);
        }
    }
}

// ------------------------------------------------------------------ launch

template <int DT, int OP, int NR, int MAXR>
static cudaError_t launch_t(const void *const *send, void *const *recv, int nranks, uint64_t count, int write_mode,
                            int root, cudaStream_t stream)
{
    constexpr int VEC = DType<DT>::kVec;
    constexpr int U = NR > 0 ? Unroll<NR>::kU : 1;
    FusedParams<MAXR> p;
    bool aligned = true;
    for (int r = 0; r < nranks; ++r) {
        p.send[r] = send[r];
        // Reduce writes only the root's buffer: the others may be NULL
        p.recv[r] = (write_mode == WRITE_ROOT && r != root) ? nullptr : recv[r];
        aligned = aligned && ((uintptr_t)send[r] % 16 == 0) && ((uintptr_t)p.recv[r] % 16 == 0);
    }
    for (int r = nranks; r < MAXR; ++r) {
        p.send[r] = nullptr;
        p.recv[r] = nullptr;
    }
    p.part.q = count / (uint64_t)nranks;
    p.part.rem = (uint32_t)(count % (uint64_t)nranks);
    p.nranks = nranks;
    p.write_mode = write_mode;
    p.root = root;
    p.vec_aligned = aligned ? 1 : 0;
    p.n_f = (float)nranks;
    p.inv_n = 1.0f / (float)nranks;
    if (NR == 0 && nranks > kSmallRanks) {
        const uint64_t lmax = p.part.q + (p.part.rem ? 1 : 0);
        const size_t smem = ((size_t)nranks + 1) * (size_t)lmax * sizeof(uint32_t);
        if (lmax <= kSmallChunkMax && smem <= kSmallChunkSmem) {
            p.tiles = 1;
            small_chunk_kernel<DT, OP, MAXR><<<(unsigned)nranks, kThreads, smem, stream>>>(p);
            count_launches(1);
            return cudaGetLastError();
        }
    }
    const uint64_t te = (uint64_t)kThreads * U * VEC;
    uint64_t tiles = (p.part.q + 1 + te - 1) / te;
    // ReduceScatter chunks at offsets that are not whole vectors take the
    // shifted path (31 vectors per warp, about twice the tiles); size the grid
    // for it only when such a chunk exists
    bool ragged = false;
    for (int c = 1; c < nranks && write_mode == WRITE_CHUNK && aligned && !ragged; ++c)
        ragged = p.part.off((uint32_t)c) % VEC != 0;
    if (ragged) {
        const uint64_t per_tile = (uint64_t)(kThreads / 32) * 31;
        const uint64_t shifted = ((p.part.q + 1) / VEC + per_tile) / per_tile + 1;
        if (shifted > tiles)
            tiles = shifted;
    }
    if (tiles > 0x7fffffffull)
        return cudaErrorInvalidValue;
    p.tiles = (uint32_t)tiles;
    dim3 grid((unsigned)tiles, (unsigned)nranks);
    fused_reduce_kernel<DT, OP, NR, MAXR><<<grid, kThreads, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

template <int DT, int OP>
static cudaError_t launch_op(const void *const *send, void *const *recv, int nranks, uint64_t count, int write_mode,
                             int root, cudaStream_t stream)
{
    switch (nranks) {
    case 2: return launch_t<DT, OP, 2, kSmallRanks>(send, recv, nranks, count, write_mode, root, stream);
    case 4: return launch_t<DT, OP, 4, kSmallRanks>(send, recv, nranks, count, write_mode, root, stream);
    case 8: return launch_t<DT, OP, 8, kSmallRanks>(send, recv, nranks, count, write_mode, root, stream);
    case 16: return launch_t<DT, OP, 16, kSmallRanks>(send, recv, nranks, count, write_mode, root, stream);
    default:
        if (nranks <= kSmallRanks)
            return launch_t<DT, OP, 0, kSmallRanks>(send, recv, nranks, count, write_mode, root, stream);
        return launch_t<DT, OP, 0, kMaxRanks>(send, recv, nranks, count, write_mode, root, stream);
    }
}

template <int DT>
static cudaError_t launch_dt(int op, const void *const *send, void *const *recv, int nranks, uint64_t count,
                             int write_mode, int root, cudaStream_t stream)
{
    switch (op) {
    case OP_SUM: return launch_op<DT, OP_SUM>(send, recv, nranks, count, write_mode, root, stream);
    case OP_AVG: return launch_op<DT, OP_AVG>(send, recv, nranks, count, write_mode, root, stream);
    case OP_MAX: return launch_op<DT, OP_MAX>(send, recv, nranks, count, write_mode, root, stream);
    case OP_PROD: return launch_op<DT, OP_PROD>(send, recv, nranks, count, write_mode, root, stream);
    case OP_MIN: return launch_op<DT, OP_MIN>(send, recv, nranks, count, write_mode, root, stream);
    case OP_AVGP: return launch_op<DT, OP_AVGP>(send, recv, nranks, count, write_mode, root, stream);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_fused_reduce(int dt, int op, const void *const *send, void *const *recv, int nranks,
                                uint64_t count, int write_mode, int root, cudaStream_t stream)
{
    if (dt == DT_FP32)
        return launch_dt<DT_FP32>(op, send, recv, nranks, count, write_mode, root, stream);
    return launch_dt<DT_BF16>(op, send, recv, nranks, count, write_mode, root, stream);
}

} // namespace ccl
