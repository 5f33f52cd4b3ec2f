// copy.cu -- the data-movement collectives: AllGather and Broadcast fan-out
// (read each source element once, write it to every rank) and segment copies
// (AllToAll / AllToAllv blocks, step-mode placement, bucket packing).
#include <algorithm>
#include <vector>

#include "ccl_internal.h"

namespace ccl {

// ------------------------------------------------------------------ segment copies

constexpr uint64_t kCopyTileBytes = (uint64_t)kThreads * 4 * 16; // 16 KiB of body per CTA

// 32-byte vector load / store (sm_100 and later); p must be 32-byte aligned
__device__ __forceinline__ void ld32(const void *p, uint4 &a, uint4 &b)
{
    a = b = make_uint4(0, 0, 0, 0);
    if (dbg_ok(p, 32))
        asm volatile("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                     : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
                     : "l"(p));
}

__device__ __forceinline__ void st32(void *p, const uint4 &a, const uint4 &b)
{
    if (dbg_ok(p, 32))
        asm volatile("st.global.L1::no_allocate.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(a.x),
                     "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
                     : "memory");
}

template <int MAXS> struct CopyParams {
    uint32_t nseg;
    uint32_t pad;
    CopySeg seg[MAXS];
};

// Alignment class of a segment: the widest power of two (<= 32) dividing the
// distance between source and destination; the body is moved in words of that
// width, aligned on the destination.
__host__ __device__ __forceinline__ uint32_t copy_grain(const char *src, const char *dst)
{
    const uintptr_t d = (uintptr_t)src ^ (uintptr_t)dst;
    if ((d & 31) == 0) return 32;
    if ((d & 15) == 0) return 16;
    if ((d & 7) == 0) return 8;
    if ((d & 3) == 0) return 4;
    if ((d & 1) == 0) return 2;
    return 1;
}

__host__ __device__ __forceinline__ void copy_split(const CopySeg &s, uint32_t g, uint64_t &head, uint64_t &body)
{
    const uint64_t mis = (uintptr_t)s.dst & (g - 1);
    head = mis ? umin64(g - mis, s.nbytes) : 0;
    body = (s.nbytes - head) / g * g;
}

__host__ __device__ __forceinline__ uint64_t copy_tiles(const CopySeg &s)
{
    uint64_t head, body;
    copy_split(s, copy_grain(s.src, s.dst), head, body);
    const uint64_t t = (body + kCopyTileBytes - 1) / kCopyTileBytes;
    return t ? t : 1;
}

template <typename W>
__device__ __forceinline__ void copy_body(const char *src, char *dst, uint64_t nbytes)
{
    const uint64_t n = nbytes / sizeof(W);
    const W *s = reinterpret_cast<const W *>(src);
    W *d = reinterpret_cast<W *>(dst);
    for (uint64_t i = threadIdx.x; i < n; i += kThreads)
        gstore<W>(d + i, gload<W>(s + i));
}

template <int MAXS>
__global__ void __launch_bounds__(kThreads) copy_segments_kernel(const __grid_constant__ CopyParams<MAXS> p)
{
    uint32_t lo = 0, hi = p.nseg - 1;
    while (lo < hi) {
        const uint32_t mid = (lo + hi + 1) >> 1;
        if (p.seg[mid].tile_begin <= blockIdx.x)
            lo = mid;
        else
            hi = mid - 1;
    }
    const CopySeg s = p.seg[lo];
    const uint64_t t = blockIdx.x - s.tile_begin;
    const uint32_t g = copy_grain(s.src, s.dst);
    uint64_t head, body;
    copy_split(s, g, head, body);
    if (t == 0) {
        for (uint64_t b = threadIdx.x; b < head; b += kThreads)
            gstore<char>(s.dst + b, gload<char>(s.src + b));
        for (uint64_t b = head + body + threadIdx.x; b < s.nbytes; b += kThreads)
            gstore<char>(s.dst + b, gload<char>(s.src + b));
    }
    const uint64_t b0 = t * kCopyTileBytes;
    if (b0 >= body)
        return;
    const uint64_t nb = umin64(kCopyTileBytes, body - b0);
    const char *src = s.src + head + b0;
    char *dst = s.dst + head + b0;
    if (g == 32) {
        // two 32-byte loads in flight per thread before the stores
        constexpr int B = 2;
        const uint64_t n = nb / 32;
        for (uint64_t i0 = threadIdx.x; i0 < n; i0 += (uint64_t)B * kThreads) {
            uint4 x[B], y[B];
#pragma unroll
            for (int k = 0; k < B; ++k) {
                const uint64_t i = i0 + (uint64_t)k * kThreads;
                if (i < n)
                    ld32(src + i * 32, x[k], y[k]);
            }
#pragma unroll
            for (int k = 0; k < B; ++k) {
                const uint64_t i = i0 + (uint64_t)k * kThreads;
                if (i < n)
                    st32(dst + i * 32, x[k], y[k]);
            }
        }
    } else if (g == 16) {
        // four 16-byte loads in flight per thread before the stores (the
        // volatile loads and stores keep program order, so they are batched
        // by hand)
        constexpr int B = 4;
        const uint64_t n = nb / 16;
        for (uint64_t i0 = threadIdx.x; i0 < n; i0 += (uint64_t)B * kThreads) {
            uint4 x[B];
#pragma unroll
            for (int k = 0; k < B; ++k) {
                const uint64_t i = i0 + (uint64_t)k * kThreads;
                if (i < n)
                    x[k] = ld16(src + i * 16);
            }
#pragma unroll
            for (int k = 0; k < B; ++k) {
                const uint64_t i = i0 + (uint64_t)k * kThreads;
                if (i < n)
                    st16(dst + i * 16, x[k]);
            }
        }
    } else if (g == 8) {
        copy_body<uint2>(src, dst, nb);
    } else if (g == 4) {
        copy_body<uint32_t>(src, dst, nb);
    } else if (g == 2) {
        copy_body<uint16_t>(src, dst, nb);
    } else {
        copy_body<uint8_t>(src, dst, nb);
    }
}

template <int MAXS>
static cudaError_t launch_copy_batch(const CopySeg *segs, size_t nseg, cudaStream_t stream)
{
    CopyParams<MAXS> p;
    p.nseg = (uint32_t)nseg;
    p.pad = 0;
    uint64_t tiles = 0;
    for (size_t i = 0; i < nseg; ++i) {
        p.seg[i] = segs[i];
        p.seg[i].tile_begin = tiles;
        tiles += copy_tiles(segs[i]);
    }
    if (tiles > 0x7fffffffull)
        return cudaErrorInvalidValue;
    copy_segments_kernel<MAXS><<<(unsigned)tiles, kThreads, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

// Parameter-block tiers: every launch carries its segment table, and a 32 KB
// block costs the GPU's front end microseconds per launch (AllToAllv over 8
// ranks, 64 segments: 140 us per call with the large block, 135 in a graph)
constexpr size_t kCopySegsSmall = 16;
constexpr size_t kCopySegsMid = 128;    // 4 KB: AllToAll(v) up to 11 ranks
constexpr size_t kCopySegsLarge = 1000; // 32 KB of kernel parameters

cudaError_t launch_copy_segments(const CopySeg *segs, size_t nseg, cudaStream_t stream)
{
    std::vector<CopySeg> live;
    live.reserve(nseg);
    for (size_t i = 0; i < nseg; ++i)
        if (segs[i].nbytes)
            live.push_back(segs[i]);
    size_t i = 0;
    while (i < live.size()) {
        const size_t n = std::min(kCopySegsLarge, live.size() - i);
        cudaError_t e = n <= kCopySegsSmall ? launch_copy_batch<kCopySegsSmall>(live.data() + i, n, stream)
                        : n <= kCopySegsMid ? launch_copy_batch<kCopySegsMid>(live.data() + i, n, stream)
                                            : launch_copy_batch<kCopySegsLarge>(live.data() + i, n, stream);
        if (e != cudaSuccess)
            return e;
        i += n;
    }
    return cudaSuccess;
}

cudaError_t preload_copy_kernels()
{
    cudaFuncAttributes a;
    cudaError_t e = cudaFuncGetAttributes(&a, copy_segments_kernel<kCopySegsSmall>);
    if (e == cudaSuccess)
        e = cudaFuncGetAttributes(&a, copy_segments_kernel<kCopySegsMid>);
    return e != cudaSuccess ? e : cudaFuncGetAttributes(&a, copy_segments_kernel<kCopySegsLarge>);
}

// ------------------------------------------------------------------ fan-out (AllGather, Broadcast)

template <int MAXR> struct FanoutParams {
    const void *src[MAXR];
    void *dst[MAXR];
    Partition part;  // chunking of the destination buffers
    int nchunks;     // sources (AllGather: N, Broadcast: 1)
    int ndst;
    int vec_aligned; // every pointer 16-byte aligned
    int vec32;       // every pointer 32-byte aligned
};

// Threads per CTA of the fan-out kernel.
constexpr int kFanThreads = kThreads;
// Shared memory each fan-out CTA reserves and does not use: with 228 KB per
// SM (1 KB of it per resident CTA) it holds the kernel to seven resident CTAs
// per SM, whatever its register count.  Measured, Gather (8 sources into one
// buffer) at N = 8, 128 MiB: 0.880 of the copy rate at eight CTAs per SM,
// 0.913-0.917 at seven, 0.903 at six, 0.874 at five; Broadcast and the ragged
// AllGather move by less than 0.4 % between five and seven, and lose 0.4-0.8 %
// at eight.  The segment copy is fastest at eight (Scatter 0.879 against 0.860
// at seven).
constexpr size_t kFanOccupancySmem = 31 * 1024;

// Eight words (one 32-byte vector) of the sixteen in w (two neighbouring
// 32-byte vectors), starting d elements in, 0 < d < 2 * (elements a 16-byte
// vector holds).
template <int DT> __device__ __forceinline__ void shift_window32(const uint32_t (&w)[16], int d, uint32_t (&o)[8])
{
    if (DT == DT_FP32) {
#define CCL_W32(D)                                                                                                     \
    case D:                                                                                                            \
        _Pragma("unroll") for (int i = 0; i < 8; ++i) o[i] = w[D + i];                                                 \
        break;
        switch (d) {
            CCL_W32(1) CCL_W32(2) CCL_W32(3) CCL_W32(4) CCL_W32(5) CCL_W32(6)
        default:
            _Pragma("unroll") for (int i = 0; i < 8; ++i) o[i] = w[7 + i];
        }
#undef CCL_W32
    } else {
        // d halfwords: whole words d/2, then half a word if d is odd
#define CCL_H32(D)                                                                                                     \
    case D:                                                                                                            \
        _Pragma("unroll") for (int i = 0; i < 8; ++i) o[i] =                                                           \
            (D & 1) ? __funnelshift_r(w[(D >> 1) + i], w[(D >> 1) + i + 1], 16) : w[(D >> 1) + i];                     \
        break;
        switch (d) {
            CCL_H32(1) CCL_H32(2) CCL_H32(3) CCL_H32(4) CCL_H32(5) CCL_H32(6) CCL_H32(7) CCL_H32(8) CCL_H32(9)
            CCL_H32(10) CCL_H32(11) CCL_H32(12) CCL_H32(13) CCL_H32(14)
        default:
            _Pragma("unroll") for (int i = 0; i < 8; ++i) o[i] = __funnelshift_r(w[7 + i], w[8 + i], 16);
        }
#undef CCL_H32
    }
}

// The ragged fan-out with 32-byte vectors (every buffer 32-byte aligned, the
// chunk at an offset that is not a whole 16-byte vector).  Each lane loads the
// two aligned 32-byte source vectors that its destination vector spans; the
// destination vector is the window s1 elements into that pair.  The second
// vector is the next lane's first, so L2 serves each source vector twice
// (DRAM once); loads are one vector in N + 1 of the traffic, and taking the
// neighbour's vector by shuffle instead queued 8 shuffles per vector in front
// of the stores (0.45 % slower at N = 16).  As in the 16-byte form, a warp
// writes 32 destination vectors that start on a multiple of 32, and the
// chunk's unaligned head and tail go element by element.
template <int DT, int MAXR>
__device__ __forceinline__ void fanout_ragged32(const FanoutParams<MAXR> &p, uint32_t t, uint64_t off, uint64_t len,
                                                const void *src, int M)
{
    constexpr int V2 = 2 * DType<DT>::kVec; // elements per 32-byte vector
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t vb = (off + V2 - 1) / V2, ve = (off + len) / V2;
    const int s1 = (int)(vb * V2 - off); // 0 < s1 < V2
    if (t == 0) {
        const uint64_t hb = vb < ve ? vb * V2 : off + len;
        for (uint64_t d = off + threadIdx.x; d < hb; d += kFanThreads) {
            const uint32_t v = ld_elem<DT>(src, d - off);
            for (int q = 0; q < M; ++q)
                st_elem<DT>(p.dst[q], d, v);
        }
        if (vb < ve)
            for (uint64_t d = ve * V2 + threadIdx.x; d < off + len; d += kFanThreads) {
                const uint32_t v = ld_elem<DT>(src, d - off);
                for (int q = 0; q < M; ++q)
                    st_elem<DT>(p.dst[q], d, v);
            }
    }
    if (vb >= ve)
        return;
    // this lane's destination vector; whole warps past the end leave together
    const uint64_t v = (vb / 32 + (uint64_t)t * (kFanThreads / 32) + warp) * 32 + lane;
    if (v - lane >= ve)
        return;
    // source vector b (32 bytes) feeds destination vectors vb + b - 1 and vb + b
    auto load_src = [&](int64_t b, uint32_t *h) {
        if (b < 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                h[k] = 0u;
        } else if ((uint64_t)(b + 1) * V2 <= len) {
            uint4 a, c;
            ld32(static_cast<const char *>(src) + (uint64_t)b * 32, a, c);
            h[0] = a.x; h[1] = a.y; h[2] = a.z; h[3] = a.w;
            h[4] = c.x; h[5] = c.y; h[6] = c.z; h[7] = c.w;
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                h[k] = 0u;
            for (int k = 0; k < V2; ++k) {
                const uint64_t e = (uint64_t)b * V2 + k;
                const uint32_t x = e < len ? ld_elem<DT>(src, e) : 0u;
                if (DT == DT_FP32)
                    h[k] = x;
                else
                    h[k >> 1] |= x << (16 * (k & 1));
            }
        }
    };
    const int64_t b = (int64_t)v - (int64_t)vb;
    if (v >= vb && v < ve) {
        uint32_t w[16];
        load_src(b, w);
        load_src(b + 1, w + 8);
        uint32_t o[8];
        shift_window32<DT>(w, s1, o);
        const uint4 a = make_uint4(o[0], o[1], o[2], o[3]), c = make_uint4(o[4], o[5], o[6], o[7]);
        for (int q = 0; q < M; ++q)
            st32(static_cast<char *>(p.dst[q]) + v * 32, a, c);
    }
}

template <int DT, int MAXR>
__global__ void __launch_bounds__(kFanThreads) fanout_kernel(const __grid_constant__ FanoutParams<MAXR> p)
{
    constexpr int VEC = DType<DT>::kVec;
    constexpr int U = 2;
    constexpr uint64_t TV = (uint64_t)kFanThreads * U;
    const uint32_t c = blockIdx.y, t = blockIdx.x;
    const uint64_t off = p.part.off(c), len = p.part.len(c);
    const void *src = p.src[c];
    const int M = p.ndst;
    if (p.vec32 && off % VEC != 0) {
        fanout_ragged32<DT, MAXR>(p, t, off, len, src, M);
        return;
    }
    if (p.vec_aligned && off % VEC != 0) {
        // The chunk lands at an offset that is not a whole vector (ragged
        // partition).  Lanes load aligned source vectors; each aligned
        // destination vector is the window s0 elements into two neighbouring
        // source vectors, exchanged with a shuffle (lane 31 loads the one
        // after its own).  A warp writes 32 destination vectors that start on
        // a multiple of 32 vectors, so every warp store covers whole 512-byte
        // blocks (3 % faster than windows at arbitrary starts).
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const uint64_t vb = (off + VEC - 1) / VEC, ve = (off + len) / VEC;
        const int s0 = (int)(vb * VEC - off); // 0 < s0 < VEC
        if (t == 0) {
            const uint64_t hb = vb < ve ? vb * VEC : off + len;
            for (uint64_t d = off + threadIdx.x; d < hb; d += kFanThreads) {
                const uint32_t v = ld_elem<DT>(src, d - off);
                for (int q = 0; q < M; ++q)
                    st_elem<DT>(p.dst[q], d, v);
            }
            if (vb < ve)
                for (uint64_t d = ve * VEC + threadIdx.x; d < off + len; d += kFanThreads) {
                    const uint32_t v = ld_elem<DT>(src, d - off);
                    for (int q = 0; q < M; ++q)
                        st_elem<DT>(p.dst[q], d, v);
                }
        }
        if (vb >= ve)
            return;
        // this lane's destination vector; whole warps past the end leave together
        const uint64_t v = (vb / 32 + (uint64_t)t * (kFanThreads / 32) + warp) * 32 + lane;
        if (v - lane >= ve)
            return;
        // source vector b feeds destination vectors vb + b - 1 and vb + b
        auto load_src = [&](int64_t b) -> uint4 {
            if (b < 0)
                return make_uint4(0, 0, 0, 0);
            if ((uint64_t)(b + 1) * VEC <= len)
                return ld16(static_cast<const char *>(src) + (uint64_t)b * 16);
            uint32_t h[VEC];
#pragma unroll
            for (int k = 0; k < VEC; ++k)
                h[k] = (uint64_t)b * VEC + k < len ? ld_elem<DT>(src, (uint64_t)b * VEC + k) : 0u;
            if (DT == DT_FP32)
                return make_uint4(h[0], h[1], h[2], h[3]);
            return make_uint4(h[0] | h[1] << 16, h[2] | h[3] << 16, h[4] | h[5] << 16, h[6] | h[7] << 16);
        };
        const int64_t b = (int64_t)v - (int64_t)vb;
        const uint4 x = load_src(b);
        const uint4 next = lane == 31 ? load_src(b + 1) : make_uint4(0, 0, 0, 0);
        uint4 nx;
        nx.x = __shfl_down_sync(0xffffffffu, x.x, 1);
        nx.y = __shfl_down_sync(0xffffffffu, x.y, 1);
        nx.z = __shfl_down_sync(0xffffffffu, x.z, 1);
        nx.w = __shfl_down_sync(0xffffffffu, x.w, 1);
        if (lane == 31)
            nx = next;
        if (v >= vb && v < ve) {
            const uint4 w = shift_window<DT>(x, nx, s0);
            for (int q = 0; q < M; ++q)
                st16(static_cast<char *>(p.dst[q]) + v * 16, w);
        }
        return;
    }
    if (!(p.vec_aligned && off % VEC == 0)) {
        const uint64_t e0 = (uint64_t)t * TV * VEC;
        for (int k = 0; k < U * VEC; ++k) {
            const uint64_t e = e0 + (uint64_t)k * kFanThreads + threadIdx.x;
            if (e < len) {
                const uint32_t v = ld_elem<DT>(src, e);
                for (int q = 0; q < M; ++q)
                    st_elem<DT>(p.dst[q], off + e, v);
            }
        }
        return;
    }
    if (p.vec32 && off % (2 * VEC) == 0) {
        // 32-byte vectors: one per thread, a warp covering 1 KiB contiguous
        const uint64_t nw = len / (2 * VEC);
        if (t == 0)
            for (uint64_t e = nw * 2 * VEC + threadIdx.x; e < len; e += kFanThreads) {
                const uint32_t v = ld_elem<DT>(src, e);
                for (int q = 0; q < M; ++q)
                    st_elem<DT>(p.dst[q], off + e, v);
            }
        const uint64_t w = (uint64_t)t * kFanThreads + threadIdx.x;
        if (w < nw) {
            uint4 a, b;
            ld32(static_cast<const char *>(src) + w * 32, a, b);
            for (int q = 0; q < M; ++q)
                st32(static_cast<char *>(p.dst[q]) + off * DType<DT>::kSize + w * 32, a, b);
        }
        return;
    }
    const uint64_t nv = len / VEC;
    if (t == 0)
        for (uint64_t e = nv * VEC + threadIdx.x; e < len; e += kFanThreads) {
            const uint32_t v = ld_elem<DT>(src, e);
            for (int q = 0; q < M; ++q)
                st_elem<DT>(p.dst[q], off + e, v);
        }
    uint4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint64_t v = (uint64_t)t * TV + (uint64_t)u * kFanThreads + threadIdx.x;
        if (v < nv)
            x[u] = ld16(static_cast<const char *>(src) + v * 16);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint64_t v = (uint64_t)t * TV + (uint64_t)u * kFanThreads + threadIdx.x;
        if (v < nv)
            for (int q = 0; q < M; ++q)
                st16(static_cast<char *>(p.dst[q]) + (off + v * VEC) * DType<DT>::kSize, x[u]);
    }
}

template <int DT, int MAXR>
static cudaError_t launch_fanout_t(const void *const *src, int nchunks, void *const *dst, int ndst, uint64_t count,
                                   cudaStream_t stream)
{
    constexpr int VEC = DType<DT>::kVec;
    FanoutParams<MAXR> p;
    bool aligned = true, aligned32 = true;
    for (int i = 0; i < MAXR; ++i) {
        p.src[i] = i < nchunks ? src[i] : nullptr;
        p.dst[i] = i < ndst ? dst[i] : nullptr;
        if (i < nchunks) {
            aligned = aligned && (uintptr_t)src[i] % 16 == 0;
            aligned32 = aligned32 && (uintptr_t)src[i] % 32 == 0;
        }
        if (i < ndst) {
            aligned = aligned && (uintptr_t)dst[i] % 16 == 0;
            aligned32 = aligned32 && (uintptr_t)dst[i] % 32 == 0;
        }
    }
    p.part.q = count / (uint64_t)nchunks;
    p.part.rem = (uint32_t)(count % (uint64_t)nchunks);
    p.nchunks = nchunks;
    p.ndst = ndst;
    p.vec_aligned = aligned ? 1 : 0;
    p.vec32 = aligned32 ? 1 : 0;
    // a tile: kFanThreads x 32 bytes (two 16-byte vectors per thread, or one 32-byte one)
    const uint64_t te = (uint64_t)kFanThreads * 2 * VEC;
    uint64_t tiles = (p.part.q + 1 + te - 1) / te;
    // A chunk whose offset is not a whole vector takes the shuffle path (one
    // vector per thread) and needs about twice as many tiles; size the grid for
    // it only when such a chunk exists, or the aligned chunks launch as many
    // empty CTAs as working ones.
    bool ragged = false;
    for (int c = 1; c < nchunks && aligned && !ragged; ++c)
        ragged = p.part.off((uint32_t)c) % VEC != 0;
    // ragged path: kFanThreads destination vectors (32-byte ones when every
    // buffer allows) per tile, the first block starting up to 31 vectors
    // before the chunk
    const uint64_t per_tile = (uint64_t)kFanThreads;
    const uint64_t shifted = ((p.part.q + 1) / (aligned32 ? 2 * VEC : VEC) + 31 + per_tile) / per_tile + 1;
    if (ragged && shifted > tiles)
        tiles = shifted;
    if (tiles > 0x7fffffffull)
        return cudaErrorInvalidValue;
    fanout_kernel<DT, MAXR><<<dim3((unsigned)tiles, (unsigned)nchunks), kFanThreads, kFanOccupancySmem, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_fanout(int dt, const void *const *src, int nchunks, void *const *dst, int ndst, uint64_t count,
                          cudaStream_t stream)
{
    const bool small = nchunks <= kSmallRanks && ndst <= kSmallRanks;
    if (dt == DT_FP32)
        return small ? launch_fanout_t<DT_FP32, kSmallRanks>(src, nchunks, dst, ndst, count, stream)
                     : launch_fanout_t<DT_FP32, kMaxRanks>(src, nchunks, dst, ndst, count, stream);
    return small ? launch_fanout_t<DT_BF16, kSmallRanks>(src, nchunks, dst, ndst, count, stream)
                 : launch_fanout_t<DT_BF16, kMaxRanks>(src, nchunks, dst, ndst, count, stream);
}

} // namespace ccl
