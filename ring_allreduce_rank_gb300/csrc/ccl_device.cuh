// ccl_device.cuh -- device-side building blocks shared by the collective kernels:
// 16-byte streaming loads/stores and the per-hop arithmetic of the ring
// reduction (one IEEE fp32 operation, round to nearest even, then a round to
// the buffer type).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ccl {

enum { DT_FP32 = 0, DT_BF16 = 1 };
enum { OP_SUM = 0, OP_AVG = 1, OP_MAX = 2, OP_PROD = 3, OP_MIN = 4, OP_AVGP = 5 };

constexpr int kThreads = 256;

template <int DT> struct DType;
template <> struct DType<DT_FP32> { static constexpr int kSize = 4; static constexpr int kVec = 4; };
template <> struct DType<DT_BF16> { static constexpr int kSize = 2; static constexpr int kVec = 8; };

// ------------------------------------------------------------------ bounds checks (debug builds)
// Built with CCL_DEBUG_BOUNDS, every global access below is checked against
// the byte ranges of the current call's buffers, which the host sets on the
// call's stream before its kernels (dbg_set_ranges).  An access outside all of
// them is counted, its address recorded, and skipped -- never performed, so a
// wrong index cannot fault the device.  Release builds compile the check to
// `true`.

#ifdef CCL_DEBUG_BOUNDS
constexpr int kDbgMaxRanges = 4096;
extern __device__ unsigned g_dbg_n;                          // ranges in use
extern __device__ unsigned long long g_dbg_r[kDbgMaxRanges][2]; // [lo, hi) byte addresses
extern __device__ unsigned g_dbg_faults;
extern __device__ unsigned long long g_dbg_first_fault;

__device__ __forceinline__ bool dbg_ok(const void *p, size_t bytes)
{
    const unsigned long long a = (unsigned long long)(uintptr_t)p, b = a + bytes;
    const unsigned n = g_dbg_n;
    for (unsigned i = 0; i < n; ++i)
        if (a >= g_dbg_r[i][0] && b <= g_dbg_r[i][1])
            return true;
    if (atomicAdd(&g_dbg_faults, 1u) == 0)
        g_dbg_first_fault = a;
    return false;
}
#else
__device__ __forceinline__ constexpr bool dbg_ok(const void *, size_t) { return true; }
#endif

// ------------------------------------------------------------------ memory
// Loads bypass L1 (every byte is used once); stores are plain write-back so
// that in-place writes land on lines the same thread just read.

__device__ __forceinline__ uint4 ld16(const void *p)
{
    uint4 v = make_uint4(0, 0, 0, 0);
    if (dbg_ok(p, 16))
        asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p));
    return v;
}

__device__ __forceinline__ void st16(void *p, const uint4 &v)
{
    if (dbg_ok(p, 16))
        asm volatile("st.global.L1::no_allocate.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                     "r"(v.w)
                     : "memory");
}

// plain global load / store of a T (vector widths the kernels use directly)
template <class T> __device__ __forceinline__ T gload(const void *p)
{
    T v{};
    if (dbg_ok(p, sizeof(T)))
        v = *static_cast<const T *>(p);
    return v;
}

template <class T> __device__ __forceinline__ void gstore(void *p, const T &v)
{
    if (dbg_ok(p, sizeof(T)))
        *static_cast<T *>(p) = v;
}

template <int DT> __device__ __forceinline__ uint32_t ld_elem(const void *base, uint64_t i)
{
    if (DT == DT_BF16)
        return gload<uint16_t>(static_cast<const uint16_t *>(base) + i);
    return gload<uint32_t>(static_cast<const uint32_t *>(base) + i);
}

template <int DT> __device__ __forceinline__ void st_elem(void *base, uint64_t i, uint32_t v)
{
    if (DT == DT_BF16)
        gstore<uint16_t>(static_cast<uint16_t *>(base) + i, static_cast<uint16_t>(v));
    else
        gstore<uint32_t>(static_cast<uint32_t *>(base) + i, v);
}

// ------------------------------------------------------------------ arithmetic

// MAX on fp32 bit patterns: NaN if either is NaN, else the larger; equal
// values give the bitwise AND (identical bits, or +0 for +0 vs -0).
__device__ __forceinline__ uint32_t max_f32_bits(uint32_t a, uint32_t b)
{
    const float fa = __uint_as_float(a), fb = __uint_as_float(b);
    if (fa != fa || fb != fb)
        return 0x7fffffffu;
    if (fa > fb)
        return a;
    if (fb > fa)
        return b;
    return a & b;
}

// MIN on fp32 bit patterns: NaN if either is NaN, else the smaller; equal
// values give the bitwise OR (identical bits, or -0 for +0 vs -0).
__device__ __forceinline__ uint32_t min_f32_bits(uint32_t a, uint32_t b)
{
    const float fa = __uint_as_float(a), fb = __uint_as_float(b);
    if (fa != fa || fb != fb)
        return 0x7fffffffu;
    if (fa < fb)
        return a;
    if (fb < fa)
        return b;
    return a | b;
}

template <int OP> __device__ __forceinline__ uint32_t minmax_f32_bits(uint32_t a, uint32_t b)
{
    return OP == OP_MAX ? max_f32_bits(a, b) : min_f32_bits(a, b);
}

template <int OP> __device__ __forceinline__ float op_f32(float local, float acc)
{
    if (OP == OP_PROD)
        return __fmul_rn(local, acc);
    return __fadd_rn(local, acc); // SUM, AVG and pre-multiplied AVG
}

// One ring hop on one fp32 element: local (+) incoming.
template <int OP> __device__ __forceinline__ uint32_t hop_f32(uint32_t local, uint32_t acc)
{
    if (OP == OP_MAX || OP == OP_MIN)
        return minmax_f32_bits<OP>(local, acc);
    return __float_as_uint(op_f32<OP>(__uint_as_float(local), __uint_as_float(acc)));
}

// One ring hop on a pair of bf16 elements packed in 32 bits (element 0 in the
// low half): widen (exact), fp32 operation, round each to bf16 (RNE).
template <int OP> __device__ __forceinline__ uint32_t hop_bf16x2(uint32_t local, uint32_t acc)
{
    if (OP == OP_MAX || OP == OP_MIN) {
        // the result is one operand unchanged (or the canonical NaN): no rounding
        const uint32_t lo = minmax_f32_bits<OP>(local << 16, acc << 16) >> 16;
        const uint32_t hi = minmax_f32_bits<OP>(local & 0xffff0000u, acc & 0xffff0000u) & 0xffff0000u;
        return lo | hi;
    }
    const float r0 = op_f32<OP>(__uint_as_float(local << 16), __uint_as_float(acc << 16));
    const float r1 = op_f32<OP>(__uint_as_float(local & 0xffff0000u), __uint_as_float(acc & 0xffff0000u));
    __nv_bfloat162 p = __floats2bfloat162_rn(r0, r1);
    return *reinterpret_cast<uint32_t *>(&p);
}

// Scalar hop on a stored element (bf16 in the low 16 bits).
template <int DT, int OP> __device__ __forceinline__ uint32_t hop_elem(uint32_t local, uint32_t acc)
{
    if (DT == DT_FP32)
        return hop_f32<OP>(local, acc);
    return hop_bf16x2<OP>(local, acc) & 0xffffu;
}

template <int DT, int OP> __device__ __forceinline__ uint4 hop_vec(const uint4 &local, const uint4 &acc)
{
    uint4 r;
    if (DT == DT_FP32) {
        r.x = hop_f32<OP>(local.x, acc.x);
        r.y = hop_f32<OP>(local.y, acc.y);
        r.z = hop_f32<OP>(local.z, acc.z);
        r.w = hop_f32<OP>(local.w, acc.w);
    } else {
        r.x = hop_bf16x2<OP>(local.x, acc.x);
        r.y = hop_bf16x2<OP>(local.y, acc.y);
        r.z = hop_bf16x2<OP>(local.z, acc.z);
        r.w = hop_bf16x2<OP>(local.w, acc.w);
    }
    return r;
}

// AVG: one fp32 division of the finished sum by N, rounded to the buffer type.
__device__ __forceinline__ uint32_t avg_f32(uint32_t v, float n)
{
    return __float_as_uint(__fdiv_rn(__uint_as_float(v), n));
}

__device__ __forceinline__ uint32_t avg_bf16x2(uint32_t v, float n)
{
    const float r0 = __fdiv_rn(__uint_as_float(v << 16), n);
    const float r1 = __fdiv_rn(__uint_as_float(v & 0xffff0000u), n);
    __nv_bfloat162 p = __floats2bfloat162_rn(r0, r1);
    return *reinterpret_cast<uint32_t *>(&p);
}

template <int DT> __device__ __forceinline__ uint32_t avg_elem(uint32_t v, float n)
{
    if (DT == DT_FP32)
        return avg_f32(v, n);
    return avg_bf16x2(v, n) & 0xffffu;
}

template <int DT> __device__ __forceinline__ uint4 avg_vec(const uint4 &v, float n)
{
    uint4 r;
    if (DT == DT_FP32) {
        r.x = avg_f32(v.x, n);
        r.y = avg_f32(v.y, n);
        r.z = avg_f32(v.z, n);
        r.w = avg_f32(v.w, n);
    } else {
        r.x = avg_bf16x2(v.x, n);
        r.y = avg_bf16x2(v.y, n);
        r.z = avg_bf16x2(v.z, n);
        r.w = avg_bf16x2(v.w, n);
    }
    return r;
}

// AVG by pre-multiplication (NCCL's pre-multiplied sum, Collective
// Communication, libraries section): a contribution x enters the ring as
// x * inv rounded to the buffer type, inv being the correctly rounded fp32
// reciprocal of N, and the ring then sums; nothing is divided at the end.
// Every other operator takes its contributions unchanged.
__device__ __forceinline__ uint32_t premul_bf16x2(uint32_t v, float inv)
{
    const float r0 = __fmul_rn(__uint_as_float(v << 16), inv);
    const float r1 = __fmul_rn(__uint_as_float(v & 0xffff0000u), inv);
    __nv_bfloat162 p = __floats2bfloat162_rn(r0, r1);
    return *reinterpret_cast<uint32_t *>(&p);
}

template <int DT, int OP> __device__ __forceinline__ uint32_t pre_elem(uint32_t v, float inv)
{
    if (OP != OP_AVGP)
        return v;
    if (DT == DT_FP32)
        return __float_as_uint(__fmul_rn(__uint_as_float(v), inv));
    return premul_bf16x2(v, inv) & 0xffffu;
}

template <int DT, int OP> __device__ __forceinline__ uint4 pre_vec(const uint4 &v, float inv)
{
    if (OP != OP_AVGP)
        return v;
    uint4 r;
    if (DT == DT_FP32) {
        r.x = __float_as_uint(__fmul_rn(__uint_as_float(v.x), inv));
        r.y = __float_as_uint(__fmul_rn(__uint_as_float(v.y), inv));
        r.z = __float_as_uint(__fmul_rn(__uint_as_float(v.z), inv));
        r.w = __float_as_uint(__fmul_rn(__uint_as_float(v.w), inv));
    } else {
        r.x = premul_bf16x2(v.x, inv);
        r.y = premul_bf16x2(v.y, inv);
        r.z = premul_bf16x2(v.z, inv);
        r.w = premul_bf16x2(v.w, inv);
    }
    return r;
}

// ------------------------------------------------------------------ ring folds over a pointer table

// Fold one 16-byte vector of every rank in ring order starting at rank c:
// x_c, then x_{c+1} (+) acc, ..., x_{c-1} (+) acc.  ptrs[r] is rank r's base.
// NR > 0: exactly NR ranks, all loads issued before the first hop.
// NR == 0: any N, ranks in groups of 8 with the next group's loads in flight.
// inv: the reciprocal of N for the pre-multiplied AVG (unused otherwise).
template <int DT, int OP, int NR>
__device__ __forceinline__ uint4 ring_fold_vec(const void *const *ptrs, int N, int c, uint64_t byte_off, float inv)
{
    if (NR > 0) {
        uint4 x[NR > 0 ? NR : 1];
        int r = c;
#pragma unroll
        for (int k = 0; k < NR; ++k) {
            x[k] = ld16(static_cast<const char *>(ptrs[r]) + byte_off);
            r = (r + 1 == NR) ? 0 : r + 1;
        }
        uint4 acc = pre_vec<DT, OP>(x[0], inv);
#pragma unroll
        for (int k = 1; k < NR; ++k)
            acc = hop_vec<DT, OP>(pre_vec<DT, OP>(x[k], inv), acc);
        return acc;
    }
    uint4 acc = make_uint4(0, 0, 0, 0);
    uint4 cur[8], nxt[8];
    int r = c;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        if (j < N) {
            cur[j] = ld16(static_cast<const char *>(ptrs[r]) + byte_off);
            r = (r + 1 == N) ? 0 : r + 1;
        }
    for (int g = 0; g < N; g += 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (g + 8 + j < N) {
                nxt[j] = ld16(static_cast<const char *>(ptrs[r]) + byte_off);
                r = (r + 1 == N) ? 0 : r + 1;
            }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (g + j < N)
                acc = (g + j == 0) ? pre_vec<DT, OP>(cur[0], inv) : hop_vec<DT, OP>(pre_vec<DT, OP>(cur[j], inv), acc);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            cur[j] = nxt[j];
    }
    return acc;
}

template <int DT, int OP>
__device__ __forceinline__ uint32_t ring_fold_elem(const void *const *ptrs, int N, int c, uint64_t e, float inv)
{
    int r = c;
    uint32_t acc = pre_elem<DT, OP>(ld_elem<DT>(ptrs[r], e), inv);
    for (int k = 1; k < N; ++k) {
        if (++r == N)
            r = 0;
        acc = hop_elem<DT, OP>(pre_elem<DT, OP>(ld_elem<DT>(ptrs[r], e), inv), acc);
    }
    return acc;
}

__host__ __device__ __forceinline__ uint64_t umin64(uint64_t a, uint64_t b) { return a < b ? a : b; }

// Output window of `d` elements into (lo, hi): the vector made of lo's
// elements d..VEC-1 followed by hi's elements 0..d-1 (0 < d < VEC).
template <int DT> __device__ __forceinline__ uint4 shift_window(const uint4 &lo, const uint4 &hi, int d)
{
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t o[4];
    if (DT == DT_FP32) {
        switch (d) {
        case 1: o[0] = w[1]; o[1] = w[2]; o[2] = w[3]; o[3] = w[4]; break;
        case 2: o[0] = w[2]; o[1] = w[3]; o[2] = w[4]; o[3] = w[5]; break;
        default: o[0] = w[3]; o[1] = w[4]; o[2] = w[5]; o[3] = w[6]; break;
        }
    } else {
        // d halfwords: whole words k = d/2, then half a word if d is odd
#define CCL_SHIFT_CASE(D)                                                                                              \
    case D:                                                                                                            \
        _Pragma("unroll") for (int i = 0; i < 4; ++i) o[i] =                                                           \
            (D & 1) ? __funnelshift_r(w[(D >> 1) + i], w[(D >> 1) + i + 1], 16) : w[(D >> 1) + i];                     \
        break;
        switch (d) {
            CCL_SHIFT_CASE(1) CCL_SHIFT_CASE(2) CCL_SHIFT_CASE(3) CCL_SHIFT_CASE(4) CCL_SHIFT_CASE(5)
            CCL_SHIFT_CASE(6)
        default:
            _Pragma("unroll") for (int i = 0; i < 4; ++i) o[i] = __funnelshift_r(w[3 + i], w[4 + i], 16);
        }
#undef CCL_SHIFT_CASE
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}


// ------------------------------------------------------------------ chunk partition

// Chunk c of a K-element buffer: len = K/N + (c < K%N), first K%N chunks longer.
struct Partition {
    uint64_t q;   // K / N
    uint32_t rem; // K % N
    __host__ __device__ __forceinline__ uint64_t off(uint32_t c) const
    {
        return (uint64_t)c * q + (c < rem ? c : rem);
    }
    __host__ __device__ __forceinline__ uint64_t len(uint32_t c) const { return q + (c < rem ? 1 : 0); }
};

__host__ __device__ __forceinline__ int ring_mod(int a, int n)
{
    int r = a % n;
    return r < 0 ? r + n : r;
}

} // namespace ccl
