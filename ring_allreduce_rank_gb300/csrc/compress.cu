// compress.cu -- compressed AllReduce with error feedback, fused in one pass.
//
// Every rank adds its residual to its gradient, u = g + e (fp32), compresses
// u, and keeps e' = u - v, the part not transmitted (Collective Communication,
// "Error feedback and residual accumulation", Definition 1.4).  Compressors:
//   INT8 block ("Blockwise quantization for gradient communication"): per
//     block of b = 64 or 128 consecutive elements, s = max|u| / 127,
//     q = round(u / s) (ties to even), v = q * s -- 4b/(b+4) fewer bytes than
//     fp32 on a real link;
//   THRESHOLD (the greedy 1-bit compressor of the pages' Tables 3 and 4):
//     v = 1 when u >= threshold, else 0.
// The transmitted values are then AllReduced in ring order in fp32 (chunk c
// folded from rank c), AVG divides once by N, and the result is rounded once
// to the gradients' type and written to every rank.
//
// Layout: one warp per compression block (the same block index in every
// rank); lane l owns elements [l*EPL, (l+1)*EPL) of it.  The warp first issues
// every rank's g and e loads, then walks the ranks: forms u, reduces the block
// maximum with shuffles, quantises, writes the new residual, and keeps v in
// registers.  Then each
// lane folds its elements over the ranks in ring order with two statically
// unrolled passes (ranks c..N-1, then 0..c-1).  Up to 16 ranks.
#include "ccl_internal.h"

namespace ccl {

constexpr int kCompMaxRanks = 16;

struct CompParams {
    void *grads[kCompMaxRanks];
    float *res[kCompMaxRanks];
    Partition part;
    uint64_t K;
    int nranks;
    int comp;  // COMP_INT8_BLOCK or COMP_THRESHOLD
    float threshold;
    float n_f;   // AVG: N (0 for SUM)
    float inv_n; // 1/N, exact when N is a power of two
    int pow2;    // N is a power of two
    int vec_ok;  // grads and residuals aligned for the lane's vector width
};

template <int DT, int EPL>
__device__ __forceinline__ void load_g(const void *base, uint64_t i, int valid, bool vec, float (&out)[EPL])
{
    if (vec && valid == EPL) {
        if (DT == DT_FP32) {
            if (EPL == 4) {
                const uint4 w = *reinterpret_cast<const uint4 *>(static_cast<const float *>(base) + i);
                out[0] = __uint_as_float(w.x); out[1] = __uint_as_float(w.y);
                out[2] = __uint_as_float(w.z); out[3] = __uint_as_float(w.w);
                return;
            }
            const uint2 w = *reinterpret_cast<const uint2 *>(static_cast<const float *>(base) + i);
            out[0] = __uint_as_float(w.x); out[1] = __uint_as_float(w.y);
            return;
        }
        if (EPL == 4) {
            const uint2 w = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(base) + i);
            out[0] = __uint_as_float(w.x << 16); out[1] = __uint_as_float(w.x & 0xffff0000u);
            out[2] = __uint_as_float(w.y << 16); out[3] = __uint_as_float(w.y & 0xffff0000u);
            return;
        }
        const uint32_t w = *reinterpret_cast<const uint32_t *>(static_cast<const uint16_t *>(base) + i);
        out[0] = __uint_as_float(w << 16); out[1] = __uint_as_float(w & 0xffff0000u);
        return;
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        const uint32_t b = j < valid ? ld_elem<DT>(base, i + j) : 0u;
        out[j] = __uint_as_float(DT == DT_BF16 ? b << 16 : b);
    }
}

template <int EPL>
__device__ __forceinline__ void load_f(const float *base, uint64_t i, int valid, bool vec, float (&out)[EPL])
{
    if (vec && valid == EPL) {
        if (EPL == 4) {
            const float4 w = *reinterpret_cast<const float4 *>(base + i);
            out[0] = w.x; out[1] = w.y; out[2] = w.z; out[3] = w.w;
        } else {
            const float2 w = *reinterpret_cast<const float2 *>(base + i);
            out[0] = w.x; out[1] = w.y;
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j)
        out[j] = j < valid ? base[i + j] : 0.0f;
}

template <int EPL>
__device__ __forceinline__ void store_f(float *base, uint64_t i, int valid, bool vec, const float (&v)[EPL])
{
    if (vec && valid == EPL) {
        if (EPL == 4)
            *reinterpret_cast<float4 *>(base + i) = make_float4(v[0], v[1], v[2], v[3]);
        else
            *reinterpret_cast<float2 *>(base + i) = make_float2(v[0], v[1]);
        return;
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j)
        if (j < valid)
            base[i + j] = v[j];
}

// q = round(u / s), ties to even, with u / s the correctly rounded fp32
// quotient -- without a division in almost every case.  For |u| <= max|u|
// = 127 s, t = u * rn(1/s) differs from rn(u / s) by less than
// 2 * 127 * 2^-24 < 2^-14, so unless t is within 2^-14 of a half-integer both
// round to the same integer; near a tie the exact quotient decides.  The
// caller handles s = 0, a NaN scale, and a reciprocal that overflows.
__device__ __forceinline__ float quantize_fast(float u, float s, float inv)
{
    const float t = __fmul_rn(u, inv);
    const float q = rintf(t);
    if (fabsf(t - q) > 0.49993896484375f) // within 2^-14 of a half-integer
        return rintf(__fdiv_rn(u, s));
    return q;
}

template <int DT>
__device__ __forceinline__ uint32_t round_to(float x)
{
    if (DT == DT_FP32)
        return __float_as_uint(x);
    __nv_bfloat162 p = __floats2bfloat162_rn(x, 0.0f);
    return *reinterpret_cast<uint32_t *>(&p) & 0xffffu;
}

template <int DT, int EPL, int NMAX>
__global__ void __launch_bounds__(kThreads, NMAX <= 8 ? 3 : 1) compressed_allreduce_kernel(const __grid_constant__ CompParams p)
{
    constexpr int B = 32 * EPL; // compression block
    const int lane = threadIdx.x & 31;
    const uint64_t blk = ((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const uint64_t b0 = blk * B;
    if (b0 >= p.K)
        return; // whole warp leaves together
    const uint64_t i0 = b0 + (uint64_t)lane * EPL;
    const int valid = i0 >= p.K ? 0 : (int)umin64(EPL, p.K - i0);
    const bool vec = p.vec_ok != 0;
    const int N = p.nranks;

    // every rank's gradient and residual loads are issued before any compute,
    // so a lane has N * EPL * (element + 4) bytes in flight
    float v[NMAX][EPL], ee[NMAX][EPL];
#pragma unroll
    for (int r = 0; r < NMAX; ++r) {
        if (r < N) {
            load_g<DT, EPL>(p.grads[r], i0, valid, vec, v[r]);
            load_f<EPL>(p.res[r], i0, valid, vec, ee[r]);
        } else {
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                v[r][j] = ee[r][j] = 0.0f; // absent ranks: never stored
        }
    }
    // u = g + e (kept in v until it is replaced by the transmitted value)
#pragma unroll
    for (int r = 0; r < NMAX; ++r)
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            v[r][j] = __fadd_rn(v[r][j], ee[r][j]);

    if (p.comp == COMP_THRESHOLD) {
#pragma unroll
        for (int r = 0; r < NMAX; ++r)
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const float u = v[r][j];
                v[r][j] = u >= p.threshold ? 1.0f : 0.0f;
                ee[r][j] = __fsub_rn(u, v[r][j]);
            }
    } else {
        // block maxima of all ranks, the shuffle chains interleaved
        float amax[NMAX];
        uint32_t nanmask = 0;
#pragma unroll
        for (int r = 0; r < NMAX; ++r) {
            amax[r] = 0.0f;
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                if (j < valid) {
                    if (v[r][j] != v[r][j])
                        nanmask |= 1u << r;
                    else
                        amax[r] = fmaxf(amax[r], fabsf(v[r][j]));
                }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                amax[r] = fmaxf(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], o));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            nanmask |= __shfl_xor_sync(0xffffffffu, nanmask, o);
#pragma unroll
        for (int r = 0; r < NMAX; ++r) {
            const float s = (nanmask >> r) & 1u ? __uint_as_float(0x7fffffffu) : __fdiv_rn(amax[r], 127.0f);
            const float inv = __frcp_rn(s);
            const bool fast = s > 0.0f && inv < __uint_as_float(0x7f800000u); // warp-uniform
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const float u = v[r][j];
                float q;
                if (fast)
                    q = quantize_fast(u, s, inv);
                else
                    q = s > 0.0f ? rintf(__fdiv_rn(u, s)) : (s == 0.0f ? 0.0f : s);
                v[r][j] = __fmul_rn(q, s);
                ee[r][j] = __fsub_rn(u, v[r][j]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NMAX; ++r)
        if (r < N)
            store_f<EPL>(p.res[r], i0, valid, vec, ee[r]);

    // ring-order fold in fp32: chunk c from rank c, then c+1, ..., c-1
    uint32_t c = 0;
    if (valid > 0) {
        const uint64_t q1 = p.part.q + 1, head = (uint64_t)p.part.rem * q1;
        c = i0 < head ? (uint32_t)(i0 / q1) : (uint32_t)(p.part.rem + (p.part.q ? (i0 - head) / p.part.q : 0));
    }
    uint32_t outb[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        while (c + 1 < (uint32_t)N && i0 + j >= p.part.off(c + 1))
            ++c;
        float acc;
        if (N == NMAX) {
            // every rank present: one static fold per rotation start (the start
            // is the same across the warp except at a chunk boundary)
            switch (c) {
#define CCL_FOLD_CASE(C)                                                                                           \
    case C:                                                                                                            \
        acc = v[C % NMAX][j];                                                                                          \
        _Pragma("unroll") for (int k = 1; k < NMAX; ++k) acc = __fadd_rn(v[(C + k) % NMAX][j], acc);                   \
        break;
                CCL_FOLD_CASE(0) CCL_FOLD_CASE(1) CCL_FOLD_CASE(2) CCL_FOLD_CASE(3)
                CCL_FOLD_CASE(4) CCL_FOLD_CASE(5) CCL_FOLD_CASE(6) CCL_FOLD_CASE(7)
                CCL_FOLD_CASE(8) CCL_FOLD_CASE(9) CCL_FOLD_CASE(10) CCL_FOLD_CASE(11)
                CCL_FOLD_CASE(12) CCL_FOLD_CASE(13) CCL_FOLD_CASE(14) CCL_FOLD_CASE(15)
#undef CCL_FOLD_CASE
            default:
                acc = 0.0f;
            }
        } else {
            acc = 0.0f;
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                if (r < N && r >= (int)c)
                    acc = r == (int)c ? v[r][j] : __fadd_rn(v[r][j], acc);
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                if (r < (int)c)
                    acc = __fadd_rn(v[r][j], acc);
        }
        if (p.n_f > 0.0f) // AVG: x / N, or x * (1/N) when N is a power of two (the same rounded value)
            acc = p.pow2 ? __fmul_rn(acc, p.inv_n) : __fdiv_rn(acc, p.n_f);
        outb[j] = round_to<DT>(acc);
    }
    // the result, packed into one vector store per rank when the lane is whole
    const bool packed = vec && valid == EPL;
    uint32_t w[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j)
        w[j] = (DT == DT_BF16) ? ((j & 1) ? 0u : outb[j] | (j + 1 < EPL ? outb[j + 1] << 16 : 0u)) : outb[j];
#pragma unroll
    for (int r = 0; r < NMAX; ++r) {
        if (r >= N)
            break;
        if (packed) {
            if (DT == DT_FP32 && EPL == 4)
                *reinterpret_cast<uint4 *>(static_cast<uint32_t *>(p.grads[r]) + i0) = make_uint4(w[0], w[1], w[2], w[3]);
            else if (DT == DT_FP32)
                *reinterpret_cast<uint2 *>(static_cast<uint32_t *>(p.grads[r]) + i0) = make_uint2(w[0], w[1]);
            else if (EPL == 4)
                *reinterpret_cast<uint2 *>(static_cast<uint16_t *>(p.grads[r]) + i0) = make_uint2(w[0], w[2]);
            else
                *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(p.grads[r]) + i0) = w[0];
        } else {
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                if (j < valid)
                    st_elem<DT>(p.grads[r], i0 + j, outb[j]);
        }
    }
}

template <int DT, int EPL, int NMAX>
static cudaError_t launch_comp_t(const CompParams &p, cudaStream_t stream)
{
    constexpr int B = 32 * EPL;
    const uint64_t warps = (p.K + B - 1) / B;
    const uint64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffull)
        return cudaErrorInvalidValue;
    compressed_allreduce_kernel<DT, EPL, NMAX><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_compressed_allreduce(int dt, bool avg, int comp, int block, float threshold,
                                        void *const *grads, float *const *res, int nranks, uint64_t count,
                                        cudaStream_t stream)
{
    if (nranks > kCompMaxRanks)
        return cudaErrorInvalidValue;
    CompParams p;
    const int epl = comp == COMP_THRESHOLD ? 4 : block / 32;
    const int es = dt == DT_BF16 ? 2 : 4;
    bool vec = true;
    for (int r = 0; r < kCompMaxRanks; ++r) {
        p.grads[r] = r < nranks ? grads[r] : nullptr;
        p.res[r] = r < nranks ? res[r] : nullptr;
        if (r < nranks)
            vec = vec && (uintptr_t)grads[r] % (uintptr_t)(epl * es) == 0 && (uintptr_t)res[r] % (uintptr_t)(epl * 4) == 0;
    }
    p.part.q = count / (uint64_t)nranks;
    p.part.rem = (uint32_t)(count % (uint64_t)nranks);
    p.K = count;
    p.nranks = nranks;
    p.comp = comp;
    p.threshold = threshold;
    p.n_f = avg ? (float)nranks : 0.0f;
    p.pow2 = (nranks & (nranks - 1)) == 0 ? 1 : 0;
    p.inv_n = 1.0f / (float)nranks;
    p.vec_ok = vec ? 1 : 0;
    const bool small = nranks <= 8;
    if (dt == DT_FP32) {
        if (epl == 4)
            return small ? launch_comp_t<DT_FP32, 4, 8>(p, stream) : launch_comp_t<DT_FP32, 4, 16>(p, stream);
        return small ? launch_comp_t<DT_FP32, 2, 8>(p, stream) : launch_comp_t<DT_FP32, 2, 16>(p, stream);
    }
    if (epl == 4)
        return small ? launch_comp_t<DT_BF16, 4, 8>(p, stream) : launch_comp_t<DT_BF16, 4, 16>(p, stream);
    return small ? launch_comp_t<DT_BF16, 2, 8>(p, stream) : launch_comp_t<DT_BF16, 2, 16>(p, stream);
}

} // namespace ccl
