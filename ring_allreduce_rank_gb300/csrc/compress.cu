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
//     v = 1 when u >= threshold, else 0;
//   TOPK ("Top-k sparsification"): v = u when the magnitude key of u (its
//     bits with the sign cleared) reaches the rank's k-th largest key tau,
//     found beforehand by the radix select in topk.cu, else 0.
// The transmitted values are then AllReduced in ring order in fp32 (chunk c
// folded from rank c), AVG divides once by N, and the result is rounded once
// to the gradients' type and written to every rank.
//
// Layout: one warp per compression block (the same block index in every
// rank); lane l owns elements [l*EPL, (l+1)*EPL) of it.  Up to 8 ranks with
// aligned buffers take the pipelined form below (shared-memory double
// buffering with cp.async); the rest take the direct form.  The warp first issues
// every rank's g and e loads, then walks the ranks: forms u, reduces the block
// maximum with shuffles, quantises, writes the new residual, and keeps v in
// registers.  Then each
// lane folds its elements over the ranks in ring order with two statically
// unrolled passes (ranks c..N-1, then 0..c-1).  Up to 16 ranks.
#include <mutex>
#include <unordered_map>

#include "ccl_internal.h"

namespace ccl {

constexpr int kCompMaxRanks = 16;

struct CompParams {
    void *grads[kCompMaxRanks];
    float *res[kCompMaxRanks];
    Partition part;
    uint64_t K;
    int nranks;
    int comp;  // COMP_INT8_BLOCK, COMP_THRESHOLD or COMP_TOPK
    float threshold;
    float n_f;   // AVG: N (0 for SUM)
    float inv_n; // 1/N, exact when N is a power of two
    int pow2;    // N is a power of two
    int vec_ok;  // grads and residuals aligned for the lane's vector width
    uint64_t first_block; // the direct kernel starts at this compression block
    uint64_t nfull;       // the pipelined kernel covers blocks [0, nfull)
    uint64_t coff[kCompMaxRanks + 1]; // chunk c starts at coff[c]; entries from N on hold K
    const uint32_t *tau;              // COMP_TOPK: each rank's threshold key (device memory)
};

// max that returns NaN when either side is NaN (PTX max.NaN), so a block's
// maximum of |u| also says whether the block holds a NaN
__device__ __forceinline__ float fmax_nan(float a, float b)
{
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// chunk holding element e: the number of chunk starts after chunk 0 at or below e
template <int NMAX>
__device__ __forceinline__ uint32_t chunk_of(const CompParams &p, uint64_t e)
{
    uint32_t c = 0;
#pragma unroll
    for (int k = 1; k < NMAX; ++k)
        c += e >= p.coff[k] ? 1u : 0u;
    return c;
}

template <int DT, int EPL>
__device__ __forceinline__ void load_g(const void *base, uint64_t i, int valid, bool vec, float (&out)[EPL])
{
    if (vec && valid == EPL) {
        if (DT == DT_FP32) {
            if (EPL == 4) {
                const uint4 w = gload<uint4>(static_cast<const float *>(base) + i);
                out[0] = __uint_as_float(w.x); out[1] = __uint_as_float(w.y);
                out[2] = __uint_as_float(w.z); out[3] = __uint_as_float(w.w);
                return;
            }
            const uint2 w = gload<uint2>(static_cast<const float *>(base) + i);
            out[0] = __uint_as_float(w.x); out[1] = __uint_as_float(w.y);
            return;
        }
        if (EPL == 4) {
            const uint2 w = gload<uint2>(static_cast<const uint16_t *>(base) + i);
            out[0] = __uint_as_float(w.x << 16); out[1] = __uint_as_float(w.x & 0xffff0000u);
            out[2] = __uint_as_float(w.y << 16); out[3] = __uint_as_float(w.y & 0xffff0000u);
            return;
        }
        const uint32_t w = gload<uint32_t>(static_cast<const uint16_t *>(base) + i);
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
            const float4 w = gload<float4>(base + i);
            out[0] = w.x; out[1] = w.y; out[2] = w.z; out[3] = w.w;
        } else {
            const float2 w = gload<float2>(base + i);
            out[0] = w.x; out[1] = w.y;
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j)
        out[j] = j < valid ? gload<float>(base + i + j) : 0.0f;
}

template <int EPL>
__device__ __forceinline__ void store_f(float *base, uint64_t i, int valid, bool vec, const float (&v)[EPL])
{
    if (vec && valid == EPL) {
        if (EPL == 4)
            gstore<float4>(base + i, make_float4(v[0], v[1], v[2], v[3]));
        else
            gstore<float2>(base + i, make_float2(v[0], v[1]));
        return;
    }
#pragma unroll
    for (int j = 0; j < EPL; ++j)
        if (j < valid)
            gstore<float>(base + i + j, v[j]);
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

// Each rank's Top-k threshold key, read once per kernel (all-ones, which no
// key reaches, for the other compressors and absent ranks).
template <int NMAX, int COMP> __device__ __forceinline__ void load_tau(const CompParams &p, uint32_t (&tau)[NMAX])
{
#pragma unroll
    for (int r = 0; r < NMAX; ++r)
        tau[r] = (COMP == COMP_TOPK && r < p.nranks) ? gload<uint32_t>(p.tau + r) : 0xffffffffu;
}

// Everything after the loads: u = g + e, compression, residual store, the
// ring-order fp32 fold and the result store.  v holds g and ee holds e on entry.
template <int DT, int EPL, int NMAX, int COMP>
__device__ __forceinline__ void compress_fold_store(const CompParams &p, uint64_t i0, int valid, bool vec,
                                                    float (&v)[NMAX][EPL], float (&ee)[NMAX][EPL],
                                                    const uint32_t (&tau)[NMAX])
{
    const int N = p.nranks;
    // u = g + e (kept in v until it is replaced by the transmitted value)
#pragma unroll
    for (int r = 0; r < NMAX; ++r)
#pragma unroll
        for (int j = 0; j < EPL; ++j)
            v[r][j] = __fadd_rn(v[r][j], ee[r][j]);

    if constexpr (COMP == COMP_THRESHOLD) {
#pragma unroll
        for (int r = 0; r < NMAX; ++r)
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const float u = v[r][j];
                v[r][j] = u >= p.threshold ? 1.0f : 0.0f;
                ee[r][j] = __fsub_rn(u, v[r][j]);
            }
    } else if constexpr (COMP == COMP_TOPK) {
#pragma unroll
        for (int r = 0; r < NMAX; ++r) {
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const float u = v[r][j];
                v[r][j] = (__float_as_uint(u) & 0x7fffffffu) >= tau[r] ? u : 0.0f;
                ee[r][j] = __fsub_rn(u, v[r][j]);
            }
        }
    } else {
        // per-rank block maxima of |u|; a NaN anywhere in the block makes the
        // maximum NaN, and the scale with it
        float amax[NMAX];
#pragma unroll
        for (int r = 0; r < NMAX; ++r) {
            amax[r] = 0.0f;
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                if (j < valid)
                    amax[r] = fmax_nan(amax[r], fabsf(v[r][j]));
        }
        float sc[NMAX], inv[NMAX];
        const int lane = threadIdx.x & 31;
        if constexpr (NMAX == 8) {
            // transposing butterfly: after the exchanges at distance 16, 8 and 4
            // lane l holds rank (l >> 2) & 7's maximum over 8 lanes, and two
            // more rounds finish it; each lane then computes that one rank's
            // scale and reciprocal, and the eight values are broadcast
            const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
            float k4[4], k2[2];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float send = b4 ? amax[k] : amax[k + 4];
                k4[k] = fmax_nan(b4 ? amax[k + 4] : amax[k], __shfl_xor_sync(0xffffffffu, send, 16));
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float send = b3 ? k4[k] : k4[k + 2];
                k2[k] = fmax_nan(b3 ? k4[k + 2] : k4[k], __shfl_xor_sync(0xffffffffu, send, 8));
            }
            float m = fmax_nan(b2 ? k2[1] : k2[0], __shfl_xor_sync(0xffffffffu, b2 ? k2[0] : k2[1], 4));
            m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, 1));
            const float s1 = m != m ? __uint_as_float(0x7fffffffu) : __fdiv_rn(m, 127.0f);
            const float i1 = __frcp_rn(s1);
#pragma unroll
            for (int r = 0; r < NMAX; ++r) {
                sc[r] = __shfl_sync(0xffffffffu, s1, r << 2);
                inv[r] = __shfl_sync(0xffffffffu, i1, r << 2);
            }
        } else {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int r = 0; r < NMAX; ++r)
                    amax[r] = fmax_nan(amax[r], __shfl_xor_sync(0xffffffffu, amax[r], o));
#pragma unroll
            for (int r = 0; r < NMAX; ++r) {
                sc[r] = amax[r] != amax[r] ? __uint_as_float(0x7fffffffu) : __fdiv_rn(amax[r], 127.0f);
                inv[r] = __frcp_rn(sc[r]);
            }
        }
#pragma unroll
        for (int r = 0; r < NMAX; ++r) {
            const float s = sc[r];
            const bool fast = s > 0.0f && inv[r] < __uint_as_float(0x7f800000u); // warp-uniform
            float q[EPL];
            if (fast) {
                // q = round(u * (1/s)) unless some element of the lane lies
                // within 2^-14 of a tie; then the lane takes the exact
                // quotient for all of them (see quantize_fast)
                float worst = 0.0f;
#pragma unroll
                for (int j = 0; j < EPL; ++j) {
                    const float t = __fmul_rn(v[r][j], inv[r]);
                    q[j] = rintf(t);
                    worst = fmaxf(worst, fabsf(t - q[j]));
                }
                if (worst > 0.49993896484375f)
#pragma unroll
                    for (int j = 0; j < EPL; ++j)
                        q[j] = rintf(__fdiv_rn(v[r][j], s));
            } else {
#pragma unroll
                for (int j = 0; j < EPL; ++j)
                    q[j] = s > 0.0f ? rintf(__fdiv_rn(v[r][j], s)) : (s == 0.0f ? 0.0f : s);
            }
#pragma unroll
            for (int j = 0; j < EPL; ++j) {
                const float u = v[r][j];
                v[r][j] = __fmul_rn(q[j], s);
                ee[r][j] = __fsub_rn(u, v[r][j]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NMAX; ++r)
        if (r < N)
            store_f<EPL>(p.res[r], i0, valid, vec, ee[r]);

    // ring-order fold in fp32: chunk c from rank c, then c+1, ..., c-1
    const uint32_t c0 = valid > 0 ? chunk_of<NMAX>(p, i0) : 0u;
    // all of the lane's elements in chunk c0 (the rule; a chunk boundary inside
    // a lane is the exception)
    const bool one_chunk = valid == 0 || c0 + 1 >= (uint32_t)N || i0 + (uint64_t)(valid - 1) < p.coff[c0 + 1];
    float accv[EPL];
    if (N == NMAX && one_chunk) {
        // every rank present: one static fold per rotation start, for all of
        // the lane's elements at once
        switch (c0) {
#define CCL_FOLD_CASE(C)                                                                                           \
    case C:                                                                                                            \
        _Pragma("unroll") for (int j = 0; j < EPL; ++j) {                                                              \
            float a = v[C % NMAX][j];                                                                                  \
            _Pragma("unroll") for (int k = 1; k < NMAX; ++k) a = __fadd_rn(v[(C + k) % NMAX][j], a);                  \
            accv[j] = a;                                                                                               \
        }                                                                                                              \
        break;
            CCL_FOLD_CASE(0) CCL_FOLD_CASE(1) CCL_FOLD_CASE(2) CCL_FOLD_CASE(3)
            CCL_FOLD_CASE(4) CCL_FOLD_CASE(5) CCL_FOLD_CASE(6) CCL_FOLD_CASE(7)
            CCL_FOLD_CASE(8) CCL_FOLD_CASE(9) CCL_FOLD_CASE(10) CCL_FOLD_CASE(11)
            CCL_FOLD_CASE(12) CCL_FOLD_CASE(13) CCL_FOLD_CASE(14) CCL_FOLD_CASE(15)
#undef CCL_FOLD_CASE
        default:
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                accv[j] = 0.0f;
        }
    } else {
        uint32_t c = c0;
#pragma unroll
        for (int j = 0; j < EPL; ++j) {
            while (c + 1 < (uint32_t)N && i0 + j >= p.coff[c + 1])
                ++c;
            float acc = 0.0f;
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                if (r < N && r >= (int)c)
                    acc = r == (int)c ? v[r][j] : __fadd_rn(v[r][j], acc);
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                if (r < (int)c)
                    acc = __fadd_rn(v[r][j], acc);
            accv[j] = acc;
        }
    }
    uint32_t outb[EPL];
#pragma unroll
    for (int j = 0; j < EPL; ++j) {
        float acc = accv[j];
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
                gstore<uint4>(static_cast<uint32_t *>(p.grads[r]) + i0, make_uint4(w[0], w[1], w[2], w[3]));
            else if (DT == DT_FP32)
                gstore<uint2>(static_cast<uint32_t *>(p.grads[r]) + i0, make_uint2(w[0], w[1]));
            else if (EPL == 4)
                gstore<uint2>(static_cast<uint16_t *>(p.grads[r]) + i0, make_uint2(w[0], w[2]));
            else
                gstore<uint32_t>(static_cast<uint16_t *>(p.grads[r]) + i0, w[0]);
        } else {
#pragma unroll
            for (int j = 0; j < EPL; ++j)
                if (j < valid)
                    st_elem<DT>(p.grads[r], i0 + j, outb[j]);
        }
    }
}

template <int DT, int EPL, int NMAX, int COMP>
__global__ void __launch_bounds__(kThreads, NMAX <= 8 ? 3 : 1) compressed_allreduce_kernel(const __grid_constant__ CompParams p)
{
    if (COMP == COMP_TOPK)
        chain_entry(); // the select's threshold comes from the kernels before
    constexpr int B = 32 * EPL; // compression block
    const int lane = threadIdx.x & 31;
    const uint64_t blk = p.first_block + (((uint64_t)blockIdx.x * kThreads + threadIdx.x) >> 5);
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
    uint32_t tau[NMAX];
    load_tau<NMAX, COMP>(p, tau);
    compress_fold_store<DT, EPL, NMAX, COMP>(p, i0, valid, vec, v, ee, tau);
}

// ------------------------------------------------------------------ pipelined form (N <= 8)
//
// Persistent CTAs walk tiles of 8 compression blocks (one per warp).  While a
// warp computes tile i from shared memory, cp.async is already copying tile
// i+1's gradients and residuals into the other stage, so memory latency hides
// behind the compute.  Each lane copies exactly the words it later reads, so
// its own cp.async.wait_group is the only synchronisation needed.  Only whole,
// aligned blocks come here; the tail block goes to the kernel above.

__device__ __forceinline__ void cp_async(void *smem, const void *gmem, int bytes)
{
    if (!dbg_ok(gmem, (size_t)bytes))
        return; // debug builds: outside the call's buffers
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    if (bytes == 16)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
    else if (bytes == 8)
        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(sa), "l"(gmem) : "memory");
    else
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}

// Shape of the pipelined kernel: 4 warps per CTA and 3 cp.async stages (two
// tiles ahead) -- 72 KB of shared memory for bf16, three CTAs per SM.  Measured
// against 8 warps x 2 stages (the first form) and the neighbours: 6,462 GB/s
// vs 6,231 (256x2), 6,232 (128x2), 5,990 (128x4), 5,927 (256x3), 6,424 (64x3),
// 6,423 (192x3); N=8 bf16, 64 Mi elements per rank.
constexpr int kPipeThreads = 128; // threads per CTA of the pipelined kernel
constexpr int kPipeStages = 3;    // cp.async stages in flight per warp (tiles ahead: stages - 1)

template <int DT, int EPL> struct PipeLayout {
    static constexpr int kWarps = kPipeThreads / 32;
    static constexpr int kGB = EPL * DType<DT>::kSize; // gradient bytes per lane and rank
    static constexpr int kEB = EPL * 4;                // residual bytes per lane and rank
    static constexpr size_t kStageG = (size_t)kWarps * 8 * 32 * kGB;
    static constexpr size_t kStage = (size_t)kWarps * 8 * 32 * (kGB + kEB);
    static constexpr size_t kBytes = kPipeStages * kStage;
};

template <int DT, int EPL, int COMP>
__global__ void __launch_bounds__(kPipeThreads) compressed_pipe_kernel(const __grid_constant__ CompParams p)
{
    if (COMP == COMP_TOPK)
        chain_entry(); // the select's threshold comes from the kernels before
    using Lay = PipeLayout<DT, EPL>;
    constexpr int B = 32 * EPL;
    constexpr int NMAX = 8;
    extern __shared__ __align__(16) unsigned char smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int N = p.nranks;
    const uint64_t ntiles = (p.nfull + Lay::kWarps - 1) / Lay::kWarps;

    auto gslot = [&](int st, int r) {
        return smem + (size_t)st * Lay::kStage + (((size_t)warp * 8 + r) * 32 + lane) * Lay::kGB;
    };
    auto eslot = [&](int st, int r) {
        return smem + (size_t)st * Lay::kStage + Lay::kStageG + (((size_t)warp * 8 + r) * 32 + lane) * Lay::kEB;
    };
    auto issue = [&](uint64_t t, int st) {
        const uint64_t b = t * Lay::kWarps + warp;
        if (b < p.nfull) {
            const uint64_t i0 = b * B + (uint64_t)lane * EPL;
#pragma unroll
            for (int r = 0; r < NMAX; ++r)
                if (r < N) {
                    cp_async(gslot(st, r), static_cast<const char *>(p.grads[r]) + i0 * DType<DT>::kSize, Lay::kGB);
                    cp_async(eslot(st, r), p.res[r] + i0, Lay::kEB);
                }
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    uint64_t t = blockIdx.x;
    if (t >= ntiles)
        return;
    uint32_t tau[NMAX];
    load_tau<NMAX, COMP>(p, tau);
    for (int k = 0; k < kPipeStages - 1; ++k)
        issue(t + (uint64_t)k * gridDim.x, k);
    for (int it = 0; t < ntiles; ++it, t += gridDim.x) {
        // tiles past the end issue empty groups, which keeps the group count uniform
        issue(t + (uint64_t)(kPipeStages - 1) * gridDim.x, (it + kPipeStages - 1) % kPipeStages);
        asm volatile("cp.async.wait_group %0;" ::"n"(kPipeStages - 1) : "memory");
        const uint64_t b = t * Lay::kWarps + warp;
        if (b >= p.nfull)
            continue;
        const uint64_t i0 = b * B + (uint64_t)lane * EPL;
        const int st = it % kPipeStages;
        float v[NMAX][EPL], ee[NMAX][EPL];
#pragma unroll
        for (int r = 0; r < NMAX; ++r) {
            if (r < N) {
                if (DT == DT_FP32) {
#pragma unroll
                    for (int j = 0; j < EPL; ++j)
                        v[r][j] = reinterpret_cast<const float *>(gslot(st, r))[j];
                } else {
#pragma unroll
                    for (int j = 0; j < EPL; j += 2) {
                        const uint32_t w = reinterpret_cast<const uint32_t *>(gslot(st, r))[j / 2];
                        v[r][j] = __uint_as_float(w << 16);
                        v[r][j + 1] = __uint_as_float(w & 0xffff0000u);
                    }
                }
#pragma unroll
                for (int j = 0; j < EPL; ++j)
                    ee[r][j] = reinterpret_cast<const float *>(eslot(st, r))[j];
            } else {
#pragma unroll
                for (int j = 0; j < EPL; ++j)
                    v[r][j] = ee[r][j] = 0.0f;
            }
        }
        compress_fold_store<DT, EPL, NMAX, COMP>(p, i0, EPL, true, v, ee, tau);
    }
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// The pipelined kernel needs more than 48 KB of dynamic shared memory, which
// is opted into per kernel and per device; the persistent grid is one full
// wave on that device.  Both are worked out once per (kernel, device).
struct PipeConfig {
    bool ready = false;
    int ctas = 0; // SMs x resident CTAs per SM
};
static std::mutex g_pipe_cfg_mu;

template <int DT, int EPL, int COMP>
static cudaError_t pipe_grid(int *ctas)
{
    using Lay = PipeLayout<DT, EPL>;
    static std::unordered_map<int, PipeConfig> cfg; // per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_pipe_cfg_mu);
    PipeConfig &c = cfg[dev];
    if (!c.ready) {
        int sms = 0, per_sm = 0;
        if ((e = cudaFuncSetAttribute(compressed_pipe_kernel<DT, EPL, COMP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)Lay::kBytes)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, compressed_pipe_kernel<DT, EPL, COMP>, kPipeThreads,
                                                               Lay::kBytes)) != cudaSuccess)
            return e;
        c.ctas = sms * (per_sm > 0 ? per_sm : 1);
        c.ready = true;
    }
    *ctas = c.ctas;
    return cudaSuccess;
}

template <int DT, int EPL, int COMP>
static cudaError_t launch_pipe_t(const CompParams &p, cudaStream_t stream)
{
    using Lay = PipeLayout<DT, EPL>;
    int ctas = 0;
    if (cudaError_t e = pipe_grid<DT, EPL, COMP>(&ctas))
        return e;
    const uint64_t ntiles = (p.nfull + Lay::kWarps - 1) / Lay::kWarps;
    uint64_t grid = (uint64_t)ctas;
    if (grid > ntiles)
        grid = ntiles;
    if (grid == 0)
        return cudaSuccess;
    if (COMP == COMP_TOPK) { // chained after the select's kernels
        cudaError_t e = launch_chained<CompParams>(compressed_pipe_kernel<DT, EPL, COMP>, dim3((unsigned)grid),
                                                   dim3(kPipeThreads), Lay::kBytes, stream, p);
        if (e != cudaSuccess)
            return e;
    } else {
        compressed_pipe_kernel<DT, EPL, COMP><<<(unsigned)grid, kPipeThreads, Lay::kBytes, stream>>>(p);
    }
    count_launches(1);
    return cudaGetLastError();
}

template <int DT, int EPL, int NMAX, int COMP>
static cudaError_t launch_comp_t(const CompParams &p, cudaStream_t stream)
{
    constexpr int B = 32 * EPL;
    const uint64_t nblocks = (p.K + B - 1) / B;
    if (nblocks <= p.first_block)
        return cudaSuccess;
    const uint64_t warps = nblocks - p.first_block;
    const uint64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
    if (blocks > 0x7fffffffull)
        return cudaErrorInvalidValue;
    if (COMP == COMP_TOPK) { // chained after the select's kernels
        cudaError_t e = launch_chained<CompParams>(compressed_allreduce_kernel<DT, EPL, NMAX, COMP>,
                                                   dim3((unsigned)blocks), dim3(kThreads), 0, stream, p);
        if (e != cudaSuccess)
            return e;
    } else {
        compressed_allreduce_kernel<DT, EPL, NMAX, COMP><<<(unsigned)blocks, kThreads, 0, stream>>>(p);
    }
    count_launches(1);
    return cudaGetLastError();
}

// N <= 8 with aligned buffers: whole blocks through the pipelined kernel, the
// last partial block (if any) through the direct one.  Otherwise all direct.
template <int DT, int EPL, int COMP>
static cudaError_t launch_comp_dt(CompParams p, cudaStream_t stream)
{
    constexpr int B = 32 * EPL;
    if (p.nranks <= 8 && p.vec_ok) {
        p.nfull = p.K / B;
        if (p.nfull) {
            cudaError_t e = launch_pipe_t<DT, EPL, COMP>(p, stream);
            if (e != cudaSuccess)
                return e;
        }
        p.first_block = p.nfull;
        return launch_comp_t<DT, EPL, 8, COMP>(p, stream);
    }
    p.first_block = 0;
    return p.nranks <= 8 ? launch_comp_t<DT, EPL, 8, COMP>(p, stream) : launch_comp_t<DT, EPL, 16, COMP>(p, stream);
}

cudaError_t launch_compressed_allreduce(int dt, bool avg, int comp, int block, float threshold,
                                        void *const *grads, float *const *res, int nranks, uint64_t count,
                                        const uint32_t *tau, cudaStream_t stream)
{
    if (nranks > kCompMaxRanks)
        return cudaErrorInvalidValue;
    CompParams p;
    const int epl = (comp == COMP_THRESHOLD || comp == COMP_TOPK) ? 4 : block / 32;
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
    for (int c = 0; c <= kCompMaxRanks; ++c)
        p.coff[c] = c < nranks ? p.part.off((uint32_t)c) : count;
    p.K = count;
    p.nranks = nranks;
    p.comp = comp;
    p.threshold = threshold;
    p.n_f = avg ? (float)nranks : 0.0f;
    p.pow2 = (nranks & (nranks - 1)) == 0 ? 1 : 0;
    p.inv_n = 1.0f / (float)nranks;
    p.vec_ok = vec ? 1 : 0;
    p.first_block = 0;
    p.nfull = 0;
    p.tau = tau;
    // one instantiation per compressor: each kernel carries only its own arithmetic
    if (comp == COMP_THRESHOLD)
        return dt == DT_FP32 ? launch_comp_dt<DT_FP32, 4, COMP_THRESHOLD>(p, stream)
                             : launch_comp_dt<DT_BF16, 4, COMP_THRESHOLD>(p, stream);
    if (comp == COMP_TOPK)
        return dt == DT_FP32 ? launch_comp_dt<DT_FP32, 4, COMP_TOPK>(p, stream)
                             : launch_comp_dt<DT_BF16, 4, COMP_TOPK>(p, stream);
    if (dt == DT_FP32)
        return epl == 4 ? launch_comp_dt<DT_FP32, 4, COMP_INT8_BLOCK>(p, stream)
                        : launch_comp_dt<DT_FP32, 2, COMP_INT8_BLOCK>(p, stream);
    return epl == 4 ? launch_comp_dt<DT_BF16, 4, COMP_INT8_BLOCK>(p, stream)
                    : launch_comp_dt<DT_BF16, 2, COMP_INT8_BLOCK>(p, stream);
}

} // namespace ccl
