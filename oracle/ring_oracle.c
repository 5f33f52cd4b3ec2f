/*
 * ring_oracle.c -- CPU oracle for the ring collectives.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may load, link or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header or table with the CUDA library.
 *
 * Plain, slow and step by step: N simulated ranks each own a buffer of K
 * elements; every ring step snapshots what each rank sends, then applies what
 * each rank receives, exactly as the pages' CPU ring simulator does (Lesson 3
 * "Distributed communication primitives", fill-in exercise and reference
 * solution).  Arithmetic is IEEE fp32 with round-to-nearest-even, followed by a
 * round to the buffer type after every hop (fp32: identity; bf16: RNE from the
 * IEEE definition).  Built with -O2 -ffp-contract=off and without fast-math, so
 * no FMA contraction, flush-to-zero or reassociation can creep in.
 *
 * Conventions fixed here (the pages leave them open):
 *   - chunk c of a K-element buffer has len_c = K/N + (c < K%N) elements, the
 *     first K%N chunks taking one extra element;
 *   - a NaN produced by an fp32 operation is the canonical quiet NaN 0x7FFFFFFF;
 *     rounding a NaN to bf16 keeps its sign and top payload bits and sets the
 *     quiet bit;
 *   - MAX: NaN if either operand is NaN, else the larger, and for +0 vs -0 the
 *     bitwise AND of the two (so +0 wins); MIN: NaN if either is NaN, else the
 *     smaller, and for +0 vs -0 the bitwise OR (so -0 wins);
 *   - AVG: SUM around the ring, then one fp32 division by N at the rank that
 *     holds the finished chunk, rounded to the buffer type, before the gather;
 *   - AVG_PREMUL (NCCL's pre-multiplied sum, Collective Communication,
 *     libraries section): every rank first multiplies each of its values by
 *     the fp32 reciprocal of N (correctly rounded), rounds the product to the
 *     buffer type, and the ring then SUMs those; nothing is divided at the end.
 *     Only the ring order takes it; the other orders reject it.
 *
 * Parity pins live in tests/test_oracle_*.py; see each function's comment for
 * which passage it follows.
 */
#define _POSIX_C_SOURCE 200809L /* pthread barriers */
#include <errno.h>
#include <pthread.h>
#include <stdint.h>
#include <time.h>
#include <stdlib.h>
#include <string.h>

#define OR_FP32 0
#define OR_BF16 1

#define OR_SUM 0
#define OR_AVG 1
#define OR_MAX 2
#define OR_PROD 3
#define OR_MIN 4
#define OR_AVGP 5 /* AVG by pre-multiplication: every contribution times rn(1/N), then SUM */

#define OR_OK 0
#define OR_EINVAL 1
#define OR_ENOMEM 2
#define OR_ETIMEDOUT 3

/* ------------------------------------------------------------------ */
/* scalar arithmetic                                                   */
/* ------------------------------------------------------------------ */

static float bits_to_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static int f32_bits_is_nan(uint32_t u) { return (u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0; }

/* IEEE-754 round-to-nearest, ties-to-even, of an fp32 bit pattern to bf16
 * (keep the top 16 bits; the dropped 16 bits decide: above half rounds the
 * magnitude up, below half truncates, exactly half rounds to the even result).
 * The magnitude increment carries into the exponent, so the largest finite
 * values round to infinity and subnormals round within the subnormal range. */
uint16_t oracle_round_bf16(uint32_t u)
{
    if (f32_bits_is_nan(u))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* Bulk form of oracle_round_bf16 (for exhaustive pattern checks). */
void oracle_round_bf16_array(const uint32_t *in, uint16_t *out, uint64_t n)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = oracle_round_bf16(in[i]);
}

/* bf16 -> fp32 is exact: the bf16 pattern is the top half of the fp32 one. */
static uint32_t widen_bits(uint32_t stored, int dtype)
{
    return dtype == OR_BF16 ? (stored << 16) : stored;
}

static uint32_t narrow_bits(uint32_t f32bits, int dtype)
{
    return dtype == OR_BF16 ? (uint32_t)oracle_round_bf16(f32bits) : f32bits;
}

/* One fp32 operation of the ring's reduction, IEEE round-to-nearest-even. */
static uint32_t op_f32(uint32_t a_bits, uint32_t b_bits, int op)
{
    float a = bits_to_f32(a_bits), b = bits_to_f32(b_bits);
    uint32_t r;
    switch (op) {
    case OR_SUM:
    case OR_AVG:
    case OR_AVGP:
        r = f32_to_bits(a + b);
        break;
    case OR_PROD:
        r = f32_to_bits(a * b);
        break;
    case OR_MAX:
        if (f32_bits_is_nan(a_bits) || f32_bits_is_nan(b_bits))
            r = 0x7fffffffu;
        else if (a > b)
            r = a_bits;
        else if (b > a)
            r = b_bits;
        else
            r = a_bits & b_bits; /* equal: identical bits, or +0 vs -0 -> +0 */
        break;
    case OR_MIN:
        if (f32_bits_is_nan(a_bits) || f32_bits_is_nan(b_bits))
            r = 0x7fffffffu;
        else if (a < b)
            r = a_bits;
        else if (b < a)
            r = b_bits;
        else
            r = a_bits | b_bits; /* equal: identical bits, or +0 vs -0 -> -0 */
        break;
    default:
        r = 0x7fffffffu;
    }
    if (f32_bits_is_nan(r))
        r = 0x7fffffffu;
    return r;
}

/* x_local (+) x_incoming, rounded to the buffer type: one ring hop
 * ("add what was received into the matching local chunk"). */
static uint32_t hop(uint32_t local, uint32_t incoming, int dtype, int op)
{
    return narrow_bits(op_f32(widen_bits(local, dtype), widen_bits(incoming, dtype), op), dtype);
}

/* AVG's single division by N, done once on the finished sum. */
static uint32_t avg_scale(uint32_t v, int N, int dtype)
{
    float x = bits_to_f32(widen_bits(v, dtype));
    uint32_t r = f32_to_bits(x / (float)N);
    if (f32_bits_is_nan(r))
        r = 0x7fffffffu;
    return narrow_bits(r, dtype);
}

/* AVG by pre-multiplication (NCCL's pre-multiplied sum, Collective
 * Communication, libraries section): each contribution x becomes
 * round_T(x * rn(1/N)) -- one fp32 multiply by the correctly rounded
 * reciprocal -- and the scaled contributions are summed around the ring with
 * no division at the end. */
static uint32_t premul(uint32_t v, int N, int dtype)
{
    const float inv = 1.0f / (float)N;
    uint32_t r = f32_to_bits(bits_to_f32(widen_bits(v, dtype)) * inv);
    if (f32_bits_is_nan(r))
        r = 0x7fffffffu;
    return narrow_bits(r, dtype);
}

/* what a rank puts into the ring for operator op */
static uint32_t contrib(uint32_t v, int N, int dtype, int op)
{
    return op == OR_AVGP ? premul(v, N, dtype) : v;
}

static size_t esize(int dtype) { return dtype == OR_BF16 ? 2 : 4; }

static uint32_t load(const void *buf, int dtype, uint64_t i)
{
    if (dtype == OR_BF16)
        return ((const uint16_t *)buf)[i];
    return ((const uint32_t *)buf)[i];
}

static void store(void *buf, int dtype, uint64_t i, uint32_t v)
{
    if (dtype == OR_BF16)
        ((uint16_t *)buf)[i] = (uint16_t)v;
    else
        ((uint32_t *)buf)[i] = v;
}

static int mod(int64_t a, int n) { int64_t r = a % n; return (int)(r < 0 ? r + n : r); }

static int bad_args(int N, int dtype, int op)
{
    return N < 1 || (dtype != OR_FP32 && dtype != OR_BF16) || op < OR_SUM || op > OR_AVGP;
}

/* ------------------------------------------------------------------ */
/* partition and schedule                                              */
/* ------------------------------------------------------------------ */

/* Split K elements into N contiguous chunks; the first K mod N chunks get one
 * extra element.  (The pages require K divisible by N -- Lesson 3 splits each
 * rank's tensor into N equal blocks -- this is the plainest extension.) */
void oracle_partition(uint64_t K, int N, uint64_t *off, uint64_t *len)
{
    uint64_t q = K / (uint64_t)N, rem = K % (uint64_t)N, o = 0;
    for (int c = 0; c < N; ++c) {
        len[c] = q + ((uint64_t)c < rem ? 1 : 0);
        off[c] = o;
        o += len[c];
    }
}

/* The ring's step table, laid out [phase][s][rank][3] = {send chunk, recv chunk,
 * source rank}.  ReduceScatter step s: rank i sends chunk (i-s) mod N to its
 * right neighbour and receives chunk (i-1-s) mod N from its left one.
 * AllGather step s: rank i forwards chunk (i+1-s) mod N and stores chunk
 * (i-s) mod N.  (Collectives and sharded matmul, "ring ReduceScatter"; AllReduce
 * survey, Ring AllReduce phase 1; Lesson 3 reference solution.) */
void oracle_ring_schedule(int N, int32_t *tab)
{
    int steps = N - 1;
    for (int phase = 0; phase < 2; ++phase)
        for (int s = 0; s < steps; ++s)
            for (int i = 0; i < N; ++i) {
                int32_t *e = tab + (((size_t)phase * steps + s) * N + i) * 3;
                if (phase == 0) {
                    e[0] = mod((int64_t)i - s, N);
                    e[1] = mod((int64_t)i - 1 - s, N);
                } else {
                    e[0] = mod((int64_t)i + 1 - s, N);
                    e[1] = mod((int64_t)i - s, N);
                }
                e[2] = mod((int64_t)i - 1, N);
            }
}

/* ------------------------------------------------------------------ */
/* step-faithful ring phases on N in-place rank buffers                */
/* ------------------------------------------------------------------ */

/* ReduceScatter phase, N-1 steps.  All sends of a step are snapshotted first,
 * then each rank adds what it received into its matching chunk, operand order
 * (local, incoming).  Afterwards rank i holds the finished chunk (i+1) mod N. */
static int rs_phase(void **buf, int N, const uint64_t *off, const uint64_t *len,
                    int dtype, int op, uint64_t *sent, void *snap, uint64_t stride)
{
    size_t es = esize(dtype);
    if (op == OR_AVGP) /* every rank scales its own contribution before it enters the ring */
        for (int i = 0; i < N; ++i)
            for (int c = 0; c < N; ++c)
                for (uint64_t e = off[c]; e < off[c] + len[c]; ++e)
                    store(buf[i], dtype, e, premul(load(buf[i], dtype, e), N, dtype));
    for (int s = 0; s < N - 1; ++s) {
        for (int i = 0; i < N; ++i) {
            int c = mod((int64_t)i - s, N);
            memcpy((char *)snap + (size_t)i * stride * es, (char *)buf[i] + off[c] * es, len[c] * es);
            if (sent)
                sent[i] += len[c];
        }
        for (int i = 0; i < N; ++i) {
            int c = mod((int64_t)i - 1 - s, N);
            int src = mod((int64_t)i - 1, N);
            const void *in = (const char *)snap + (size_t)src * stride * es;
            for (uint64_t e = 0; e < len[c]; ++e) {
                uint64_t g = off[c] + e;
                store(buf[i], dtype, g, hop(load(buf[i], dtype, g), load(in, dtype, e), dtype, op));
            }
        }
    }
    if (op == OR_AVG)
        for (int i = 0; i < N; ++i) {
            int c = mod((int64_t)i + 1, N);
            for (uint64_t e = 0; e < len[c]; ++e)
                store(buf[i], dtype, off[c] + e, avg_scale(load(buf[i], dtype, off[c] + e), N, dtype));
        }
    return OR_OK;
}

/* AllGather phase after ReduceScatter, N-1 steps: rank i forwards chunk
 * (i+1-s) mod N and stores the chunk (i-s) mod N it receives. */
static void ag_phase_after_rs(void **buf, int N, const uint64_t *off, const uint64_t *len,
                              int dtype, uint64_t *sent, void *snap, uint64_t stride)
{
    size_t es = esize(dtype);
    for (int s = 0; s < N - 1; ++s) {
        for (int i = 0; i < N; ++i) {
            int c = mod((int64_t)i + 1 - s, N);
            memcpy((char *)snap + (size_t)i * stride * es, (char *)buf[i] + off[c] * es, len[c] * es);
            if (sent)
                sent[i] += len[c];
        }
        for (int i = 0; i < N; ++i) {
            int c = mod((int64_t)i - s, N);
            int src = mod((int64_t)i - 1, N);
            memcpy((char *)buf[i] + off[c] * es, (char *)snap + (size_t)src * stride * es, len[c] * es);
        }
    }
}

/* Ring AllReduce, step by step, in place on buf[0..N-1] (K elements each).
 * ReduceScatter phase, AVG scaling at the holders, AllGather phase.
 * sent[i] (optional) accumulates the number of elements rank i sent, which for
 * K divisible by N is 2(N-1)K/N (Lesson 3, traffic check). */
int oracle_ring_allreduce(void **buf, int N, uint64_t K, int dtype, int op, uint64_t *sent)
{
    if (bad_args(N, dtype, op))
        return OR_EINVAL;
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)N), *len = malloc(sizeof(uint64_t) * (size_t)N);
    uint64_t stride = K / (uint64_t)N + 1;
    void *snap = malloc((size_t)N * stride * esize(dtype));
    if (!off || !len || !snap) {
        free(off); free(len); free(snap);
        return OR_ENOMEM;
    }
    oracle_partition(K, N, off, len);
    if (sent)
        memset(sent, 0, sizeof(uint64_t) * (size_t)N);
    rs_phase(buf, N, off, len, dtype, op, sent, snap, stride);
    ag_phase_after_rs(buf, N, off, len, dtype, sent, snap, stride);
    free(off); free(len); free(snap);
    return OR_OK;
}

/* The same ring with the ranks spread over threads, for timing the CPU
 * baseline on several cores (N rank-threads with a barrier per step).  Thread
 * t owns ranks [r0, r1).  Every step is: all threads snapshot what their ranks
 * send, a barrier, all threads apply what their ranks receive, a barrier --
 * the operations of oracle_ring_allreduce in the same order for every
 * element, so the bits are the same (pinned by a test). */
typedef struct {
    pthread_mutex_t mu;
    pthread_cond_t cv;
    int go; /* 0: wait, 1: run, -1: leave without running */
} start_gate;

/* A barrier whose wait gives up after a deadline.  A rank that never arrives
 * (it left, or failed) breaks the barrier for everyone: every wait from then
 * on returns at once with an error, so no thread hangs (the pages: a rank that
 * exits early hangs the others until a timeout; Lesson 3, pitfalls). */
typedef struct {
    pthread_mutex_t mu;
    pthread_cond_t cv;
    unsigned n, arrived, generation;
    int broken;
    long timeout_ms;
} timed_barrier;

static int timed_barrier_wait(timed_barrier *b)
{
    pthread_mutex_lock(&b->mu);
    if (b->broken) {
        pthread_mutex_unlock(&b->mu);
        return -1;
    }
    const unsigned gen = b->generation;
    if (++b->arrived == b->n) {
        b->arrived = 0;
        ++b->generation;
        pthread_cond_broadcast(&b->cv);
        pthread_mutex_unlock(&b->mu);
        return 0;
    }
    struct timespec until;
    clock_gettime(CLOCK_REALTIME, &until);
    until.tv_sec += b->timeout_ms / 1000;
    until.tv_nsec += (b->timeout_ms % 1000) * 1000000L;
    if (until.tv_nsec >= 1000000000L) {
        until.tv_sec += 1;
        until.tv_nsec -= 1000000000L;
    }
    int rc = 0;
    while (b->generation == gen && !b->broken && rc != ETIMEDOUT)
        rc = pthread_cond_timedwait(&b->cv, &b->mu, &until);
    const int ok = b->generation != gen;
    if (!ok && !b->broken) {
        b->broken = 1; /* this wait ran out: release everyone */
        pthread_cond_broadcast(&b->cv);
    }
    pthread_mutex_unlock(&b->mu);
    return ok ? 0 : -1;
}

typedef struct {
    void **buf;
    int N, dtype, op, r0, r1;
    const uint64_t *off, *len;
    char *snap;
    uint64_t stride;
    timed_barrier *bar;
    start_gate *gate;
    int withhold; /* this thread leaves before its first send (a failed rank) */
} ring_part;

#define RING_SYNC(p)                                                                                          \
    do {                                                                                                               \
        if (timed_barrier_wait((p)->bar) != 0)                                                                          \
            return NULL;                                                                                               \
    } while (0)

static void *ring_part_run(void *arg)
{
    const ring_part *p = (const ring_part *)arg;
    const int N = p->N;
    const size_t es = esize(p->dtype);
    if (p->withhold)
        return NULL;
    if (p->op == OR_AVGP) /* each thread scales its own ranks' contributions */
        for (int i = p->r0; i < p->r1; ++i)
            for (int c = 0; c < N; ++c)
                for (uint64_t e = p->off[c]; e < p->off[c] + p->len[c]; ++e)
                    store(p->buf[i], p->dtype, e, premul(load(p->buf[i], p->dtype, e), N, p->dtype));
    for (int s = 0; s < N - 1; ++s) { /* ReduceScatter phase */
        for (int i = p->r0; i < p->r1; ++i) {
            int c = mod((int64_t)i - s, N);
            memcpy(p->snap + (size_t)i * p->stride * es, (char *)p->buf[i] + p->off[c] * es, p->len[c] * es);
        }
        RING_SYNC(p);
        for (int i = p->r0; i < p->r1; ++i) {
            int c = mod((int64_t)i - 1 - s, N);
            const void *in = p->snap + (size_t)mod((int64_t)i - 1, N) * p->stride * es;
            for (uint64_t e = 0; e < p->len[c]; ++e) {
                uint64_t g = p->off[c] + e;
                store(p->buf[i], p->dtype, g,
                      hop(load(p->buf[i], p->dtype, g), load(in, p->dtype, e), p->dtype, p->op));
            }
        }
        RING_SYNC(p);
    }
    if (p->op == OR_AVG)
        for (int i = p->r0; i < p->r1; ++i) {
            int c = mod((int64_t)i + 1, N);
            for (uint64_t e = 0; e < p->len[c]; ++e)
                store(p->buf[i], p->dtype, p->off[c] + e,
                      avg_scale(load(p->buf[i], p->dtype, p->off[c] + e), N, p->dtype));
        }
    RING_SYNC(p);
    for (int s = 0; s < N - 1; ++s) { /* AllGather phase */
        for (int i = p->r0; i < p->r1; ++i) {
            int c = mod((int64_t)i + 1 - s, N);
            memcpy(p->snap + (size_t)i * p->stride * es, (char *)p->buf[i] + p->off[c] * es, p->len[c] * es);
        }
        RING_SYNC(p);
        for (int i = p->r0; i < p->r1; ++i) {
            int c = mod((int64_t)i - s, N);
            memcpy((char *)p->buf[i] + p->off[c] * es, p->snap + (size_t)mod((int64_t)i - 1, N) * p->stride * es,
                   p->len[c] * es);
        }
        RING_SYNC(p);
    }
    return NULL;
}

/* Helper threads wait at the gate until every thread exists, so that a failed
 * pthread_create never leaves some of them waiting at the barrier. */
static void *ring_part_gated(void *arg)
{
    const ring_part *p = (const ring_part *)arg;
    pthread_mutex_lock(&p->gate->mu);
    while (p->gate->go == 0)
        pthread_cond_wait(&p->gate->cv, &p->gate->mu);
    const int go = p->gate->go;
    pthread_mutex_unlock(&p->gate->mu);
    return go > 0 ? ring_part_run(arg) : NULL;
}

static void open_gate(start_gate *g, int go)
{
    pthread_mutex_lock(&g->mu);
    g->go = go;
    pthread_cond_broadcast(&g->cv);
    pthread_mutex_unlock(&g->mu);
}

/* withhold_rank >= 0: the thread that owns that rank leaves before its first
 * send, as a failed rank would; the others' waits then run out after
 * timeout_ms and the call returns OR_ETIMEDOUT (the buffers are left
 * partly updated).  The plain call waits up to a minute per step. */
int oracle_ring_allreduce_threads_ex(void **buf, int N, uint64_t K, int dtype, int op, int nthreads,
                                     int withhold_rank, long timeout_ms)
{
    if (bad_args(N, dtype, op) || nthreads < 1 || timeout_ms < 1 || withhold_rank >= N)
        return OR_EINVAL;
    if (withhold_rank >= 0 && (nthreads < 2 || N < 2))
        return OR_EINVAL; /* a failure needs another thread to notice it */
    if (nthreads > N)
        nthreads = N;
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)N), *len = malloc(sizeof(uint64_t) * (size_t)N);
    uint64_t stride = K / (uint64_t)N + 1;
    char *snap = malloc((size_t)N * stride * esize(dtype));
    ring_part *parts = malloc(sizeof(ring_part) * (size_t)nthreads);
    pthread_t *th = malloc(sizeof(pthread_t) * (size_t)nthreads);
    timed_barrier bar = {PTHREAD_MUTEX_INITIALIZER, PTHREAD_COND_INITIALIZER, (unsigned)nthreads, 0, 0, 0, timeout_ms};
    start_gate gate = {PTHREAD_MUTEX_INITIALIZER, PTHREAD_COND_INITIALIZER, 0};
    int started = 1;
    if (!off || !len || !snap || !parts || !th) {
        free(off); free(len); free(snap); free(parts); free(th);
        return OR_ENOMEM;
    }
    oracle_partition(K, N, off, len);
    for (int t = 0; t < nthreads; ++t) {
        const int r0 = (int)((int64_t)N * t / nthreads), r1 = (int)((int64_t)N * (t + 1) / nthreads);
        ring_part q = {buf, N, dtype, op, r0, r1, off, len, snap, stride, &bar, &gate,
                       withhold_rank >= r0 && withhold_rank < r1};
        parts[t] = q;
    }
    while (started < nthreads && pthread_create(&th[started], NULL, ring_part_gated, &parts[started]) == 0)
        ++started;
    const int all = started == nthreads;
    open_gate(&gate, all ? 1 : -1);
    if (all)
        ring_part_run(&parts[0]); /* the calling thread is thread 0 */
    for (int t = 1; t < started; ++t)
        pthread_join(th[t], NULL);
    const int broken = bar.broken;
    free(off); free(len); free(snap); free(parts); free(th);
    if (!all) /* not every thread could be started: the one-thread ring, the same bits */
        return withhold_rank >= 0 ? OR_ENOMEM : oracle_ring_allreduce(buf, N, K, dtype, op, NULL);
    return broken ? OR_ETIMEDOUT : OR_OK;
}

int oracle_ring_allreduce_threads(void **buf, int N, uint64_t K, int dtype, int op, int nthreads)
{
    return oracle_ring_allreduce_threads_ex(buf, N, K, dtype, op, nthreads, -1, 60000);
}

/* Second, independent formulation (closed form).  Chunk c starts at rank c at
 * step 0 and collects one contribution per hop, finishing at rank c-1 after N-1
 * hops, so each of its elements is the left fold
 *     R = x_{c-1} (+) ( ... (x_{c+2} (+) (x_{c+1} (+) x_c)) ... )
 * with a round to the buffer type after every (+); AVG divides once, while
 * AVG_PREMUL scales each x_r before it enters the fold; every rank receives R.
 * in[] and out[] may alias per rank. */
int oracle_ring_allreduce_closed(const void **in, void **out, int N, uint64_t K, int dtype, int op)
{
    if (bad_args(N, dtype, op))
        return OR_EINVAL;
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)N), *len = malloc(sizeof(uint64_t) * (size_t)N);
    if (!off || !len) {
        free(off); free(len);
        return OR_ENOMEM;
    }
    oracle_partition(K, N, off, len);
    for (int c = 0; c < N; ++c)
        for (uint64_t e = off[c]; e < off[c] + len[c]; ++e) {
            uint32_t acc = contrib(load(in[c], dtype, e), N, dtype, op);
            for (int k = 1; k < N; ++k)
                acc = hop(contrib(load(in[(c + k) % N], dtype, e), N, dtype, op), acc, dtype, op);
            if (op == OR_AVG)
                acc = avg_scale(acc, N, dtype);
            for (int r = 0; r < N; ++r)
                store(out[r], dtype, e, acc);
        }
    free(off); free(len);
    return OR_OK;
}

/* Closed form evaluated only at the listed element indices (for spot checks of
 * buffers too large to reduce in full on the CPU).  out receives one element
 * per index, in the buffer type. */
int oracle_ring_allreduce_at(const void **in, int N, uint64_t K, int dtype, int op,
                             const uint64_t *idx, uint64_t n, void *out)
{
    if (bad_args(N, dtype, op))
        return OR_EINVAL;
    uint64_t q = K / (uint64_t)N, rem = K % (uint64_t)N;
    for (uint64_t t = 0; t < n; ++t) {
        uint64_t e = idx[t];
        if (e >= K)
            return OR_EINVAL;
        /* chunk of e under the front-loaded partition */
        int c;
        if (e < rem * (q + 1))
            c = (int)(e / (q + 1));
        else
            c = (int)(rem + (e - rem * (q + 1)) / q);
        uint32_t acc = contrib(load(in[c], dtype, e), N, dtype, op);
        for (int k = 1; k < N; ++k)
            acc = hop(contrib(load(in[(c + k) % N], dtype, e), N, dtype, op), acc, dtype, op);
        if (op == OR_AVG)
            acc = avg_scale(acc, N, dtype);
        store(out, dtype, t, acc);
    }
    return OR_OK;
}

/* Closed form at listed positions, from the contributions already gathered:
 * vals[r][t] is rank r's element at index idx[t] of a K-element buffer.  Lets
 * a caller check huge buffers whose inputs it can regenerate at the sampled
 * positions without materialising them. */
int oracle_ring_allreduce_gathered(const void **vals, int N, uint64_t K, int dtype, int op,
                                   const uint64_t *idx, uint64_t n, void *out)
{
    if (bad_args(N, dtype, op))
        return OR_EINVAL;
    uint64_t q = K / (uint64_t)N, rem = K % (uint64_t)N;
    for (uint64_t t = 0; t < n; ++t) {
        uint64_t e = idx[t];
        if (e >= K)
            return OR_EINVAL;
        int c;
        if (e < rem * (q + 1))
            c = (int)(e / (q + 1));
        else
            c = (int)(rem + (e - rem * (q + 1)) / q);
        uint32_t acc = contrib(load(vals[c], dtype, t), N, dtype, op);
        for (int k = 1; k < N; ++k)
            acc = hop(contrib(load(vals[(c + k) % N], dtype, t), N, dtype, op), acc, dtype, op);
        if (op == OR_AVG)
            acc = avg_scale(acc, N, dtype);
        store(out, dtype, t, acc);
    }
    return OR_OK;
}

/* ReduceScatter API: rank r receives the finished chunk r (len_r elements).
 * Runs the ring ReduceScatter phase step by step on copies of the inputs; the
 * phase leaves chunk r at rank r-1, and the API hands it to rank r
 * (Collectives and sharded matmul, "Scatter and ReduceScatter": rank r gets the
 * sum of block r). */
int oracle_reduce_scatter(const void **in, void **out, int N, uint64_t K, int dtype, int op)
{
    if (bad_args(N, dtype, op))
        return OR_EINVAL;
    size_t es = esize(dtype);
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)N), *len = malloc(sizeof(uint64_t) * (size_t)N);
    uint64_t stride = K / (uint64_t)N + 1;
    void *snap = malloc((size_t)N * stride * es);
    void **work = calloc((size_t)N, sizeof(void *));
    int rc = OR_OK;
    if (!off || !len || !snap || !work) {
        rc = OR_ENOMEM;
        goto done;
    }
    for (int r = 0; r < N; ++r) {
        work[r] = malloc(K * es + 1);
        if (!work[r]) {
            rc = OR_ENOMEM;
            goto done;
        }
        memcpy(work[r], in[r], K * es);
    }
    oracle_partition(K, N, off, len);
    rs_phase(work, N, off, len, dtype, op, NULL, snap, stride);
    for (int r = 0; r < N; ++r)
        memcpy(out[r], (char *)work[mod((int64_t)r - 1, N)] + off[r] * es, len[r] * es);
done:
    if (work)
        for (int r = 0; r < N; ++r)
            free(work[r]);
    free(work); free(off); free(len); free(snap);
    return rc;
}

/* Reduce to one rank: only out[root] receives the reduction; every other
 * out[r] is left untouched.  AllReduce is a Reduce followed by a Broadcast
 * (Lesson 3, core concepts: "Reduce (many-to-one)" and AllReduce), so the
 * root receives exactly the AllReduce's bits: the ring's ReduceScatter phase,
 * then each finished chunk c brought from rank c-1 to the root. */
int oracle_reduce(const void **in, void **out, int N, int root, uint64_t K, int dtype, int op)
{
    if (bad_args(N, dtype, op) || root < 0 || root >= N)
        return OR_EINVAL;
    size_t es = esize(dtype);
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)N), *len = malloc(sizeof(uint64_t) * (size_t)N);
    uint64_t stride = K / (uint64_t)N + 1;
    void *snap = malloc((size_t)N * stride * es);
    void **work = calloc((size_t)N, sizeof(void *));
    int rc = OR_OK;
    if (!off || !len || !snap || !work) {
        rc = OR_ENOMEM;
        goto done;
    }
    for (int r = 0; r < N; ++r) {
        work[r] = malloc(K * es + 1);
        if (!work[r]) {
            rc = OR_ENOMEM;
            goto done;
        }
        memcpy(work[r], in[r], K * es);
    }
    oracle_partition(K, N, off, len);
    rs_phase(work, N, off, len, dtype, op, NULL, snap, stride);
    for (int c = 0; c < N; ++c)
        memcpy((char *)out[root] + off[c] * es, (char *)work[mod((int64_t)c - 1, N)] + off[c] * es, len[c] * es);
done:
    if (work)
        for (int r = 0; r < N; ++r)
            free(work[r]);
    free(work); free(off); free(len); free(snap);
    return rc;
}

/* Gather: the root receives every rank's slice, concatenated in rank order
 * (Lesson 3, core concepts: "Gather (many-to-one)"); in[r] is chunk r
 * (len_r elements) of the K-element result. */
int oracle_gather(const void **in, void *out_root, int N, uint64_t K, int dtype)
{
    if (bad_args(N, dtype, OR_SUM))
        return OR_EINVAL;
    size_t es = esize(dtype);
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)N), *len = malloc(sizeof(uint64_t) * (size_t)N);
    if (!off || !len) {
        free(off); free(len);
        return OR_ENOMEM;
    }
    oracle_partition(K, N, off, len);
    for (int r = 0; r < N; ++r)
        memcpy((char *)out_root + off[r] * es, in[r], len[r] * es);
    free(off); free(len);
    return OR_OK;
}

/* Scatter: the root's K elements split into the N chunks, chunk r to rank r
 * (Lesson 3, core concepts: "Scatter (one-to-many)", the inverse of Gather). */
int oracle_scatter(const void *in_root, void **out, int N, uint64_t K, int dtype)
{
    if (bad_args(N, dtype, OR_SUM))
        return OR_EINVAL;
    size_t es = esize(dtype);
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)N), *len = malloc(sizeof(uint64_t) * (size_t)N);
    if (!off || !len) {
        free(off); free(len);
        return OR_ENOMEM;
    }
    oracle_partition(K, N, off, len);
    for (int r = 0; r < N; ++r)
        memcpy(out[r], (const char *)in_root + off[r] * es, len[r] * es);
    free(off); free(len);
    return OR_OK;
}

/* AllGather API: rank r contributes chunk r (len_r elements, in[r]); every
 * rank ends with the concatenation of all chunks in rank order.  Ring steps:
 * rank i starts holding chunk i; at step s it forwards chunk (i-s) mod N and
 * stores the chunk (i-1-s) mod N arriving from its left neighbour
 * (Collectives and sharded matmul, "ring AllGather"). */
int oracle_allgather(const void **in, void **out, int N, uint64_t K, int dtype)
{
    if (bad_args(N, dtype, OR_SUM))
        return OR_EINVAL;
    size_t es = esize(dtype);
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)N), *len = malloc(sizeof(uint64_t) * (size_t)N);
    uint64_t stride = K / (uint64_t)N + 1;
    void *snap = malloc((size_t)N * stride * es);
    if (!off || !len || !snap) {
        free(off); free(len); free(snap);
        return OR_ENOMEM;
    }
    oracle_partition(K, N, off, len);
    for (int r = 0; r < N; ++r)
        memcpy((char *)out[r] + off[r] * es, in[r], len[r] * es);
    for (int s = 0; s < N - 1; ++s) {
        for (int i = 0; i < N; ++i) {
            int c = mod((int64_t)i - s, N);
            memcpy((char *)snap + (size_t)i * stride * es, (char *)out[i] + off[c] * es, len[c] * es);
        }
        for (int i = 0; i < N; ++i) {
            int c = mod((int64_t)i - 1 - s, N);
            int src = mod((int64_t)i - 1, N);
            memcpy((char *)out[i] + off[c] * es, (char *)snap + (size_t)src * stride * es, len[c] * es);
        }
    }
    free(off); free(len); free(snap);
    return OR_OK;
}

/* Broadcast: every rank ends with root's K elements.  Chain order root ->
 * root+1 -> ... around the ring, one hop per step (copies, so the order cannot
 * change any bit).  in[r] for r != root is not read. */
int oracle_broadcast(const void **in, void **out, int N, int root, uint64_t K, int dtype)
{
    if (bad_args(N, dtype, OR_SUM) || root < 0 || root >= N)
        return OR_EINVAL;
    size_t es = esize(dtype);
    if (out[root] != in[root])
        memmove(out[root], in[root], K * es);
    for (int s = 0; s < N - 1; ++s) {
        int from = (root + s) % N, to = (root + s + 1) % N;
        memmove(out[to], out[from], K * es);
    }
    return OR_OK;
}

/* AllToAllv: counts[i*N+j] elements go from rank i to rank j.  Rank i's send
 * buffer holds its blocks ordered by destination, rank j's receive buffer holds
 * its blocks ordered by source (displacements are prefix sums).  Pairwise steps:
 * at step k rank i sends to (i+k) mod N, so block (i,j) lands in recv_j at the
 * position of source i ("rank = row, block = column: a transpose").
 * (Distributed LLM collectives, "Pairwise algorithm"; Collectives and sharded
 * matmul, "AllToAll".) */
int oracle_alltoallv(const void **in, void **out, int N, const uint64_t *counts, int dtype)
{
    if (bad_args(N, dtype, OR_SUM))
        return OR_EINVAL;
    size_t es = esize(dtype);
    uint64_t *sd = malloc(sizeof(uint64_t) * (size_t)N * N), *rd = malloc(sizeof(uint64_t) * (size_t)N * N);
    if (!sd || !rd) {
        free(sd); free(rd);
        return OR_ENOMEM;
    }
    for (int i = 0; i < N; ++i) {
        uint64_t o = 0;
        for (int j = 0; j < N; ++j) {
            sd[(size_t)i * N + j] = o;
            o += counts[(size_t)i * N + j];
        }
    }
    for (int j = 0; j < N; ++j) {
        uint64_t o = 0;
        for (int i = 0; i < N; ++i) {
            rd[(size_t)j * N + i] = o;
            o += counts[(size_t)i * N + j];
        }
    }
    for (int k = 0; k < N; ++k)
        for (int i = 0; i < N; ++i) {
            int j = (i + k) % N;
            memcpy((char *)out[j] + rd[(size_t)j * N + i] * es,
                   (const char *)in[i] + sd[(size_t)i * N + j] * es,
                   counts[(size_t)i * N + j] * es);
        }
    free(sd); free(rd);
    return OR_OK;
}

/* Bucket-fused AllReduce.  Each rank registers T gradient tensors in forward
 * order (tensors[r*T + t], numels[t] elements).  The tensors are laid end to end
 * in REVERSE registration order, the stream is cut into buckets of bucket_elems
 * elements (the last one partial; a tensor may span buckets), and each bucket is
 * AllReduced on its own with the ring above, its own N-chunk partition included.
 * (Collective Communication, "Bucket fusion": DDP fills buckets in reverse order
 * of use in the forward pass.)  In place on the tensors. */
int oracle_bucket_allreduce(void **tensors, const uint64_t *numels, int T, int N,
                            uint64_t bucket_elems, int dtype, int op)
{
    if (bad_args(N, dtype, op) || T < 0 || bucket_elems == 0)
        return OR_EINVAL;
    size_t es = esize(dtype);
    uint64_t total = 0;
    for (int t = 0; t < T; ++t)
        total += numels[t];
    void **bk = calloc((size_t)N, sizeof(void *));
    int rc = OR_OK;
    if (!bk)
        return OR_ENOMEM;
    for (int r = 0; r < N; ++r) {
        bk[r] = malloc(bucket_elems * es + 1);
        if (!bk[r]) {
            rc = OR_ENOMEM;
            goto done;
        }
    }
    for (uint64_t b0 = 0; b0 < total; b0 += bucket_elems) {
        uint64_t blen = total - b0 < bucket_elems ? total - b0 : bucket_elems;
        /* gather (pack) stream range [b0, b0+blen) of every rank */
        for (int dir = 0; dir < 2; ++dir) {
            uint64_t pos = 0; /* stream position of the current tensor's first element */
            for (int t = T - 1; t >= 0; --t) {
                uint64_t lo = pos > b0 ? pos : b0;
                uint64_t hi = pos + numels[t] < b0 + blen ? pos + numels[t] : b0 + blen;
                if (lo < hi)
                    for (int r = 0; r < N; ++r) {
                        char *tp = (char *)tensors[(size_t)r * T + t] + (lo - pos) * es;
                        char *bp = (char *)bk[r] + (lo - b0) * es;
                        if (dir == 0)
                            memcpy(bp, tp, (hi - lo) * es);
                        else
                            memcpy(tp, bp, (hi - lo) * es);
                    }
                pos += numels[t];
            }
            if (dir == 0) {
                rc = oracle_ring_allreduce(bk, N, blen, dtype, op, NULL);
                if (rc != OR_OK)
                    goto done;
            }
        }
    }
done:
    for (int r = 0; r < N; ++r)
        free(bk[r]);
    free(bk);
    return rc;
}

/* ------------------------------------------------------------------ */
/* other schedules: the same reduction, other summation orders          */
/* ------------------------------------------------------------------ */

static void scale_range(void *buf, uint64_t lo, uint64_t hi, int N, int dtype)
{
    for (uint64_t e = lo; e < hi; ++e)
        store(buf, dtype, e, avg_scale(load(buf, dtype, e), N, dtype));
}

/* Recursive halving-doubling AllReduce, step by step, in place
 * (Collective Communication, "Recursive halving-doubling (butterfly)": in
 * round k rank i pairs with i XOR 2^k, each keeps half of its current range
 * and adds the partner's copy of that half; the AllGather phase reverses the
 * rounds.  Distributed LLM collectives, "Recursive Halving-Doubling": for p not
 * a power of two, r = p - 2^floor(log2 p) and the first 2r ranks are reduced
 * pairwise into r ranks first, and get the result back at the end.)
 * Readings fixed here: the pre-fold pairs ranks (2v, 2v+1) and rank 2v+1
 * keeps the sum; virtual rank v is real rank 2v+1 for v < r, v+r otherwise;
 * the rank whose bit k is 0 keeps the lower half [lo, lo + ceil((hi-lo)/2)). */
int oracle_allreduce_hd(void **buf, int N, uint64_t K, int dtype, int op)
{
    if (bad_args(N, dtype, op) || op == OR_AVGP)
        return OR_EINVAL;
    int sop = op == OR_AVG ? OR_SUM : op;
    int pw = 1;
    while (pw * 2 <= N)
        pw *= 2;
    int r = N - pw, m = 0;
    while ((1 << m) < pw)
        ++m;
    uint64_t *lo = malloc(sizeof(uint64_t) * (size_t)pw), *hi = malloc(sizeof(uint64_t) * (size_t)pw);
    void **vb = malloc(sizeof(void *) * (size_t)pw);
    if (!lo || !hi || !vb) {
        free(lo); free(hi); free(vb);
        return OR_ENOMEM;
    }
    /* pre-fold: rank 2v+1 adds rank 2v's buffer */
    for (int v = 0; v < r; ++v)
        for (uint64_t e = 0; e < K; ++e)
            store(buf[2 * v + 1], dtype, e, hop(load(buf[2 * v + 1], dtype, e), load(buf[2 * v], dtype, e), dtype, sop));
    for (int v = 0; v < pw; ++v) {
        vb[v] = buf[v < r ? 2 * v + 1 : v + r];
        lo[v] = 0;
        hi[v] = K;
    }
    /* halving: round k pairs v with v ^ 2^k; both halves are disjoint, so
     * each rank reads its partner's kept-by-me half before anyone writes it */
    for (int k = 0; k < m; ++k) {
        for (int v = 0; v < pw; ++v) {
            uint64_t mid = lo[v] + (hi[v] - lo[v] + 1) / 2;
            int upper = (v >> k) & 1;
            uint64_t a = upper ? mid : lo[v], b = upper ? hi[v] : mid;
            void *partner = vb[v ^ (1 << k)];
            for (uint64_t e = a; e < b; ++e)
                store(vb[v], dtype, e, hop(load(vb[v], dtype, e), load(partner, dtype, e), dtype, sop));
            lo[v] = a;
            hi[v] = b;
        }
    }
    if (op == OR_AVG)
        for (int v = 0; v < pw; ++v)
            scale_range(vb[v], lo[v], hi[v], N, dtype);
    /* doubling: reverse rounds, each copies its partner's block */
    size_t es = esize(dtype);
    uint64_t *nlo = malloc(sizeof(uint64_t) * (size_t)pw * 2), *nhi;
    if (!nlo) {
        free(lo); free(hi); free(vb);
        return OR_ENOMEM;
    }
    nhi = nlo + pw;
    for (int k = m - 1; k >= 0; --k) {
        for (int v = 0; v < pw; ++v) {
            int w = v ^ (1 << k);
            memcpy((char *)vb[v] + lo[w] * es, (char *)vb[w] + lo[w] * es, (hi[w] - lo[w]) * es);
            nlo[v] = lo[v] < lo[w] ? lo[v] : lo[w];
            nhi[v] = hi[v] > hi[w] ? hi[v] : hi[w];
        }
        for (int v = 0; v < pw; ++v) {
            lo[v] = nlo[v];
            hi[v] = nhi[v];
        }
    }
    /* post: rank 2v gets the result back from rank 2v+1 */
    for (int v = 0; v < r; ++v)
        memcpy(buf[2 * v], buf[2 * v + 1], K * es);
    free(lo); free(hi); free(vb); free(nlo);
    return OR_OK;
}

/* Binomial-tree AllReduce, step by step, in place (Collective Communication,
 * "Tree AllReduce": leaves send to their parent, which adds what it receives
 * and passes it up, log2 N steps to the root, then the root's result is
 * broadcast back down).  Reading: at level k, rank i (a multiple of 2^(k+1))
 * receives from rank i + 2^k when that rank exists; the root is rank 0. */
int oracle_allreduce_tree(void **buf, int N, uint64_t K, int dtype, int op)
{
    if (bad_args(N, dtype, op) || op == OR_AVGP)
        return OR_EINVAL;
    int sop = op == OR_AVG ? OR_SUM : op;
    size_t es = esize(dtype);
    int top = 0;
    while ((1 << top) < N)
        ++top;
    for (int k = 0; k < top; ++k)
        for (int i = 0; i + (1 << k) < N; i += 1 << (k + 1))
            for (uint64_t e = 0; e < K; ++e)
                store(buf[i], dtype, e, hop(load(buf[i], dtype, e), load(buf[i + (1 << k)], dtype, e), dtype, sop));
    if (op == OR_AVG)
        scale_range(buf[0], 0, K, N, dtype);
    for (int k = top - 1; k >= 0; --k)
        for (int i = 0; i + (1 << k) < N; i += 1 << (k + 1))
            memcpy(buf[i + (1 << k)], buf[i], K * es);
    return OR_OK;
}

/* Two-level hierarchical AllReduce, step by step, in place (AllReduce survey,
 * "multi-dimensional hierarchical AllReduce", two-level table: ReduceScatter
 * inside each group of L ranks, AllReduce among the G = N/L group
 * representatives on the M/L shard, AllGather inside each group).  Groups are
 * consecutive ranks [gL, gL+L); every level is the ring of this file.  The
 * representative of intra chunk c in group g is the rank that finished it,
 * local rank (c-1) mod L; the inter ring partitions chunk c into G
 * sub-chunks.  AVG divides once by N, at the inter ring's holders. */
int oracle_allreduce_hier(void **buf, int N, int L, uint64_t K, int dtype, int op)
{
    if (bad_args(N, dtype, op) || op == OR_AVGP || L < 1 || N % L != 0)
        return OR_EINVAL;
    int G = N / L;
    int sop = op == OR_AVG ? OR_SUM : op;
    size_t es = esize(dtype);
    uint64_t *off = malloc(sizeof(uint64_t) * (size_t)(L > G ? L : G) * 2);
    uint64_t *len = off + (L > G ? L : G);
    uint64_t *soff = malloc(sizeof(uint64_t) * (size_t)G * 2), *slen;
    uint64_t stride = K + 1;
    void *snap = malloc((size_t)(L > G ? L : G) * stride * es);
    void **grp = malloc(sizeof(void *) * (size_t)(L > G ? L : G));
    if (!off || !soff || !snap || !grp) {
        free(off); free(soff); free(snap); free(grp);
        return OR_ENOMEM;
    }
    slen = soff + G;
    oracle_partition(K, L, off, len);
    /* 1. ReduceScatter inside every group */
    for (int g = 0; g < G; ++g) {
        for (int j = 0; j < L; ++j)
            grp[j] = buf[g * L + j];
        rs_phase(grp, L, off, len, dtype, sop, NULL, snap, stride);
    }
    /* 2. ring AllReduce of each chunk among the groups' representatives */
    uint64_t coff[1024], clen[1024];
    if (L > 1024) {
        free(off); free(soff); free(snap); free(grp);
        return OR_EINVAL;
    }
    for (int c = 0; c < L; ++c) {
        coff[c] = off[c];
        clen[c] = len[c];
    }
    for (int c = 0; c < L; ++c) {
        int rep = mod((int64_t)c - 1, L);
        for (int g = 0; g < G; ++g)
            grp[g] = (char *)buf[g * L + rep] + coff[c] * es;
        oracle_partition(clen[c], G, soff, slen);
        rs_phase(grp, G, soff, slen, dtype, sop, NULL, snap, stride);
        if (op == OR_AVG)
            for (int g = 0; g < G; ++g) {
                int d = mod((int64_t)g + 1, G);
                scale_range(grp[g], soff[d], soff[d] + slen[d], N, dtype);
            }
        ag_phase_after_rs(grp, G, soff, slen, dtype, NULL, snap, stride);
    }
    /* 3. AllGather inside every group */
    for (int g = 0; g < G; ++g) {
        for (int j = 0; j < L; ++j)
            grp[j] = buf[g * L + j];
        ag_phase_after_rs(grp, L, off, len, dtype, NULL, snap, stride);
    }
    free(off); free(soff); free(snap); free(grp);
    return OR_OK;
}

/* Closed forms of the three orders for one element (the second formulation):
 * x[r] is rank r's element (stored bits), e its index, K the buffer length.
 *   algo 1 halving-doubling: a balanced binary tree over the virtual leaves
 *          (x_{2v} (+) x_{2v+1} for v < r, then x_{v+r}), adjacent leaves first;
 *   algo 2 binomial tree: leaves in rank order, a subtree of 2^k ranks rooted
 *          at i combines with the one rooted at i + 2^k, the root's own
 *          subtrees folding from the smallest up;
 *   algo 3 hierarchical (group size L): a ring fold over groups, starting at
 *          group d, of ring folds inside each group starting at local rank c,
 *          where c is e's intra chunk and d its sub-chunk within chunk c. */
static uint32_t tree_fold(const uint32_t *x, int lo, int n, int dtype, int op)
{
    /* subtree of n ranks starting at lo in a binomial tree: the node lo
     * absorbs subtrees of size 1, 2, 4, ... rooted at lo+1, lo+2, lo+4 ... */
    uint32_t acc = x[lo];
    for (int s = 1; s < n; s *= 2) {
        int cnt = (n - s) < s ? (n - s) : s;
        acc = hop(acc, tree_fold(x, lo + s, cnt, dtype, op), dtype, op);
    }
    return acc;
}

static uint32_t balanced(const uint32_t *leaf, int lo, int n, int dtype, int op)
{
    if (n == 1)
        return leaf[lo];
    int h = n / 2;
    return hop(balanced(leaf, lo, h, dtype, op), balanced(leaf, lo + h, n - h, dtype, op), dtype, op);
}

int oracle_allreduce_order_at(const void **in, int N, uint64_t K, int dtype, int op, int algo, int L,
                              const uint64_t *idx, uint64_t n, void *out)
{
    if (bad_args(N, dtype, op) || op == OR_AVGP || algo < 1 || algo > 3 || N > 1024 || (algo == 3 && (L < 1 || N % L)))
        return OR_EINVAL;
    int sop = op == OR_AVG ? OR_SUM : op;
    uint32_t x[1024], leaf[1024];
    for (uint64_t t = 0; t < n; ++t) {
        uint64_t e = idx[t];
        if (e >= K)
            return OR_EINVAL;
        for (int r = 0; r < N; ++r)
            x[r] = load(in[r], dtype, e);
        uint32_t acc;
        if (algo == 1) {
            int pw = 1;
            while (pw * 2 <= N)
                pw *= 2;
            int r = N - pw;
            for (int v = 0; v < pw; ++v)
                leaf[v] = v < r ? hop(x[2 * v + 1], x[2 * v], dtype, sop) : x[v + r];
            acc = balanced(leaf, 0, pw, dtype, sop);
        } else if (algo == 2) {
            acc = tree_fold(x, 0, N, dtype, sop);
        } else {
            int G = N / L;
            uint64_t q = K / (uint64_t)L, rem = K % (uint64_t)L;
            int c = e < rem * (q + 1) ? (int)(e / (q + 1)) : (int)(rem + (e - rem * (q + 1)) / q);
            uint64_t oc = (uint64_t)c * q + ((uint64_t)c < rem ? (uint64_t)c : rem);
            uint64_t lc = q + ((uint64_t)c < rem ? 1 : 0);
            uint64_t ec = e - oc, q2 = lc / (uint64_t)G, rem2 = lc % (uint64_t)G;
            int d = ec < rem2 * (q2 + 1) ? (int)(ec / (q2 + 1)) : (int)(rem2 + (ec - rem2 * (q2 + 1)) / q2);
            acc = 0;
            for (int k = 0; k < G; ++k) {
                int g = (d + k) % G;
                uint32_t p = x[g * L + c];
                for (int j = 1; j < L; ++j)
                    p = hop(x[g * L + (c + j) % L], p, dtype, sop);
                acc = k == 0 ? p : hop(p, acc, dtype, sop);
            }
        }
        if (op == OR_AVG)
            acc = avg_scale(acc, N, dtype);
        store(out, dtype, t, acc);
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* compressed AllReduce with error feedback                            */
/* ------------------------------------------------------------------ */

#define OR_COMP_INT8_BLOCK 0
#define OR_COMP_THRESHOLD 1
#define OR_COMP_TOPK 2

static uint32_t canon(uint32_t r) { return f32_bits_is_nan(r) ? 0x7fffffffu : r; }
static float fcanon(float x) { return bits_to_f32(canon(f32_to_bits(x))); }

/* Round an fp32 value to the nearest integer, ties to even (the IEEE
 * roundToIntegralTiesToEven operation), written from its definition. */
static float round_half_even(float x)
{
    if (x != x || x - x != 0.0f) /* NaN or infinity */
        return fcanon(x);
    double d = (double)x, f = (double)(int64_t)d; /* |x| < 2^63 here: q is at most ~127 */
    if (d < 0 && f != d)
        f -= 1.0; /* floor */
    double frac = d - f;
    double r = frac > 0.5 ? f + 1.0 : frac < 0.5 ? f : (((int64_t)f & 1) ? f + 1.0 : f);
    if (r == 0.0)
        return d < 0 ? -0.0f : 0.0f;
    return (float)r;
}

/* Compress one rank's error-corrected gradient u = g + e (fp32), in place:
 * u is replaced by the transmitted value v and e by the new residual
 * e' = u - v (Collective Communication, "Error feedback and residual
 * accumulation", Definition 1.4: e_{t+1} = g_t + e_t - v_t).
 *   INT8 block ("Blockwise quantization for gradient communication"): per block
 *     of `block` consecutive elements, s = max|u| / 127, q = round(u / s) (ties
 *     to even; q = 0 when s = 0), v = q * s; a NaN anywhere in the block makes
 *     s NaN.
 *   THRESHOLD (the greedy 1-bit compressor of Tables 3 and 4): v = 1 when
 *     u >= threshold, else 0.
 *   TOPK ("Top-k sparsification"): v = u where |u| >= |u|_(k), the k-th
 *     largest magnitude, else 0 -- every element tied with the k-th is kept.
 *     Magnitudes are ordered as the bit patterns of |u|, so a NaN counts as
 *     larger than any number and is always kept (it reaches the result, as a
 *     NaN in an INT8 block does).  k = 0 keeps nothing; k >= K keeps all. */
static int cmp_desc_u32(const void *a, const void *b)
{
    const uint32_t x = *(const uint32_t *)a, y = *(const uint32_t *)b;
    return x < y ? 1 : (x > y ? -1 : 0);
}

static int compress_topk(float *u, float *e, uint64_t K, uint64_t k)
{
    uint32_t tau = 0xffffffffu; /* k = 0: no magnitude reaches it */
    if (k > 0 && K > 0) {
        uint32_t *mag = malloc(K * sizeof(uint32_t));
        if (!mag)
            return OR_ENOMEM;
        for (uint64_t i = 0; i < K; ++i)
            mag[i] = f32_to_bits(u[i]) & 0x7fffffffu;
        qsort(mag, K, sizeof(uint32_t), cmp_desc_u32); /* largest first */
        tau = mag[(k < K ? k : K) - 1];
        free(mag);
    }
    for (uint64_t i = 0; i < K; ++i) {
        float v = (f32_to_bits(u[i]) & 0x7fffffffu) >= tau ? u[i] : 0.0f;
        e[i] = fcanon(u[i] - v);
        u[i] = v;
    }
    return OR_OK;
}

static void compress(float *u, float *e, uint64_t K, int comp, int block, float threshold)
{
    if (comp == OR_COMP_THRESHOLD) {
        for (uint64_t i = 0; i < K; ++i) {
            float v = u[i] >= threshold ? 1.0f : 0.0f;
            e[i] = fcanon(u[i] - v);
            u[i] = v;
        }
        return;
    }
    for (uint64_t b0 = 0; b0 < K; b0 += (uint64_t)block) {
        uint64_t b1 = b0 + (uint64_t)block < K ? b0 + (uint64_t)block : K;
        float amax = 0.0f;
        int nan = 0;
        for (uint64_t i = b0; i < b1; ++i) {
            float a = u[i] < 0 ? -u[i] : u[i];
            if (u[i] != u[i])
                nan = 1;
            else if (a > amax)
                amax = a;
        }
        float sc = nan ? bits_to_f32(0x7fffffffu) : fcanon(amax / 127.0f);
        for (uint64_t i = b0; i < b1; ++i) {
            float q = sc > 0.0f ? round_half_even(fcanon(u[i] / sc)) : (sc == 0.0f ? 0.0f : sc);
            float v = fcanon(q * sc);
            e[i] = fcanon(u[i] - v);
            u[i] = v;
        }
    }
}

/* Compressed AllReduce, in place: grads[r] (K elements of dtype) and the
 * residuals res[r] (K fp32, start at zero).  Every rank compresses u = g + e,
 * keeps its residual, and the transmitted values are AllReduced with the ring
 * of this file in fp32 (SUM, or AVG dividing once by N); the result is rounded
 * once to the buffer type and written to every rank's grads. */
int oracle_allreduce_compressed_k(void **grads, float **res, int N, uint64_t K, int dtype, int op, int comp,
                                  int block, float threshold, uint64_t topk)
{
    if (bad_args(N, dtype, op) || (op != OR_SUM && op != OR_AVG) || (comp != OR_COMP_INT8_BLOCK &&
        comp != OR_COMP_THRESHOLD && comp != OR_COMP_TOPK) || (comp == OR_COMP_INT8_BLOCK && block < 1))
        return OR_EINVAL;
    void **v = calloc((size_t)N, sizeof(void *));
    int rc = OR_OK;
    if (!v)
        return OR_ENOMEM;
    for (int r = 0; r < N; ++r) {
        float *u = malloc(K * sizeof(float) + 4);
        if (!u) {
            rc = OR_ENOMEM;
            goto done;
        }
        for (uint64_t i = 0; i < K; ++i)
            u[i] = fcanon(bits_to_f32(widen_bits(load(grads[r], dtype, i), dtype)) + res[r][i]);
        v[r] = u;
        if (comp == OR_COMP_TOPK) {
            if ((rc = compress_topk(u, res[r], K, topk)) != OR_OK)
                goto done;
        } else {
            compress(u, res[r], K, comp, block, threshold);
        }
    }
    rc = oracle_ring_allreduce(v, N, K, OR_FP32, op, NULL);
    if (rc != OR_OK)
        goto done;
    for (int r = 0; r < N; ++r)
        for (uint64_t i = 0; i < K; ++i)
            store(grads[r], dtype, i, narrow_bits(((uint32_t *)v[r])[i], dtype));
done:
    for (int r = 0; r < N; ++r)
        free(v[r]);
    free(v);
    return rc;
}

/* The INT8 block and threshold compressors (no k). */
int oracle_allreduce_compressed(void **grads, float **res, int N, uint64_t K, int dtype, int op, int comp,
                                int block, float threshold)
{
    if (comp == OR_COMP_TOPK)
        return OR_EINVAL;
    return oracle_allreduce_compressed_k(grads, res, N, K, dtype, op, comp, block, threshold, 0);
}

/* Plain fp64 reference of the reduction (the definition y = sum_r x_r with no
 * ring and no intermediate rounding), plus sum_r |x_r|, the scale against which
 * relative error is measured.  SUM/AVG only. */
int oracle_sum_f64(const void **in, int N, uint64_t K, int dtype, int op, double *y, double *absum)
{
    if (bad_args(N, dtype, op) || (op != OR_SUM && op != OR_AVG && op != OR_AVGP))
        return OR_EINVAL;
    if (op == OR_AVGP)
        op = OR_AVG; /* the same mean */
    for (uint64_t e = 0; e < K; ++e) {
        double s = 0.0, a = 0.0;
        for (int r = 0; r < N; ++r) {
            double x = (double)bits_to_f32(widen_bits(load(in[r], dtype, e), dtype));
            s += x;
            a += x < 0 ? -x : x;
        }
        y[e] = op == OR_AVG ? s / (double)N : s;
        absum[e] = op == OR_AVG ? a / (double)N : a;
    }
    return OR_OK;
}
