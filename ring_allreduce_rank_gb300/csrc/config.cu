// config.cu -- library-wide settings read from the environment.
//
// Collective Communication (libraries section) describes how NCCL is steered
// without touching the program: environment variables pick the algorithm and
// protocol (NCCL_ALGO, NCCL_PROTO) or turn on logging (NCCL_DEBUG), and data
// parallelism's gradient buckets are sized by one knob (bucket_cap_mb, 25 MB
// by default; bucket fusion section).  This library has the same kind of
// knobs:
//   CCL_MODE=fused|step  forces that mode on every call that takes a mode, so
//                        a program can be re-run with the ring executed step
//                        by step, without changing its calls;
//   CCL_BUCKET_MB=<MiB>  the bucket size of bucket AllReduce calls that pass
//                        bucket_bytes = 0;
//   CCL_HOST_PATH=staged|direct  whether the host-buffer AllReduce stages
//                        slices through device memory (staged) or may work on
//                        page-locked host buffers in place (direct);
//   CCL_TRACE, CCL_CHECK (check.cu).
// Each is read once, on first use; the setters replace what was read.
#include <atomic>
#include <cerrno>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <strings.h>

#include "../../include/ccl.h"
#include "ccl_internal.h"

namespace ccl {

namespace {
constexpr int kModeUnread = -2;  // CCL_MODE not looked at yet
constexpr int kModeNone = -1;    // no override: each call's own argument
constexpr unsigned long long kBucketUnread = 0;
// Largest bucket accepted from the environment: 1 TiB (any bucket larger than
// the whole gradient stream behaves like one bucket anyway).
constexpr double kMaxBucketMiB = 1024.0 * 1024.0;

constexpr int kHostPathUnread = -1;
std::atomic<int> g_mode{kModeUnread};
std::atomic<int> g_host_path{kHostPathUnread};
std::atomic<unsigned long long> g_bucket{kBucketUnread};

int mode_from_env()
{
    const char *e = std::getenv("CCL_MODE");
    if (!e || !e[0])
        return kModeNone;
    if (strcasecmp(e, "fused") == 0)
        return CCL_MODE_FUSED;
    if (strcasecmp(e, "step") == 0)
        return CCL_MODE_STEP;
    std::fprintf(stderr, "ccl: ignoring CCL_MODE=%s (expected fused or step)\n", e);
    return kModeNone;
}

unsigned long long bucket_from_env()
{
    const char *e = std::getenv("CCL_BUCKET_MB");
    if (!e || !e[0])
        return CCL_DEFAULT_BUCKET_BYTES;
    errno = 0;
    char *end = nullptr;
    const double mib = std::strtod(e, &end);
    const bool ok = errno == 0 && end && *end == '\0' && std::isfinite(mib) && mib > 0.0 && mib <= kMaxBucketMiB;
    const double bytes = ok ? std::floor(mib * 1048576.0 + 0.5) : 0.0;
    if (!ok || bytes < 4.0) { // a bucket must hold at least one fp32 element
        std::fprintf(stderr, "ccl: ignoring CCL_BUCKET_MB=%s (expected a size in MiB, at least 4 bytes)\n", e);
        return CCL_DEFAULT_BUCKET_BYTES;
    }
    return (unsigned long long)bytes;
}

int host_path_from_env()
{
    const char *e = std::getenv("CCL_HOST_PATH");
    if (!e || !e[0] || strcasecmp(e, "staged") == 0)
        return CCL_HOST_PATH_STAGED;
    if (strcasecmp(e, "direct") == 0)
        return CCL_HOST_PATH_DIRECT;
    std::fprintf(stderr, "ccl: ignoring CCL_HOST_PATH=%s (expected staged or direct)\n", e);
    return CCL_HOST_PATH_STAGED;
}

int mode_override()
{
    int v = g_mode.load(std::memory_order_relaxed);
    if (v == kModeUnread) {
        int expected = kModeUnread;
        g_mode.compare_exchange_strong(expected, mode_from_env(), std::memory_order_relaxed);
        v = g_mode.load(std::memory_order_relaxed);
    }
    return v;
}
} // namespace

ccl_mode_t effective_mode(ccl_mode_t requested)
{
    // an invalid argument stays invalid: the call rejects it as before
    if (requested != CCL_MODE_FUSED && requested != CCL_MODE_STEP)
        return requested;
    const int v = mode_override();
    return v == kModeNone ? requested : (ccl_mode_t)v;
}

int host_path()
{
    int v = g_host_path.load(std::memory_order_relaxed);
    if (v == kHostPathUnread) {
        int expected = kHostPathUnread;
        g_host_path.compare_exchange_strong(expected, host_path_from_env(), std::memory_order_relaxed);
        v = g_host_path.load(std::memory_order_relaxed);
    }
    return v;
}

size_t default_bucket_bytes()
{
    unsigned long long v = g_bucket.load(std::memory_order_relaxed);
    if (v == kBucketUnread) {
        unsigned long long expected = kBucketUnread;
        g_bucket.compare_exchange_strong(expected, bucket_from_env(), std::memory_order_relaxed);
        v = g_bucket.load(std::memory_order_relaxed);
    }
    return (size_t)v;
}

} // namespace ccl

using namespace ccl;

extern "C" {

ccl_status_t ccl_get_config(ccl_config_t *out)
{
    if (!out)
        return CCL_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof *out);
    out->mode_override = mode_override();
    out->trace = trace_enabled() ? 1 : 0;
    out->check = check_enabled() ? 1 : 0;
    out->default_bucket_bytes = default_bucket_bytes();
    out->host_path = host_path();
    return CCL_OK;
}

ccl_status_t ccl_set_host_path(int path)
{
    if (path != CCL_HOST_PATH_STAGED && path != CCL_HOST_PATH_DIRECT)
        return CCL_ERR_INVALID_ARG;
    g_host_path.store(path, std::memory_order_relaxed);
    return CCL_OK;
}

ccl_status_t ccl_set_mode_override(int mode)
{
    if (mode != kModeNone && mode != CCL_MODE_FUSED && mode != CCL_MODE_STEP)
        return CCL_ERR_INVALID_ARG;
    g_mode.store(mode, std::memory_order_relaxed);
    return CCL_OK;
}

ccl_status_t ccl_set_default_bucket_bytes(size_t bytes)
{
    if (bytes != 0 && bytes < 4)
        return CCL_ERR_INVALID_ARG;
    g_bucket.store(bytes ? (unsigned long long)bytes : (unsigned long long)CCL_DEFAULT_BUCKET_BYTES,
                   std::memory_order_relaxed);
    return CCL_OK;
}

} // extern "C"
