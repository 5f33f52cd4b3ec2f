/*
 * The library used from plain C: include/ccl.h, libccl.so and the CUDA
 * runtime, nothing else.  N ranks of small integers are reduced exactly, so
 * every expected value is a plain integer sum computed here.
 *   1. AllReduce SUM (fused) on device buffers, in place.
 *   2. ReduceScatter then AllGather, out of place: the same bits as 1.
 *   3. The host-buffer AllReduce on page-locked host buffers, on both paths.
 *   4. Argument errors come back as status codes, before any launch.
 * Prints "c abi ok" and exits 0 when every check holds.
 */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ccl.h"

#define NR 5
#define K 10007

static int fail(const char *what)
{
    fprintf(stderr, "c abi: %s\n", what);
    return 1;
}

#define CUDA_OK(x) do { if ((x) != cudaSuccess) return fail(#x); } while (0)
#define CCL_OK_(x) do { ccl_status_t s_ = (x); if (s_ != CCL_OK) { fprintf(stderr, "%s\n", ccl_status_string(s_)); return fail(#x); } } while (0)

static float value(int r, int i) { return (float)((i * 7 + r * 13) % 31 - 15); }

int main(void)
{
    void *dev[NR], *rs[NR], *ag[NR];
    float *h = (float *)malloc(sizeof(float) * K), *want = (float *)malloc(sizeof(float) * K);
    size_t off[NR], len[NR];
    if (!h || !want)
        return fail("malloc");
    CCL_OK_(ccl_plan_chunks(K, NR, off, len));
    for (int i = 0; i < K; ++i) {
        float s = 0.0f;
        for (int r = 0; r < NR; ++r)
            s += value(r, i); /* integers: exact in any order */
        want[i] = s;
    }
    for (int r = 0; r < NR; ++r) {
        CUDA_OK(cudaMalloc(&dev[r], K * sizeof(float)));
        CUDA_OK(cudaMalloc(&rs[r], len[r] * sizeof(float)));
        CUDA_OK(cudaMalloc(&ag[r], K * sizeof(float)));
        for (int i = 0; i < K; ++i)
            h[i] = value(r, i);
        CUDA_OK(cudaMemcpy(dev[r], h, K * sizeof(float), cudaMemcpyHostToDevice));
    }

    /* 2 first (it reads the inputs), then 1 in place */
    CCL_OK_(ccl_reduce_scatter((const void *const *)dev, rs, NR, K, CCL_FP32, CCL_SUM, CCL_MODE_FUSED, 0));
    CCL_OK_(ccl_allgather((const void *const *)rs, ag, NR, K, CCL_FP32, CCL_MODE_FUSED, 0));
    CCL_OK_(ccl_allreduce((const void *const *)dev, dev, NR, K, CCL_FP32, CCL_SUM, CCL_MODE_FUSED, 0));
    CUDA_OK(cudaDeviceSynchronize());
    for (int r = 0; r < NR; ++r) {
        CUDA_OK(cudaMemcpy(h, dev[r], K * sizeof(float), cudaMemcpyDeviceToHost));
        if (memcmp(h, want, K * sizeof(float)) != 0)
            return fail("AllReduce result");
        CUDA_OK(cudaMemcpy(h, ag[r], K * sizeof(float), cudaMemcpyDeviceToHost));
        if (memcmp(h, want, K * sizeof(float)) != 0)
            return fail("ReduceScatter + AllGather result");
    }

    /* 3: page-locked host rank buffers, staged through a small work buffer
     * (the default path), then in place over the host link */
    void *hs[NR], *work = NULL;
    const size_t work_bytes = (size_t)3 * NR * 1024 * sizeof(float);
    CUDA_OK(cudaMalloc(&work, work_bytes));
    for (int r = 0; r < NR; ++r)
        CUDA_OK(cudaHostAlloc(&hs[r], K * sizeof(float), cudaHostAllocDefault));
    size_t nslices = 0;
    CCL_OK_(ccl_plan_host_slices(K, NR, CCL_FP32, work_bytes, NULL, NULL, 0, &nslices));
    if (nslices < 2)
        return fail("expected several slices");
    for (int path = CCL_HOST_PATH_STAGED; path <= CCL_HOST_PATH_DIRECT; ++path) {
        for (int r = 0; r < NR; ++r)
            for (int i = 0; i < K; ++i)
                ((float *)hs[r])[i] = value(r, i);
        CCL_OK_(ccl_set_host_path(path));
        CCL_OK_(ccl_allreduce_host((const void *const *)hs, hs, NR, K, CCL_FP32, CCL_SUM, work, work_bytes, 0));
        CUDA_OK(cudaDeviceSynchronize());
        for (int r = 0; r < NR; ++r)
            if (memcmp(hs[r], want, K * sizeof(float)) != 0)
                return fail(path == CCL_HOST_PATH_DIRECT ? "host-buffer AllReduce result (in place)"
                                                         : "host-buffer AllReduce result (staged)");
    }
    CCL_OK_(ccl_set_host_path(CCL_HOST_PATH_STAGED));

    /* 4: errors are status codes */
    if (ccl_allreduce((const void *const *)dev, dev, 0, K, CCL_FP32, CCL_SUM, CCL_MODE_FUSED, 0) != CCL_ERR_INVALID_ARG)
        return fail("nranks = 0 accepted");
    if (ccl_allreduce((const void *const *)dev, ag, NR, K, (ccl_dtype_t)9, CCL_SUM, CCL_MODE_FUSED, 0) !=
        CCL_ERR_INVALID_ARG)
        return fail("unknown dtype accepted");
    void *shifted[NR];
    for (int r = 0; r < NR; ++r)
        shifted[r] = (char *)dev[r] + 4; /* overlaps its own input by all but one element */
    if (ccl_allreduce((const void *const *)dev, shifted, NR, K - 1, CCL_FP32, CCL_SUM, CCL_MODE_FUSED, 0) !=
        CCL_ERR_OVERLAP)
        return fail("partial overlap accepted");
    if (ccl_launch_count() < 4)
        return fail("launch count");

    for (int r = 0; r < NR; ++r) {
        cudaFree(dev[r]);
        cudaFree(rs[r]);
        cudaFree(ag[r]);
        cudaFreeHost(hs[r]);
    }
    cudaFree(work);
    free(h);
    free(want);
    printf("c abi ok (library version %d)\n", ccl_version());
    return 0;
}
