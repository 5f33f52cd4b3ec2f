// fused.h -- what the one-pass ring-order reduction kernel (reduce.cu) is
// built from besides the device helpers: its parameter block, write modes and
// launcher.  Kept apart from the library's other internal declarations so that
// the kernel's source set is exactly reduce.cu, ccl_device.cuh and this file.
#pragma once

#include <cuda_runtime_api.h>
#include <stdint.h>

#include "ccl_device.cuh"

namespace ccl {

constexpr int kSmallRanks = 16;
constexpr int kMaxRanks = 1024;

// ------------------------------------------------------------------ fused reduce
template <int MAXR> struct FusedParams {
    const void *send[MAXR];
    void *recv[MAXR];
    Partition part;
    int nranks;
    int write_mode;  // WRITE_CHUNK, WRITE_ALL or WRITE_ROOT
    int root;        // WRITE_ROOT: the one rank that receives the result
    int vec_aligned; // every pointer is 16-byte aligned
    uint32_t tiles;  // tiles per chunk (gridDim.x)
    float n_f;       // (float)nranks, the AVG divisor
    float inv_n;     // 1/nranks correctly rounded, the pre-multiplied AVG's scale
};

enum WriteMode {
    WRITE_CHUNK = 0, // ReduceScatter: chunk c goes to recv[c], chunk-local
    WRITE_ALL = 1,   // AllReduce: every rank receives the whole result
    WRITE_ROOT = 2   // Reduce: only recv[root] receives the whole result
};

// Launch the one-pass ring-order reduction (AllReduce, ReduceScatter or Reduce).
cudaError_t launch_fused_reduce(int dt, int op, const void *const *send, void *const *recv, int nranks,
                                uint64_t count, int write_mode, int root, cudaStream_t stream);

void count_launches(unsigned long long n);

} // namespace ccl
