"""Single-GPU ring collectives for GB300 (sm_103a).

N ranks are simulated on one GPU, each a buffer in one HBM arena; the
collectives compute the ring algorithm's exact data semantics in hand-written
CUDA kernels behind a C ABI (include/ccl.h, libccl.so).  This package is the
thin Python binding of that library plus the arena helper and the seeded
synthetic workloads.
"""
from .ccl import (CclBucketer, CclError, ccl_allgather, ccl_allreduce, ccl_allreduce_algo, ccl_allreduce_compressed, ccl_allreduce_host, ccl_allreduce_topk, ccl_alltoall, ccl_alltoallv, ccl_arena_layout,
                  ccl_broadcast, ccl_bucket_allreduce, ccl_check_identical, ccl_check_read, ccl_debug_faults, ccl_finalize, ccl_gather, ccl_get_config, ccl_launch_count, ccl_plan_alltoallv, ccl_plan_compressed_bytes,
                  ccl_plan_topk_bytes, ccl_plan_topk_sample, ccl_plan_topk_work_bytes, ccl_plan_buckets, ccl_plan_chunks, ccl_plan_host_slices, ccl_plan_ring_schedule, ccl_reduce, ccl_reduce_scatter,
                  ccl_scatter, ccl_set_check, ccl_set_default_bucket_bytes, ccl_set_host_path, ccl_set_mode_override, ccl_set_trace, ccl_status_string, ccl_step_sent, ccl_trace_clear, ccl_trace_read, lib)

__all__ = ["CclBucketer", "CclError", "ccl_allgather", "ccl_allreduce", "ccl_allreduce_algo", "ccl_allreduce_compressed", "ccl_allreduce_host", "ccl_allreduce_topk", "ccl_alltoall", "ccl_alltoallv", "ccl_arena_layout",
           "ccl_broadcast", "ccl_bucket_allreduce", "ccl_check_identical", "ccl_check_read", "ccl_debug_faults", "ccl_finalize", "ccl_gather", "ccl_get_config", "ccl_launch_count",
           "ccl_plan_alltoallv", "ccl_plan_compressed_bytes", "ccl_plan_topk_bytes", "ccl_plan_topk_sample", "ccl_plan_topk_work_bytes", "ccl_plan_buckets", "ccl_plan_chunks", "ccl_plan_host_slices", "ccl_plan_ring_schedule", "ccl_reduce",
           "ccl_reduce_scatter", "ccl_scatter", "ccl_set_check", "ccl_set_default_bucket_bytes", "ccl_set_host_path", "ccl_set_mode_override", "ccl_set_trace", "ccl_status_string", "ccl_step_sent", "ccl_trace_clear", "ccl_trace_read", "lib"]
