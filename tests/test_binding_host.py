"""The Python binding's own checks, made before anything reaches the C ABI
(no GPU): only contiguous float32/bfloat16 tensors become rank pointers, the
host-buffer AllReduce needs a device work tensor, and library errors surface as
CclError with the status name."""
import pytest
import torch

import ring_allreduce_rank_gb300 as ccl
from ring_allreduce_rank_gb300 import ccl as C


@pytest.fixture(scope="module", autouse=True)
def _built():
    from ring_allreduce_rank_gb300 import build
    build.build()
    ccl.lib()


def test_only_float32_and_bfloat16():
    bufs = [torch.zeros(16, dtype=torch.float16) for _ in range(2)]
    with pytest.raises(TypeError, match="float32 and bfloat16"):
        ccl.ccl_allreduce(bufs)


def test_rank_buffers_must_be_contiguous():
    strided = [torch.zeros(8, 4)[:, 0] for _ in range(2)]
    assert not strided[0].is_contiguous()
    with pytest.raises(ValueError, match="contiguous"):
        ccl.ccl_allreduce(strided)


def test_unknown_op_and_mode_names():
    bufs = [torch.zeros(16) for _ in range(2)]
    with pytest.raises(KeyError):
        ccl.ccl_allreduce(bufs, op="mean")
    with pytest.raises(KeyError):
        ccl.ccl_set_mode_override("pipelined")


def test_host_allreduce_needs_a_device_work_tensor():
    host = [torch.zeros(1024) for _ in range(2)]
    with pytest.raises(ValueError, match="work"):
        ccl.ccl_allreduce_host(host)
    with pytest.raises(ValueError, match="work"):
        ccl.ccl_allreduce_host(host, work=torch.zeros(1 << 16, dtype=torch.uint8))


def test_check_counter_must_be_one_int64_device_element():
    bufs = [torch.zeros(16) for _ in range(2)]
    with pytest.raises(TypeError, match="int64"):
        ccl.ccl_check_identical(bufs, torch.zeros(1, dtype=torch.float32))


def test_library_errors_surface_with_their_status():
    with pytest.raises(C.CclError) as e:
        ccl.ccl_plan_chunks(10, 0)
    assert e.value.status == 1 and "CCL_ERR_INVALID_ARG" in str(e.value) and "ccl_plan_chunks" in str(e.value)
    with pytest.raises(C.CclError) as e:
        ccl.ccl_arena_layout(3, 1000, 100)  # alignment not a power of two
    assert e.value.status == 1
