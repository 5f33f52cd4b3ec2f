"""The boundary is a C ABI: include/ccl.h compiles as strict C and C++, and a
plain C program (tests/c_abi_example.c) builds against it and libccl.so with
gcc alone -- no Python, no torch -- and, on a GPU, runs collectives through it
with exact integer results.  A second program (tests/c_abi_host_example.c)
uses the host-only entry points from C on a machine without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
EXAMPLE = os.path.join(ROOT, "tests", "c_abi_example.c")
HOST_EXAMPLE = os.path.join(ROOT, "tests", "c_abi_host_example.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _cuda_include():
    inc = os.path.join(CUDA, "include")
    if not os.path.exists(os.path.join(inc, "cuda_runtime_api.h")):
        pytest.skip("CUDA headers not found")
    return inc


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c", "c11"), ("c++", "c++17")])
def test_header_compiles_strictly(lang, std, tmp_path):
    src = tmp_path / ("h." + ("c" if lang == "c" else "cpp"))
    src.write_text('#include "ccl.h"\nint main(void) { return ccl_version() > 0 ? 0 : 1; }\n')
    cc = "gcc" if lang == "c" else "g++"
    # CUDA's own headers are system headers here: the strict flags apply to ccl.h alone
    subprocess.run([cc, "-std=" + std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only", "-I", INCLUDE,
                    "-isystem", _cuda_include(), str(src)], check=True)


def _build_example(out, src=EXAMPLE):
    from ring_allreduce_rank_gb300 import build
    lib = build.build()
    libdir = os.path.dirname(lib)
    cudalib = os.path.join(CUDA, "lib64")
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1", "-I", INCLUDE, "-isystem", _cuda_include(),
                    src, "-o", out, "-L", libdir, "-lccl", "-Wl,-rpath," + libdir, "-L", cudalib, "-lcudart",
                    "-Wl,-rpath," + cudalib], check=True)
    return out


def test_host_example_runs_without_a_gpu(tmp_path):
    """The planner, the settings (ccl_config_t read from C), the step-mode
    traffic counter and argument validation, from plain C with no device."""
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    exe = _build_example(str(tmp_path / "c_abi_host_example"), HOST_EXAMPLE)
    env = {k: v for k, v in os.environ.items() if not k.startswith("CCL_")}
    env["CUDA_VISIBLE_DEVICES"] = ""
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120, env=env)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "c abi host ok" in res.stdout


def test_example_builds_with_gcc_alone(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    assert os.path.exists(_build_example(str(tmp_path / "c_abi_example")))


@pytest.mark.gpu
def test_example_runs_on_the_gpu(tmp_path):
    exe = _build_example(str(tmp_path / "c_abi_example"))
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "c abi ok" in res.stdout
