"""Library settings on the host (no GPU): CCL_MODE, CCL_BUCKET_MB,
CCL_HOST_PATH, CCL_TRACE and CCL_CHECK as read from the environment, the warnings for values that
cannot be read, and the setters that replace them.  Each case runs in a child
process, because the environment is read once per process; the children see no
GPU and make no collective call."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MiB = 1 << 20

CHILD = r"""
import json, sys
sys.path.insert(0, %r)
import ring_allreduce_rank_gb300 as ccl
out = {"env": ccl.ccl_get_config()}
for step in json.loads(sys.argv[1]):
    kind, arg = step
    try:
        if kind == "mode":
            ccl.ccl_set_mode_override(arg)
        elif kind == "host":
            ccl.ccl_set_host_path(arg)
        elif kind == "host_raw":  # the C setter itself, with any int
            rc = ccl.lib().ccl_set_host_path(arg)
            if rc:
                raise ccl.CclError(rc, "ccl_set_host_path")
        else:
            ccl.ccl_set_default_bucket_bytes(arg)
        out.setdefault("rc", []).append("ok")
    except ccl.CclError as e:
        out.setdefault("rc", []).append(e.status)
out["after"] = ccl.ccl_get_config()
print(json.dumps(out))
""" % ROOT


@pytest.fixture(scope="module")
def built():
    from ring_allreduce_rank_gb300 import build
    build.build()


def run_child(env_extra, steps=()):
    env = {k: v for k, v in os.environ.items() if not k.startswith("CCL_")}
    env.update(env_extra)
    env["CUDA_VISIBLE_DEVICES"] = ""
    p = subprocess.run([sys.executable, "-c", CHILD, json.dumps(list(steps))], env=env, capture_output=True,
                       text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    return json.loads(p.stdout.strip().splitlines()[-1]), p.stderr


def test_defaults_without_environment(built):
    out, err = run_child({})
    assert out["env"] == {"mode_override": None, "trace": False, "check": False, "default_bucket_bytes": 25 * MiB,
                          "host_path": "staged"}
    assert "ignoring" not in err


@pytest.mark.parametrize("value,want", [("step", "step"), ("STEP", "step"), ("fused", "fused"), ("Fused", "fused"),
                                        ("", None)])
def test_mode_from_environment(built, value, want):
    out, err = run_child({"CCL_MODE": value})
    assert out["env"]["mode_override"] == want
    assert "ignoring" not in err


@pytest.mark.parametrize("value", ["steps", "1", "auto", " step"])
def test_unreadable_mode_is_ignored_with_a_warning(built, value):
    out, err = run_child({"CCL_MODE": value})
    assert out["env"]["mode_override"] is None
    assert err.count("ignoring CCL_MODE") == 1


@pytest.mark.parametrize("value,want", [("25", 25 * MiB), ("1.5", 3 * MiB // 2), ("0.5", MiB // 2),
                                        ("100", 100 * MiB), ("4e-6", 4), ("1048576", 1 << 40)])
def test_bucket_size_from_environment(built, value, want):
    out, err = run_child({"CCL_BUCKET_MB": value})
    assert out["env"]["default_bucket_bytes"] == want
    assert "ignoring" not in err


@pytest.mark.parametrize("value", ["0", "-1", "abc", "25MB", "inf", "nan", "1e-7", "2e6"])
def test_unreadable_bucket_size_is_ignored_with_a_warning(built, value):
    out, err = run_child({"CCL_BUCKET_MB": value})
    assert out["env"]["default_bucket_bytes"] == 25 * MiB
    assert err.count("ignoring CCL_BUCKET_MB") == 1


def test_trace_and_check_flags_are_reported(built):
    out, _ = run_child({"CCL_TRACE": "1", "CCL_CHECK": "1"})
    assert out["env"]["trace"] and out["env"]["check"]
    out, _ = run_child({"CCL_TRACE": "0", "CCL_CHECK": "0"})
    assert not out["env"]["trace"] and not out["env"]["check"]


def test_setters_replace_the_environment(built):
    out, _ = run_child({"CCL_MODE": "step", "CCL_BUCKET_MB": "2"},
                       [["mode", "fused"], ["bucket", 4096]])
    assert out["env"]["mode_override"] == "step" and out["env"]["default_bucket_bytes"] == 2 * MiB
    assert out["rc"] == ["ok", "ok"]
    assert out["after"]["mode_override"] == "fused" and out["after"]["default_bucket_bytes"] == 4096
    # None removes the override for good; 0 restores 25 MiB
    out, _ = run_child({"CCL_MODE": "step", "CCL_BUCKET_MB": "2"}, [["mode", None], ["bucket", 0]])
    assert out["after"]["mode_override"] is None and out["after"]["default_bucket_bytes"] == 25 * MiB


def test_setters_reject_bad_values_and_change_nothing(built):
    out, _ = run_child({"CCL_MODE": "step"}, [["mode", 2], ["mode", -2], ["bucket", 3], ["bucket", 1]])
    assert out["rc"] == [1, 1, 1, 1]  # CCL_ERR_INVALID_ARG each time
    assert out["after"] == out["env"]


@pytest.mark.parametrize("value,want", [("staged", "staged"), ("STAGED", "staged"), ("direct", "direct"),
                                        ("Direct", "direct"), ("", "staged")])
def test_host_path_from_environment(built, value, want):
    out, err = run_child({"CCL_HOST_PATH": value})
    assert out["env"]["host_path"] == want
    assert "ignoring" not in err


@pytest.mark.parametrize("value", ["auto", "1", "stage", " direct"])
def test_unreadable_host_path_is_ignored_with_a_warning(built, value):
    out, err = run_child({"CCL_HOST_PATH": value})
    assert out["env"]["host_path"] == "staged"
    assert err.count("ignoring CCL_HOST_PATH") == 1


def test_host_path_setter(built):
    out, _ = run_child({"CCL_HOST_PATH": "direct"}, [["host", "staged"]])
    assert out["env"]["host_path"] == "direct" and out["after"]["host_path"] == "staged"
    out, _ = run_child({}, [["host_raw", 1], ["host_raw", 2], ["host_raw", -1]])
    assert out["rc"] == ["ok", 1, 1]  # CCL_ERR_INVALID_ARG, nothing changed
    assert out["after"]["host_path"] == "direct"
