"""Host-side C++ units of the library, built with g++ and run on the CPU:
the per-device-context set-up flags (csrc/device_once.h) that the kernel
launchers use to raise each kernel's shared-memory limit once per device
context, checked with made-up device ordinals and context ids."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "long_context_causal_blockwise_gb300", "csrc")


@pytest.mark.skipif(shutil.which("g++") is None, reason="g++ not installed")
def test_device_once_is_keyed_by_device_and_context(tmp_path):
    exe = tmp_path / "device_once_check"
    src = os.path.join(ROOT, "tests", "host", "device_once_check.cc")
    subprocess.run(["g++", "-std=c++17", "-O1", "-Wall", "-Werror", "-I" + CSRC, src, "-o", str(exe), "-lpthread"],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.strip() == "ok"


def test_no_launcher_keeps_a_process_wide_attribute_flag():
    """Every kernel launcher raises its shared-memory limit through the
    per-device-context flags; none keeps a process-wide static bool."""
    import re

    for name in os.listdir(CSRC):
        if not name.endswith(".cu"):
            continue
        text = open(os.path.join(CSRC, name)).read()
        assert not re.search(r"static\s+bool", text), name
        for m in re.finditer(r"cudaFuncSetAttribute\(", text):
            assert name == "api.cu", f"{name} sets a function attribute outside set_smem_limit_once"
