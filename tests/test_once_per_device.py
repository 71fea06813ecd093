"""Host-only check of the per-device attribute opt-in logic of the kernel
launchers (once_on_device in csrc/da_internal.h): compiled with the host
compiler against the CUDA headers and run on the CPU (no GPU call)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "cpp", "once_per_device_check.cc")
CSRC = os.path.join(ROOT, "differential_attention_causal_gb300", "csrc")


def _cuda_include():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "include", "cuda_runtime.h")):
            return os.path.join(c, "include")
    return None


def test_once_per_device_logic(tmp_path):
    inc = _cuda_include()
    cxx = shutil.which("g++")
    if inc is None or cxx is None:
        pytest.skip("no CUDA headers or host C++ compiler")
    exe = str(tmp_path / "once_check")
    subprocess.run([cxx, "-std=c++17", "-O1", "-pthread", "-I", inc, "-I", CSRC, SRC, "-o", exe], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
