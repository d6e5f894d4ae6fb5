"""Kernel attributes (the dynamic shared-memory limit of the top-k, attention
and decode kernels) belong to one device's context, so the library sets them
once per device index and returns the CUDA result of that set-up on every
later launch from the same device. The per-device logic is plain C++
(csrc/device_once.h); this test compiles it with a fake device getter and
counts the set-ups, without a GPU."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "lazy_sparse_attention_token_b300", "csrc")
SRC = os.path.join(ROOT, "tests", "native", "device_once_check.cpp")


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_attribute_setup_runs_once_per_device(tmp_path):
    exe = str(tmp_path / "device_once_check")
    subprocess.check_call(["g++", "-std=c++17", "-O1", "-pthread", "-I", CSRC, SRC, "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr


def test_every_attribute_setter_goes_through_the_per_device_helper():
    """No launcher sets a kernel attribute under a process-wide once-flag."""
    for name in os.listdir(CSRC):
        if not name.endswith(".cu"):
            continue
        text = open(os.path.join(CSRC, name)).read()
        n_set = text.count("cudaFuncSetAttribute(")
        if n_set:
            assert "once_per_device(" in text, name
            # every setter sits inside a per-device once lambda whose result is checked
            assert text.count("once_per_device(") >= 1 and "if (ea != cudaSuccess) return ea;" in text, name
