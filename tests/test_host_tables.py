"""Host logic of the library that needs no GPU: the table that sets each kernel's
shared-memory attribute once per (kernel, device), compiled with the system C++
compiler from the same header the library uses."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "sparse_attention_mla_gb300", "csrc")


def test_per_device_once_table(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "host_once_check"
    subprocess.check_call([cxx, "-std=c++17", "-O1", "-pthread", "-I", CSRC,
                           os.path.join(ROOT, "tests", "host_once_check.cpp"), "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
