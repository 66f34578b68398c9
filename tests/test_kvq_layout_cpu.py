"""The Q8_0 cache layout shared by the quantiser and the attention kernel, checked on the host: the native
check (tests/native/kvq_layout_check.cu, compiled here with nvcc for the host only) runs the layout's own
position functions and restates the attention kernel's staging and read addresses."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_kvq_layout(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc) and not shutil.which("nvcc"):
        pytest.skip("nvcc not available")
    exe = tmp_path / "kvq_layout_check"
    src = os.path.join(HERE, "native", "kvq_layout_check.cu")
    r = subprocess.run([nvcc, "-std=c++17", "-O1", src, "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
