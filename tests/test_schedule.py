"""The tensor-core kernel's static work partition over CTAs, checked
on the host with the same inline functions the kernels use (compiled with
g++).  No GPU."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "paged_kv_cache_245_gb300", "csrc")
CUDA_INC = "/usr/local/cuda/include"


@pytest.mark.skipif(not os.path.isdir(CUDA_INC) or shutil.which("g++") is None,
                    reason="needs g++ and the CUDA headers")
def test_cta_ranges_tile_exactly_and_owner_inverts(tmp_path):
    exe = tmp_path / "schedule_check"
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, "-I", CUDA_INC,
                    os.path.join(HERE, "schedule_check.cpp"), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "partition check ok" in r.stdout
