"""The standalone measurement programs under tests/microbench build and run on the GPU.

They time the decode kernels' inner loops and code-load patterns in isolation (the figures behind the
decode-kernel design notes); this test checks that they compile for sm_103a, finish and report every
case.  Their numbers are read from their output, not asserted here.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "microbench")
NVCC = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17"]


def _build_and_run(tmp_path, name, extra=()):
    exe = str(tmp_path / name)
    subprocess.run([NVCC, *ARCH, "-o", exe, os.path.join(HERE, name + ".cu"), *extra], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    return r.stdout


@pytest.mark.gpu
def test_decode_loop(tmp_path):
    out = _build_and_run(tmp_path, "decode_loop")
    assert out.count("base-3 step") == 12 and out.count("2-bit group") == 12, out


@pytest.mark.gpu
def test_load_pattern(tmp_path):
    out = _build_and_run(tmp_path, "load_pattern", ["-lcuda"])
    assert out.count("us per launch") == 7, out


@pytest.mark.gpu
def test_mma_fp8_vs_f16(tmp_path):
    out = _build_and_run(tmp_path, "mma_fp8_vs_f16")
    assert out.count("weights/clk/SM") == 6 and "accuracy" in out, out
