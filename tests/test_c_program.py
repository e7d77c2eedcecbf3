"""The C ABI used from a plain C program (tests/c/nvfp4_abi_demo.c), compiled
with gcc against include/nvfp4.h and linked to the library."""
import os
import subprocess

import pytest

import nvfp4_bit_block_gb300 as nv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_demo(tmp_path):
    lib = nv.build()
    exe = str(tmp_path / "nvfp4_abi_demo")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c", "nvfp4_abi_demo.c"),
           "-o", exe, lib, "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(lib), "-Wl,-rpath," + os.path.join(CUDA, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_host_checks(tmp_path):
    r = subprocess.run([build_demo(tmp_path)], capture_output=True, text=True, timeout=120,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stdout + r.stderr
    assert "host checks passed" in r.stdout


@pytest.mark.gpu
def test_c_program_on_the_gpu(tmp_path):
    r = subprocess.run([build_demo(tmp_path)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "gpu checks passed" in r.stdout
