"""The C ABI used from plain C: build tests/c_abi_example.c against
include/kmassign.h and libkmassign.so, run it (needs a GB300)."""

import os
import shutil
import subprocess

import pytest
import torch

from means_nearest_centroid_gb300 import _build

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


def test_plain_c_program(tmp_path):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = _build.build()
    nvcc = _build.nvcc()
    exe = str(tmp_path / "c_abi_example")
    cuda_root = os.path.dirname(os.path.dirname(nvcc))
    cmd = [shutil.which("gcc") or "gcc", "-std=c11", "-O1", os.path.join(HERE, "c_abi_example.c"),
           "-I", _build.INCLUDE, "-I", os.path.join(cuda_root, "include"),
           "-L", os.path.dirname(lib), "-lkmassign", "-L", os.path.join(cuda_root, "lib64"),
           "-lcudart", "-Wl,-rpath," + os.path.dirname(lib),
           "-Wl,-rpath," + os.path.join(cuda_root, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok" in r.stdout
