"""AddressSanitizer + UndefinedBehaviorSanitizer builds of the host code,
run without a GPU (compute-sanitizer, the device-side tool, is closed on this
pool; these cover the CPU side).

* the C oracle, linked with tests/sanitize/oracle_driver.c, on small inputs
  with special values and edge shapes;
* libkmassign's host code (argument checks, error texts, the planner)
  compiled by nvcc with the sanitizers on its host side and driven by
  tests/sanitize/host_driver.c through the C ABI.

Each driver exits non-zero on the first sanitizer report (recovery off) or
failed property."""

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
from means_nearest_centroid_gb300 import _build  # noqa: E402

HERE = os.path.join(ROOT, "tests", "sanitize")
SAN_C = ["-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-fno-omit-frame-pointer"]
ENV = dict(os.environ, ASAN_OPTIONS="protect_shadow_gap=0:detect_leaks=0:abort_on_error=0",
           UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")


def _have_sanitizers(tmp):
    gcc = shutil.which("gcc")
    if gcc is None:
        return False
    src = os.path.join(tmp, "probe.c")
    with open(src, "w") as f:
        f.write("int main(void){return 0;}\n")
    r = subprocess.run([gcc, *SAN_C, src, "-o", os.path.join(tmp, "probe")],
                       capture_output=True, text=True)
    return r.returncode == 0


def test_oracle_under_asan_ubsan(tmp_path):
    if not _have_sanitizers(str(tmp_path)):
        pytest.skip("gcc with AddressSanitizer/UBSan not available")
    exe = str(tmp_path / "oracle_driver")
    cmd = ["gcc", "-std=c11", "-O1", "-g", *SAN_C, "-fno-fast-math", "-ffp-contract=off",
           os.path.join(HERE, "oracle_driver.c"), os.path.join(ROOT, "oracle", "kmassign_oracle.c"),
           "-o", exe, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, env=ENV, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok" in r.stdout


def test_library_host_code_under_asan_ubsan(tmp_path):
    if not _have_sanitizers(str(tmp_path)):
        pytest.skip("gcc with AddressSanitizer/UBSan not available")
    try:
        nvcc = _build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    san = []
    for flag in SAN_C:
        for part in flag.split(","):   # nvcc splits -Xcompiler values at commas
            if part.startswith("-"):
                san += ["-Xcompiler", part]
            else:
                san += ["-Xcompiler", "-fsanitize=" + part]
    objs, procs = [], []
    for src in _build.SOURCES:
        obj = str(tmp_path / (os.path.splitext(src)[0] + ".o"))
        objs.append(obj)
        procs.append(subprocess.Popen(
            [nvcc, *_build.ARCH, "-O1", "-g", "-std=c++17", "-Xcompiler", "-fPIC", *san,
             "-I", _build.INCLUDE, "-c", os.path.join(_build.CSRC, src), "-o", obj],
            stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    for p in procs:
        out, err = p.communicate()
        assert p.returncode == 0, err
    lib = str(tmp_path / "libkmassign_san.so")
    r = subprocess.run([nvcc, *_build.ARCH, "-shared", "-Xcompiler", "-fsanitize=address",
                        "-Xcompiler", "-fsanitize=undefined", "-o", lib, *objs],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    exe = str(tmp_path / "host_driver")
    r = subprocess.run(["gcc", "-std=c11", "-O1", "-g", *SAN_C, "-I", _build.INCLUDE,
                        os.path.join(HERE, "host_driver.c"), "-L", str(tmp_path),
                        "-lkmassign_san", "-Wl,-rpath," + str(tmp_path), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, env=ENV, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok" in r.stdout
