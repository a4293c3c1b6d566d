"""The C ABI used from C: tests/c_abi_client.c is compiled against include/clcgemm.h,
linked with the library, the CUDA runtime and (as the comparator) the CPU oracle, and run."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client(tmp_path):
    import blackwell_clc_dynamic_gb300 as m
    import oracle
    oracle._load()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "c_abi_client"
    cc = shutil.which("gcc") or "cc"
    cmd = [cc, "-std=c11", "-O1", os.path.join(ROOT, "tests", "c_abi_client.c"), "-o", str(exe),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           m.LIB_PATH, oracle.LIB_PATH, "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-Wl,-rpath," + os.path.dirname(m.LIB_PATH), "-Wl,-rpath," + os.path.dirname(oracle.LIB_PATH),
           "-Wl,-rpath," + os.path.join(cuda, "lib64"), "-lm"]
    subprocess.run(cmd, check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C client ok" in r.stdout
