"""The C ABI from a plain C99 program (tests/cuda/abi_roundtrip.c): built
with nvcc against include/moe_ep.h and the in-tree libmoe_ep.so, it runs
layout -> bf16 dispatch -> identity expert -> combine with its own CUDA
runtime allocations and checks the round trip bit for bit."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_roundtrip(tmp_path):
    from combine_moe_dispatch_02_gb300 import build
    build.build()
    pkg = os.path.dirname(build.LIB_PATH)
    exe = str(tmp_path / "abi_roundtrip")
    cmd = [build.nvcc(), "-x", "c", "-O2", "-Xcompiler", "-std=c99,-Wall", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "cuda", "abi_roundtrip.c"), "-o", exe,
           "-L", pkg, "-lmoe_ep", "-Xlinker", f"-rpath={pkg}"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "abi roundtrip ok" in r.stdout
