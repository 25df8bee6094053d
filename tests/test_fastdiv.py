"""The dispatch kernels decode an item index into (token, segment) with a
multiply-high by a host-computed constant instead of a division
(csrc/fastdiv.h: Granlund and Montgomery's round-up method).  The host
copy of the same code is compiled with the host C++ compiler and checked
against the division operator for every divisor up to 4096 and a few
large ones, on small, boundary, random and top-of-range numerators."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "combine_moe_dispatch_02_gb300", "csrc")


def test_fastdiv_matches_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "fastdiv_check"
    subprocess.check_call([cxx, "-O2", "-std=c++17", "-I", CSRC, os.path.join(HERE, "cuda", "fastdiv_check.cpp"),
                           "-o", str(exe)])
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout
    bad, n = (int(v) for v in r.stdout.split()[-2:])
    assert bad == 0 and n > 50_000_000
