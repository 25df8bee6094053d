"""The FP8 dispatch divides each value by its block scale with Markstein's
FMA-corrected quotient (see csrc/fp8_quant.cuh).  This checks it against
CUDA's IEEE division __fdiv_rn bit for bit: every bf16 value x with
|x| <= amax, for a few thousand block maxima amax spread over the whole
bf16 exponent range (s = amax / 448)."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.fixture(scope="module")
def divcheck():
    assert torch.cuda.is_available()
    out_dir = os.path.join(HERE, "cuda", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libfp8_div_check.so")
    from combine_moe_dispatch_02_gb300 import build
    subprocess.check_call([build.nvcc(), *build.ARCH, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                           "-I", build.CSRC, "-I", build.INCLUDE, os.path.join(HERE, "cuda", "fp8_div_check.cu"),
                           "-o", so])
    lib = ctypes.CDLL(so)
    lib.fp8_div_check.restype = ctypes.c_int
    lib.fp8_div_check.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                  ctypes.c_void_p]
    return lib


def test_fast_quotient_matches_ieee_division(divcheck):
    rng = np.random.default_rng(0)
    # positive finite bf16 maxima: random patterns over all exponents, powers of
    # two, all-ones mantissas, and the smallest / largest magnitudes
    pats = set(int(p) for p in rng.integers(0x0001, 0x7F80, 3000))
    pats |= {e << 7 for e in range(1, 255)}
    pats |= {(e << 7) | 0x7F for e in range(0, 255)}
    pats |= {0x0001, 0x0080, 0x7F7F, 0x3F80, 0x4000, 0x43E0}
    amax = torch.tensor(sorted(pats), dtype=torch.int32).to(torch.int16).cuda()
    mism = torch.zeros(1, dtype=torch.int64, device="cuda")
    checked = torch.zeros(1, dtype=torch.int64, device="cuda")
    ex = torch.zeros(64, dtype=torch.int32, device="cuda")
    rc = divcheck.fp8_div_check(amax.data_ptr(), amax.numel(), mism.data_ptr(), ex.data_ptr(), 16,
                                checked.data_ptr())
    assert rc == 0
    n_bad, n = int(mism.item()), int(checked.item())
    assert n > 50_000_000
    assert n_bad == 0, ex.view(-1, 4)[:min(n_bad, 16)].cpu().numpy()
