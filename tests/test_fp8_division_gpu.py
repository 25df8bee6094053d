"""The FP8 dispatch replaces divisions by fused multiply-adds (Markstein's
correction step, csrc/fp8_quant.cuh).  This checks it against CUDA's IEEE
operations: the block scale amax/448 and the reciprocal 1/s for every
positive finite bf16 block maximum, and the quotient x/s for every bf16
value x with |x| <= amax, for a few thousand block maxima spread over the
whole bf16 exponent range: scales and reciprocals agree bit for bit, the
quotients wherever the method is claimed exact, and the E4M3 codes
everywhere; the same for the magnitude form (quotient of |x|, sign bit of x
OR'ed into the code) that the wide dispatch kernel uses, whose packed
two-value form must equal the scalar one bit for bit."""
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
    lib.fp8_div_check.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    return lib


def _run(divcheck, pats):
    amax = torch.tensor(sorted(pats), dtype=torch.int32).to(torch.int16).cuda()
    counters = torch.zeros(8, dtype=torch.int64, device="cuda")
    ex = torch.zeros(2 * 16 * 4, dtype=torch.int32, device="cuda")
    rc = divcheck.fp8_div_check(amax.data_ptr(), amax.numel(), counters.data_ptr(), ex.data_ptr(), 16)
    assert rc == 0
    return [int(v) for v in counters.cpu()], ex.view(2, 16, 4).cpu().numpy()


def test_scale_and_reciprocal_for_every_bf16_block_max(divcheck):
    (_, _, _, scale_bad, recip_bad, _, _, _), _ = _run(divcheck, range(0x0001, 0x7F80))
    assert scale_bad == 0 and recip_bad == 0


def test_fast_quotient_matches_ieee_division(divcheck):
    rng = np.random.default_rng(0)
    # positive finite bf16 maxima: random patterns over all exponents, powers of
    # two, all-ones mantissas, and the smallest / largest magnitudes
    pats = set(int(p) for p in rng.integers(0x0001, 0x7F80, 3000))
    pats |= {e << 7 for e in range(1, 255)}
    pats |= {(e << 7) | 0x7F for e in range(0, 255)}
    pats |= {0x0001, 0x0080, 0x7F7F, 0x3F80, 0x4000, 0x43E0}
    (q_bad, code_bad, n, scale_bad, recip_bad, mag_bad, sign_bad, packed_bad), ex = _run(divcheck, pats)
    assert n > 20_000_000                       # pairs inside the fast scale range
    assert q_bad == 0, ex[0][:min(q_bad, 16)]
    assert code_bad == 0, ex[1][:min(code_bad, 16)]
    assert scale_bad == 0 and recip_bad == 0
    # the wide dispatch kernel quantises |x| and ORs the sign of x into the code
    assert mag_bad == 0 and sign_bad == 0
    assert packed_bad == 0
