"""The pins catch plausible mistakes.  Each case plants one mistake in a
copy of the oracle source (a textual edit, compiled to a temporary library),
routes the oracle through it, and checks that at least one pin fails; the
unmodified oracle passes the same pins."""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_backward as B
import test_oracle_codecs as C
import test_oracle_dispatch_combine as D
import test_oracle_layout as LY
import test_oracle_lowlatency as LL
import test_oracle_sources as SRC

HERE = os.path.dirname(os.path.abspath(oracle.__file__))

MUTANTS = [
    ("combine sums k in descending order",
     "for (int32_t k = 0; k < K; ++k) {\n            int64_t row = expert_slot",
     "for (int32_t k = K - 1; k >= 0; --k) {\n            int64_t row = expert_slot"),
    ("combine multiplies and adds separately",
     "acc[h] = fmaf(w, moe_ref_bf16_decode(y[row * H + h]), acc[h]);",
     "acc[h] = acc[h] + w * moe_ref_bf16_decode(y[row * H + h]);"),
    ("bf16 rounds half up",
     "(dropped == 0x8000u && (upper & 1u))", "(dropped == 0x8000u)"),
    ("bf16 truncates",
     "if (dropped > 0x8000u || (dropped == 0x8000u && (upper & 1u))) upper += 1u;", ""),
    ("e4m3 rounds half away from zero",
     "double mant = nearbyint((2.0 * f - 1.0) * 8.0);", "double mant = round((2.0 * f - 1.0) * 8.0);"),
    ("e4m3 saturates to NaN",
     "if (a >= 448.0) return (uint8_t)(sign | 0x7E);", "if (a >= 448.0) return (uint8_t)(sign | 0x7F);"),
    ("e4m3 drops subnormals",
     "double m = nearbyint(a * 512.0);", "double m = 0.0;"),
    ("e4m3 off-by-one exponent bias",
     "((ex + 7) << 3)", "((ex + 8) << 3)"),
    ("fp8 scale uses 480",
     "float s = amax / 448.0f;", "float s = amax / 480.0f;"),
    ("fp8 drops the sign of zero",
     "if (isnan(v)) return 0x7F;\n    uint8_t sign = signbit(v) ? 0x80 : 0x00;",
     "if (isnan(v)) return 0x7F;\n    uint8_t sign = (v < 0) ? 0x80 : 0x00;"),
    ("layout takes the largest id as primary",
     "if (p < 0 || e < p) p = e;", "if (p < 0 || e > p) p = e;"),
    ("layout maps experts to ranks round-robin",
     "if (e < 0 || e >= E || e / m != r) continue;", "if (e < 0 || e >= E || e % R != r) continue;"),
    ("layout counts duplicate ids once",
     "tokens_per_expert[e] += 1;", "tokens_per_expert[e] = 1;"),
    ("layout orders receive rows by token only",
     "slot = recv_expert_offset[p] + seen[p];", "slot = recv_expert_offset[r * m] + seen[r * m];"),
    ("multi-source regions sized by one source",
     "slot = (int32_t)((int64_t)r * T + used);", "slot = (int32_t)((int64_t)r * Ts + used);"),
    ("multi-source walks each source's tokens backwards",
     "for (int32_t t = 0; t < Ts; ++t) {\n                int64_t g = (int64_t)s * Ts + t;",
     "for (int32_t t = Ts - 1; t >= 0; --t) {\n                int64_t g = (int64_t)s * Ts + t;"),
    ("multi-source never writes the per-source offsets",
     "recv_source_offset[(int64_t)r * (S + 1) + s] = used;\n            for",
     "for"),
    ("multi-source leaves region tails uncleared",
     "for (int64_t i = 0; i < (int64_t)R * T; ++i) recv_src_token[i] = -1;", ""),
    ("mxfp8 shared exponent one too large",
     "shared_exp = (e2 - 1) - 8;", "shared_exp = e2 - 8;"),
    ("mxfp8 E8M0 bias 128",
     "recv_scales[slot * nb + b] = (uint8_t)(shared_exp + 127);",
     "recv_scales[slot * nb + b] = (uint8_t)(shared_exp + 128);"),
    ("dispatch backward sums ranks in descending order",
     "for (int32_t r = 0; r < R; ++r) {\n            int64_t row = recv_slot[t * R + r];",
     "for (int32_t r = R - 1; r >= 0; --r) {\n            int64_t row = recv_slot[t * R + r];"),
    ("combine backward leaves grad_y unweighted",
     "float prod = w * g;", "float prod = g;"),
    ("combine backward weights grad_w",
     "dot += (double)g * (double)moe_ref_bf16_decode(y[row * H + h]);",
     "dot += (double)(w * g) * (double)moe_ref_bf16_decode(y[row * H + h]);"),
    ("low-latency ranks entries by k, then token",
     "for (int64_t t = 0; t < T; ++t)\n        for (int32_t k = 0; k < K; ++k) {\n            int32_t e = topk_idx[t * K + k];",
     "for (int32_t k = 0; k < K; ++k)\n        for (int64_t t = 0; t < T; ++t) {\n            int32_t e = topk_idx[t * K + k];"),
    ("low-latency counts dropped entries",
     "int32_t j = tokens_per_expert[e];\n                if (j < cap) {\n                    slot = e * cap + j;\n"
     "                    tokens_per_expert[e] = j + 1;",
     "int32_t j = tokens_per_expert[e]++;\n                if (j < cap) {\n                    slot = e * cap + j;"),
]


def _pins():
    """(name, callable) for a set of pins that run in a few seconds."""
    o = oracle
    return [
        ("e4m3 golden", lambda: C.test_e4m3_golden_values(o)),
        ("e4m3 brute force", lambda: C.test_e4m3_encode_vs_brute_force_random(o)),
        ("e4m3 exact", lambda: C.test_e4m3_encode_vs_exact_rounding(o)),
        ("bf16 golden", lambda: C.test_bf16_golden_values(o)),
        ("bf16 exact", lambda: C.test_bf16_encode_vs_exact_rounding(o)),
        ("layout golden", lambda: LY.test_layout_worked_example(o)),
        ("layout brute force", lambda: LY.test_layout_vs_brute_force(o, 13, 4, 8, 2, 0.2, True, 3)),
        ("sources golden", lambda: SRC.test_sources_worked_example(o)),
        ("sources by sorting", lambda: SRC.test_sources_vs_sorting(o, 3, 20, 4, 16, 4, 0.2, True, 1)),
        ("fp8 exact pipeline", lambda: D.test_dispatch_fp8_vs_exact_pipeline(o)),
        ("combine exact chain", lambda: D.test_combine_vs_exact_fma_chain(o)),
        ("combine ascending k", D.test_combine_sums_in_ascending_k),
        ("combine fused", D.test_combine_uses_fused_multiply_add),
        ("mxfp8 golden", lambda: D.test_mxfp8_golden_values(o)),
        ("mxfp8 exact pipeline", lambda: D.test_mxfp8_vs_exact_pipeline(o)),
        ("low-latency golden", lambda: LL.test_ll_worked_example(o)),
        ("low-latency brute force", lambda: LL.test_ll_vs_brute_force(o, 50, 4, 16, 50, 0.1, False, 0)),
        ("low-latency overflow", lambda: LL.test_ll_vs_brute_force(o, 20, 3, 4, 8, 0.0, True, 2)),
        ("dispatch backward exact", lambda: B.test_dispatch_backward_vs_exact_sum(o)),
        ("dispatch backward ascending r", B.test_dispatch_backward_sums_in_ascending_rank),
        ("combine backward grad_y exact", lambda: B.test_combine_backward_grad_y_exact(o)),
        ("combine backward grad_w fp64", lambda: B.test_combine_backward_grad_w_vs_numpy_fp64(o)),
    ]


def _failing_pins():
    failed = []
    for name, fn in _pins():
        try:
            fn()
        except Exception:          # a failed assertion, or a value the pin cannot even read (NaN)
            failed.append(name)
    return failed


def _build_mutant(tmp, old, new):
    src = open(os.path.join(HERE, "moe_oracle.c")).read()
    assert old in src, "mutation site not found"
    mutated = src.replace(old, new)
    shutil.copy(os.path.join(HERE, "moe_oracle.h"), tmp)
    path_c = os.path.join(tmp, "moe_oracle.c")
    open(path_c, "w").write(mutated)
    so = os.path.join(tmp, "libmutant.so")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-o", so, path_c, "-lm"])
    return oracle.load(so)


def test_unmodified_oracle_passes_the_pins():
    oracle.set_library(None)
    assert _failing_pins() == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new):
    with tempfile.TemporaryDirectory() as tmp:
        try:
            oracle.set_library(_build_mutant(tmp, old, new))
            failed = _failing_pins()
        finally:
            oracle.set_library(None)
    assert failed, f"no pin caught: {name}"
