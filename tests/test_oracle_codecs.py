"""Pins for the oracle's number codecs (bf16 and FP8 E4M3).

Expected values come from hand-derived fixtures (tests/golden), exact rational
rounding written from the format definitions (tests/exact.py), a brute-force
nearest-code search, and torch's CPU conversions as a library special case --
never from the oracle itself.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from exact import bf16_value, rn_bf16, rn_e4m3_sat

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            parts = line.split()
            rows.append((float(parts[0]), int(parts[1], 16)))
    return rows


def _torch_e4m3_values():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


# ------------------------------------------------------------------ E4M3

def test_e4m3_golden_values(oracle_lib):
    for v, code in _read_table("e4m3_values.txt"):
        assert oracle_lib.e4m3_encode(v) == code, (v, hex(code), hex(oracle_lib.e4m3_encode(v)))


def test_e4m3_decode_matches_library_table(oracle_lib):
    table = _torch_e4m3_values()
    for q in range(256):
        ours = oracle_lib.e4m3_decode(q)
        if np.isnan(table[q]):
            assert np.isnan(ours), q
        else:
            assert ours == table[q], (q, ours, table[q])
    # the NaN codes are exactly S.1111.111
    assert [q for q in range(256) if np.isnan(table[q])] == [0x7F, 0xFF]


def test_e4m3_encode_roundtrips_every_finite_code(oracle_lib):
    table = _torch_e4m3_values()
    for q in range(256):
        if q in (0x7F, 0xFF):
            continue
        assert oracle_lib.e4m3_encode(float(table[q])) == q, hex(q)


def _structured_f32_inputs():
    """Every exponent that matters for E4M3 (2^-12 .. 2^9) x every pattern of the
    top 8 mantissa bits x low-bit patterns that hit exact ties and their
    neighbours, both signs."""
    exps = np.arange(127 - 12, 127 + 10, dtype=np.uint32)
    top = np.arange(256, dtype=np.uint32) << 15
    low = np.array([0, 1, 0x3FFF, 0x4000, 0x4001, 0x7FFF], dtype=np.uint32)
    bits = (exps[:, None, None] << 23) | top[None, :, None] | low[None, None, :]
    bits = bits.ravel()
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    return bits.view(np.float32)


def _brute_force_e4m3(v: np.ndarray) -> np.ndarray:
    """Nearest finite E4M3 code by exhaustive distance to all 127 non-negative
    finite codes; ties -> the code whose lowest mantissa bit is 0; magnitudes
    past 448 saturate.  Code values come from torch's decode table."""
    table = _torch_e4m3_values()
    pos_codes = np.arange(0x7F)                      # 0x00 .. 0x7E, increasing values
    pos_vals = table[pos_codes]
    a = np.abs(v.astype(np.float64))
    d = np.abs(a[:, None] - pos_vals[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    # among the nearest codes prefer an even one (there are at most two)
    even = (pos_codes[None, :] % 2 == 0) & cand
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    codes = pos_codes[pick]
    codes = np.where(a >= 448.0, 0x7E, codes)
    return (codes | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


def test_e4m3_encode_vs_brute_force_structured(oracle_lib):
    v = _structured_f32_inputs()
    ours = oracle_lib.e4m3_encode_array(v)
    ref = _brute_force_e4m3(v)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(ours[i]), hex(ref[i])) for i in bad[:10]]


def test_e4m3_encode_vs_brute_force_random(oracle_lib):
    rng = np.random.default_rng(1234)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 100,
        (rng.standard_normal(20000) * 0.01).astype(np.float32),
        rng.uniform(-600, 600, 5000).astype(np.float32),
    ])
    ours = oracle_lib.e4m3_encode_array(v)
    assert np.array_equal(ours, _brute_force_e4m3(v))


def test_e4m3_encode_vs_library_conversion(oracle_lib):
    """torch's float -> float8_e4m3fn (round to nearest even) agrees on every
    input inside the finite range (torch does not saturate, so |v| <= 448)."""
    v = _structured_f32_inputs()
    v = v[np.abs(v) <= 448.0]
    ours = oracle_lib.e4m3_encode_array(v)
    lib = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, lib)


def test_e4m3_encode_vs_exact_rounding(oracle_lib):
    rng = np.random.default_rng(99)
    v = np.concatenate([rng.standard_normal(3000) * 50, rng.standard_normal(1000) * 0.003]).astype(np.float32)
    table = _torch_e4m3_values()
    for x in v:
        want = rn_e4m3_sat(Fraction(float(x)))
        got = table[oracle_lib.e4m3_encode(float(x))]
        assert Fraction(float(got)) == want, (float(x), got, float(want))


def test_e4m3_nan_maps_to_nan_code(oracle_lib):
    assert oracle_lib.e4m3_encode(float("nan")) == 0x7F


# ------------------------------------------------------------------ bf16

def test_bf16_golden_values(oracle_lib):
    for v, code in _read_table("bf16_values.txt"):
        assert oracle_lib.bf16_encode(v) == code, (v, hex(code), hex(oracle_lib.bf16_encode(v)))


def test_bf16_encode_vs_library(oracle_lib):
    rng = np.random.default_rng(7)
    bits = np.concatenate([
        rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32),
        # exact ties and neighbours around them
        (rng.integers(0, 2 ** 16, 20000, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8000),
        (rng.integers(0, 2 ** 16, 20000, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x7FFF),
        (rng.integers(0, 2 ** 16, 20000, dtype=np.uint64).astype(np.uint32) << 16) | np.uint32(0x8001),
    ])
    v = bits.view(np.float32)
    v = v[~np.isnan(v)]
    lib = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    f = oracle_lib.lib().moe_ref_bf16_encode
    ours = np.fromiter((f(float(x)) for x in v), dtype=np.uint16, count=v.size)
    assert np.array_equal(ours, lib)


def test_bf16_encode_vs_exact_rounding(oracle_lib):
    rng = np.random.default_rng(3)
    for x in rng.standard_normal(3000).astype(np.float32) * 10:
        got = bf16_value(oracle_lib.bf16_encode(float(x)))
        assert got == rn_bf16(Fraction(float(x))), float(x)


def test_bf16_decode_is_upper_half(oracle_lib):
    for b in (0x0000, 0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8001):
        assert Fraction(oracle_lib.bf16_decode(b)) == bf16_value(b)
