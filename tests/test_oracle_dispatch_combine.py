"""Pins for the oracle's dispatch (bf16, FP8) and combine.

Expected values come from exact rational arithmetic written from the IEEE /
OCP rounding definitions (tests/exact.py), numpy + torch CPU library
routines composed step by step, closed forms and error bounds, and the
dispatch -> identity expert -> combine invariant; never from the oracle.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from combine_moe_dispatch_02_gb300.inputs import (WORKLOADS, bf16_bits, make_inputs, random_routing,
                                                  random_weights)
from exact import bf16_value, bits_of_f32, rn_bf16, rn_e4m3_sat, rn_f32


def _x_bits(T, H, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return bf16_bits((torch.randn(T, H, generator=g) * scale).to(torch.bfloat16))


def _torch_e4m3_table():
    return torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn).float().numpy()


# ---------------------------------------------------------------- bf16 dispatch

def test_dispatch_bf16_copies_rows(oracle_lib):
    T, H, E, R, K = 37, 64, 12, 4, 3
    idx = random_routing(T, K, E, 11, mask_frac=0.15).numpy()
    L = oracle_lib.layout(idx, None, E, R)
    x = _x_bits(T, H, 1)
    sentinel = np.full((L.capacity, H), 0xABCD, np.uint16)
    recv, st = oracle_lib.dispatch_bf16(x, L, sentinel.copy())
    assert st == 0
    written = np.zeros(L.capacity, bool)
    for t in range(T):
        for r in range(R):
            s = L.recv_slot[t, r]
            if s >= 0:
                assert np.array_equal(recv[s], x[t])
                written[s] = True
    assert np.all(recv[~written] == 0xABCD)            # rows past the last pair untouched
    assert written.sum() == L.n_pairs


# ---------------------------------------------------------------- FP8 dispatch

def _exact_fp8_block(xb):
    """Exact pipeline for one 128-column block: amax (exact), s = RN32(amax/448),
    q = E4M3_RNE_sat(RN32(x/s)); all-zero block -> s = 0, q = +0."""
    vals = [bf16_value(int(b)) for b in xb]
    amax = max(abs(v) for v in vals)
    s = rn_f32(amax / 448)
    if amax == 0:
        return [Fraction(0)] * len(vals), s
    return [rn_e4m3_sat(rn_f32(v / s)) for v in vals], s


def test_dispatch_fp8_vs_exact_pipeline(oracle_lib):
    T, H, E, R, K = 3, 256, 8, 2, 2
    idx = np.array([[0, 5], [7, 6], [2, 3]], np.int32)
    L = oracle_lib.layout(idx, None, E, R)
    x = _x_bits(T, H, 5, scale=3.0)
    x[1, 128:] = 0                                        # an all-zero block
    x[2, 7] = 0x8000                                      # a negative zero in a live block
    q, s, st = oracle_lib.dispatch_fp8(x, L)
    assert st == 0
    table = _torch_e4m3_table()
    for t in range(T):
        for b in range(H // 128):
            want_q, want_s = _exact_fp8_block(x[t, b * 128:(b + 1) * 128])
            for r in range(R):
                slot = L.recv_slot[t, r]
                if slot < 0:
                    continue
                assert Fraction(float(s[slot, b])) == want_s
                got = [Fraction(float(table[c])) for c in q[slot, b * 128:(b + 1) * 128]]
                assert got == want_q, (t, b)
    z = L.recv_slot[1][L.recv_slot[1] >= 0]
    assert np.all(q[z, 128:] == 0x00) and np.all(s[z, 1] == 0.0)
    neg0 = L.recv_slot[2][L.recv_slot[2] >= 0]
    assert np.all(q[neg0, 7] == 0x80)


def test_dispatch_fp8_vs_library_pipeline(oracle_lib):
    """Same recipe composed from numpy (exact max, IEEE fp32 divisions) and
    torch's float8_e4m3fn conversion, on a DeepSeek-V3-shaped slice."""
    T, H, E, R, K = 64, 7168, 256, 8, 8
    inp = make_inputs(WORKLOADS["dsv3"].scaled(T), with_y=False)
    L = oracle_lib.layout(inp.topk_idx.numpy(), None, E, R)
    x = bf16_bits(inp.x)
    q, s, st = oracle_lib.dispatch_fp8(x, L)
    assert st == 0
    xf = inp.x.float().numpy().reshape(T, H // 128, 128)
    amax = np.abs(xf).max(axis=2)
    scale = (amax / np.float32(448.0)).astype(np.float32)
    with np.errstate(invalid="ignore", divide="ignore"):
        v = (xf / scale[:, :, None]).astype(np.float32)
    v = np.clip(v, -448, 448)                      # torch's conversion does not saturate
    ref_q = torch.from_numpy(v.reshape(T, H)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t in range(T):
        for r in range(R):
            slot = L.recv_slot[t, r]
            if slot >= 0:
                assert np.array_equal(q[slot], ref_q[t])
                assert np.array_equal(s[slot], scale[t])


def test_dispatch_fp8_error_bound_and_full_scale(oracle_lib):
    T, H, E, R, K = 48, 1024, 16, 4, 4
    idx = random_routing(T, K, E, 21).numpy()
    L = oracle_lib.layout(idx, None, E, R)
    x = _x_bits(T, H, 9, scale=10.0)
    q, s, st = oracle_lib.dispatch_fp8(x, L)
    assert st == 0
    table = _torch_e4m3_table().astype(np.float64)
    xf = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    for t in range(T):
        slot = L.recv_slot[t][L.recv_slot[t] >= 0][0]
        for b in range(H // 128):
            xb = xf[t, b * 128:(b + 1) * 128]
            qb = table[q[slot, b * 128:(b + 1) * 128]]
            sb = float(s[slot, b])
            # closed form: the block's largest magnitude maps to +-448 exactly
            assert np.max(np.abs(qb)) == 448.0
            # E4M3 keeps 3 mantissa bits: half-ulp relative error 2^-4 for normal
            # results, absolute 2^-10 (half of the 2^-9 quantum) for subnormal ones;
            # plus the fp32 rounding of x/s (relative 2^-24).
            v = xb / sb
            err = np.abs(qb - v)
            normal = np.abs(qb) >= 2.0 ** -6
            assert np.all(err[normal] <= (2.0 ** -4 + 2.0 ** -20) * np.abs(v[normal]))
            assert np.all(err[~normal] <= 2.0 ** -10 + 2.0 ** -20)


# ---------------------------------------------------------------- combine

def _exact_combine(y_rows, w_row):
    """fp32 fused multiply-add chain in ascending k, exact per step, then RNE bf16."""
    acc = Fraction(0)
    for yb, w in zip(y_rows, w_row):
        acc = rn_f32(Fraction(float(w)) * bf16_value(int(yb)) + acc)
    return rn_bf16(acc)


def _bf16_bits_of_fraction(q: Fraction) -> int:
    return bits_of_f32(float(q)) >> 16


def test_combine_vs_exact_fma_chain(oracle_lib):
    T, H, E, R, K = 12, 48, 8, 4, 5
    idx = random_routing(T, K, E, 31, mask_frac=0.2).numpy()
    w = random_weights(T, K, 31).numpy()
    L = oracle_lib.layout(idx, w, E, R)
    y = _x_bits(T * K, H, 77, scale=2.0)
    out, st = oracle_lib.combine(y, L.expert_slot, w)
    assert st == 0
    for t in range(T):
        ks = [k for k in range(K) if L.expert_slot[t, k] >= 0]
        for h in range(H):
            want = _exact_combine([y[L.expert_slot[t, k], h] for k in ks], [w[t, k] for k in ks])
            assert out[t, h] == _bf16_bits_of_fraction(want), (t, h)


def test_combine_sums_in_ascending_k():
    """2^24 + 1 - 2^24 in fp32: ascending order gives 0 (the +1 is absorbed),
    any order that adds -2^24 before +1 gives 1."""
    import oracle
    y = np.array([[0x4B80], [0x3F80], [0xCB80]], np.uint16)     # 2^24, 1, -2^24 in bf16
    slot = np.array([[0, 1, 2]], np.int32)
    w = np.ones((1, 3), np.float32)
    out, st = oracle.combine(y, slot, w)
    assert st == 0 and out[0, 0] == 0x0000


def test_combine_uses_fused_multiply_add():
    """w1*y1 = 1 exactly; w2*y2 = 2^-8 + 2^-24 + d with 0 < d < 2^-32.  Fused:
    fp32(1 + 2^-8 + 2^-24 + d) = 1 + 2^-8 + 2^-23, which rounds up to bf16
    1 + 2^-7.  Unfused: fp32(w2*y2) = 2^-8 + 2^-24, the sum is an fp32 tie that
    goes to 1 + 2^-8, a bf16 tie that goes to 1.0."""
    import oracle
    target_lo = Fraction(1, 2 ** 8) + Fraction(1, 2 ** 24)
    found = None
    for ym in range(1, 128):                      # y2 = 1 + ym/128, a bf16 value
        y2 = 1 + Fraction(ym, 128)
        n = (target_lo / y2) * 2 ** 31            # w2 = n * 2^-31 lies in [2^-9, 2^-8): 24-bit grid
        n = int(n) + 1
        w2 = Fraction(n, 2 ** 31)
        d = w2 * y2 - target_lo
        if 0 < d < Fraction(1, 2 ** 32) and n < 2 ** 24:
            found = (ym, w2)
            break
    assert found is not None
    ym, w2 = found
    y2_bits = 0x3F80 + ym
    y = np.array([[0x3F80], [y2_bits]], np.uint16)
    slot = np.array([[0, 1]], np.int32)
    w = np.array([[1.0, float(w2)]], np.float32)
    assert Fraction(float(w[0, 1])) == w2
    out, st = oracle.combine(y, slot, w)
    assert st == 0 and out[0, 0] == 0x3F81


def test_combine_masked_token_gives_positive_zero(oracle_lib):
    y = np.full((2, 16), 0x3F80, np.uint16)
    slot = np.array([[-1, -1], [0, -1]], np.int32)
    w = np.array([[0.5, 0.5], [-1.0, 3.0]], np.float32)
    out, st = oracle_lib.combine(y, slot, w)
    assert st == 0
    assert np.all(out[0] == 0x0000) and np.all(out[1] == 0xBF80)


def test_combine_within_one_ulp_of_fp64(oracle_lib):
    T, H, E, R, K = 256, 128, 16, 4, 2
    inp = make_inputs(WORKLOADS["tiny"])
    L = oracle_lib.layout(inp.topk_idx.numpy(), inp.topk_w.numpy(), E, R)
    y = bf16_bits(inp.y)
    out, st = oracle_lib.combine(y, L.expert_slot, inp.topk_w.numpy())
    assert st == 0
    yd = inp.y.double().numpy()
    wd = inp.topk_w.double().numpy()
    ref = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            ref[t] += wd[t, k] * yd[L.expert_slot[t, k]]
    got = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).double().numpy()
    # one bf16 ulp at the reference's magnitude (8 significand bits)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -126))) - 7)
    assert np.all(np.abs(got - ref) <= ulp)


@pytest.mark.parametrize("name", ["tiny", "ds16_wide"])
def test_dispatch_identity_combine_returns_x(oracle_lib, name):
    """bf16 dispatch -> identity expert -> combine with weights summing to 1
    gives back x exactly (the fp32 sum differs from x by ~K * 2^-24 relative,
    far inside half a bf16 ulp)."""
    wl = WORKLOADS[name]
    if wl.T > 1024:
        wl = wl.scaled(1024)
    inp = make_inputs(wl, with_y=False)
    L = oracle_lib.layout(inp.topk_idx.numpy(), inp.topk_w.numpy(), wl.E, wl.R)
    x = bf16_bits(inp.x)
    recv, st = oracle_lib.dispatch_bf16(x, L)
    assert st == 0
    n = wl.T * wl.K
    y = recv[L.expert_src_row[:n]]                 # identity expert, expert-major rows
    out, st = oracle_lib.combine(y, L.expert_slot, inp.topk_w.numpy())
    assert st == 0
    assert np.array_equal(out, x)


# ---------------------------------------------------------------- MXFP8 dispatch

def _read_mx_golden():
    import os
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "mxfp8_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                p = line.split()
                rows.append((float(p[0]), int(p[1]), int(p[2]), float(p[3]), int(p[4], 16)))
    return rows


def _bf16_bits_of(v: float) -> int:
    return int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()) & 0xFFFF


def test_mxfp8_golden_values(oracle_lib):
    """Each golden line becomes one 32-value block: amax at column 0 (as +amax),
    x at column 1, zeros elsewhere (a zero-amax line: an all-zero block)."""
    rows = _read_mx_golden()
    T, H = len(rows), 32
    x = np.zeros((T, H), np.uint16)
    for t, (amax, _, _, xv, _) in enumerate(rows):
        x[t, 0] = _bf16_bits_of(amax)
        x[t, 1] = _bf16_bits_of(xv)
        assert float(torch.tensor([xv]).to(torch.bfloat16)) == xv      # fixtures are bf16 values
    idx = np.arange(T, dtype=np.int32).reshape(T, 1) % 4
    L = oracle_lib.layout(idx, None, 4, 4)
    q, s, st = oracle_lib.dispatch_mxfp8(x, L)
    assert st == 0
    for t, (amax, se, byte, xv, code) in enumerate(rows):
        slot = L.recv_slot[t][L.recv_slot[t] >= 0][0]
        assert s[slot, 0] == byte == se + 127, (t, s[slot, 0], byte)
        assert q[slot, 1] == code, (t, hex(q[slot, 1]), hex(code))


def _exact_mx_block(xb):
    """From the OCP MX definition, exactly: s = floor(log2 amax) - 8 (clamped), q = E4M3(RN32(x * 2^-s))."""
    import math
    vals = [bf16_value(int(b)) for b in xb]
    amax = max(abs(v) for v in vals)
    if amax == 0:
        s = -127
    else:
        s = math.floor(math.log2(amax))
        while Fraction(2) ** s > amax:          # guard the float log2
            s -= 1
        while Fraction(2) ** (s + 1) <= amax:
            s += 1
        s = min(max(s - 8, -127), 127)
    return [rn_e4m3_sat(rn_f32(v * Fraction(2) ** (-s))) for v in vals], s


def test_mxfp8_vs_exact_pipeline(oracle_lib):
    T, H, E, R, K = 6, 128, 8, 2, 2
    idx = random_routing(T, K, E, 12).numpy()
    L = oracle_lib.layout(idx, None, E, R)
    x = _x_bits(T, H, 17, scale=4.0)
    x[0, 32:64] = 0                                   # zero block
    x[1, :32] = _x_bits(1, 32, 3, scale=1e-36)[0]     # tiny (subnormal-range) block
    x[2, 70] = 0x8000                                 # negative zero in a live block
    q, s, st = oracle_lib.dispatch_mxfp8(x, L)
    assert st == 0
    table = _torch_e4m3_table()
    for t in range(T):
        for b in range(H // 32):
            want_q, want_s = _exact_mx_block(x[t, b * 32:(b + 1) * 32])
            for slot in L.recv_slot[t][L.recv_slot[t] >= 0]:
                assert int(s[slot, b]) == want_s + 127, (t, b)
                got = [Fraction(float(table[c])) for c in q[slot, b * 32:(b + 1) * 32]]
                assert got == want_q, (t, b)
    z = L.recv_slot[2][L.recv_slot[2] >= 0]
    assert np.all(q[z, 70] == 0x80)


def test_mxfp8_vs_library_pipeline(oracle_lib):
    """torch's float8_e8m0fnu decodes the scale bytes, numpy multiplies by the
    power of two, torch's float8_e4m3fn converts; on a DeepSeek-V3 slice."""
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    T, H, E, R = 32, 7168, 256, 8
    inp = make_inputs(WORKLOADS["dsv3"].scaled(T), with_y=False)
    L = oracle_lib.layout(inp.topk_idx.numpy(), None, E, R)
    q, s, st = oracle_lib.dispatch_mxfp8(bf16_bits(inp.x), L)
    assert st == 0
    xf = inp.x.float().numpy().reshape(T, H // 32, 32)
    amax = np.abs(xf).max(axis=2)
    for t in range(T):
        slot = L.recv_slot[t][L.recv_slot[t] >= 0][0]
        scale = torch.from_numpy(s[slot].copy()).view(torch.float8_e8m0fnu).float().numpy()
        # the scale puts the block max in [256, 512)
        assert np.all((amax[t] / scale >= 256) & (amax[t] / scale < 512))
        v = np.clip((xf[t] / scale[:, None]).astype(np.float32), -448, 448)
        ref = torch.from_numpy(v.reshape(H)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q[slot], ref)
