"""Pins for the oracle's backward operators: adjoint identities in exact
arithmetic (integer-valued data keeps every fp32 sum exact), exact rational
pipelines, and an independent fp64 computation with numpy."""
from fractions import Fraction

import numpy as np
import torch

from combine_moe_dispatch_02_gb300.inputs import bf16_bits, random_routing, random_weights
from exact import bf16_value, bits_of_f32, rn_bf16, rn_f32


def _int_bits(shape, seed, lo=-8, hi=8):
    """bf16 patterns of small integers (every fp32 sum of a few stays exact)."""
    g = torch.Generator().manual_seed(seed)
    v = torch.randint(lo, hi + 1, shape, generator=g).float()
    return bf16_bits(v.to(torch.bfloat16)), v.double().numpy()


def test_dispatch_backward_is_the_adjoint(oracle_lib):
    """<dispatch(x), g> == <x, dispatch_backward(g)> for integer-valued data."""
    T, H, E, R, K = 40, 16, 12, 4, 3
    idx = random_routing(T, K, E, 1, mask_frac=0.1).numpy()
    L = oracle_lib.layout(idx, None, E, R)
    xb, xv = _int_bits((T, H), 2)
    gb, gv = _int_bits((L.capacity, H), 3)
    recv, st = oracle_lib.dispatch_bf16(xb, L)
    assert st == 0
    recv_v = torch.from_numpy(recv.view(np.int16)).view(torch.bfloat16).double().numpy()
    gx, st = oracle_lib.dispatch_backward(gb, L.recv_slot)
    assert st == 0
    gx_v = torch.from_numpy(gx.view(np.int16)).view(torch.bfloat16).double().numpy()
    used = np.zeros(L.capacity, bool)
    used[:L.n_pairs] = True
    assert np.sum(recv_v[used] * gv[used]) == np.sum(xv * gx_v)


def test_dispatch_backward_vs_exact_sum(oracle_lib):
    T, H, E, R, K = 7, 24, 16, 8, 4
    idx = random_routing(T, K, E, 4).numpy()
    L = oracle_lib.layout(idx, None, E, R)
    g = torch.Generator().manual_seed(5)
    gb = bf16_bits((torch.randn(L.capacity, H, generator=g) * 3).to(torch.bfloat16))
    gx, st = oracle_lib.dispatch_backward(gb, L.recv_slot)
    assert st == 0
    for t in range(T):
        for h in range(H):
            acc = Fraction(0)
            for r in range(R):
                s = L.recv_slot[t, r]
                if s >= 0:
                    acc = rn_f32(acc + bf16_value(int(gb[s, h])))
            assert gx[t, h] == bits_of_f32(float(rn_bf16(acc))) >> 16, (t, h)


def test_dispatch_backward_sums_in_ascending_rank():
    """One token on ranks 0, 1 and 2 (one expert per rank) whose receive rows
    hold 2^24, 1 and -2^24: the fp32 chain in ascending rank order gives
    (2^24 + 1) - 2^24 = 2^24 - 2^24 = 0 (2^24 + 1 rounds to the even 2^24);
    descending order gives (-2^24 + 1) + 2^24 = 1."""
    import oracle
    oracle.build()
    L = oracle.layout(np.array([[0, 1, 2]], np.int32), None, 3, 3)
    H = 8
    g = np.zeros((L.capacity, H), np.uint16)
    for r, bits in enumerate((0x4B80, 0x3F80, 0xCB80)):      # bf16 2^24, 1, -2^24
        g[L.recv_slot[0, r]] = bits
    gx, st = oracle.dispatch_backward(g, L.recv_slot)
    assert st == 0
    assert np.all(gx == 0x0000)


def test_combine_backward_grad_y_exact(oracle_lib):
    T, H, E, R, K = 9, 20, 8, 4, 3
    idx = random_routing(T, K, E, 6, mask_frac=0.2).numpy()
    w = random_weights(T, K, 6).numpy()
    L = oracle_lib.layout(idx, w, E, R)
    g = torch.Generator().manual_seed(7)
    go = bf16_bits(torch.randn(T, H, generator=g).to(torch.bfloat16))
    y = bf16_bits(torch.randn(T * K, H, generator=g).to(torch.bfloat16))
    sentinel = np.full((T * K, H), 0x7E7E, np.uint16)
    gy, gw, st = oracle_lib.combine_backward(go, y, L.expert_slot, w, sentinel.copy())
    assert st == 0
    touched = np.zeros(T * K, bool)
    for t in range(T):
        for k in range(K):
            row = L.expert_slot[t, k]
            if row < 0:
                assert gw[t, k] == 0.0
                continue
            touched[row] = True
            for h in range(H):
                want = rn_bf16(rn_f32(Fraction(float(w[t, k])) * bf16_value(int(go[t, h]))))
                assert gy[row, h] == bits_of_f32(float(want)) >> 16
    assert np.all(gy[~touched] == 0x7E7E)


def test_combine_backward_grad_w_vs_numpy_fp64(oracle_lib):
    T, H, E, R, K = 64, 256, 16, 4, 4
    idx = random_routing(T, K, E, 8).numpy()
    w = random_weights(T, K, 8).numpy()
    L = oracle_lib.layout(idx, w, E, R)
    g = torch.Generator().manual_seed(9)
    go_t = torch.randn(T, H, generator=g).to(torch.bfloat16)
    y_t = torch.randn(T * K, H, generator=g).to(torch.bfloat16)
    _, gw, st = oracle_lib.combine_backward(bf16_bits(go_t), bf16_bits(y_t), L.expert_slot, w)
    assert st == 0
    go, y = go_t.double().numpy(), y_t.double().numpy()
    ref = np.einsum("th,tkh->tk", go, y[L.expert_slot])            # numpy, fp64
    assert np.allclose(gw, ref, rtol=1e-12, atol=1e-12)


def test_combine_backward_adjoint_identity(oracle_lib):
    """sum_t <combine(y, w)[t], g[t]> == sum_{t,k} w[t,k] * grad_w[t,k]
    (the combine is linear in w), in exact arithmetic on integer-valued data
    with power-of-two weights."""
    T, H, E, R, K = 30, 12, 8, 4, 2
    idx = random_routing(T, K, E, 10).numpy()
    w = np.full((T, K), 0.5, np.float32)
    L = oracle_lib.layout(idx, w, E, R)
    yb, yv = _int_bits((T * K, H), 11)
    gb, gv = _int_bits((T, H), 12)
    out, st = oracle_lib.combine(yb, L.expert_slot, w)
    assert st == 0
    out_v = torch.from_numpy(out.view(np.int16)).view(torch.bfloat16).double().numpy()
    _, gw, st = oracle_lib.combine_backward(gb, yb, L.expert_slot, w)
    assert st == 0
    assert np.sum(out_v * gv) == np.sum(w.astype(np.float64) * gw)
